"""fp64 CPU oracle for the O = f(A.B).C unit -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``chain_gb300``) never touches it.

This module only marshals arguments into ``oracle.c`` (plain C, fp64,
OpenMP); every step of the arithmetic lives there, written from the
definitions cited in its header.  Inputs are torch CPU tensors or numpy
arrays holding bf16, e4m3, fp32 or fp64 values; outputs are fp64 numpy
arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32, F64, E4M3 = 0, 1, 2, 3
F_IDENTITY, F_SOFTMAX, F_GELU_TANH = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
           "-fopenmp", "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            ci = ctypes.c_int
            lib.oracle_num_threads.restype = ci
            lib.oracle_softmax_fwd.argtypes = [ci, vp, vp, vp, i64, i64, i64, i64, dbl, ci,
                                               i64, vp, vp, vp, vp]
            lib.oracle_softmax_fwd_blocked.argtypes = [ci, vp, vp, vp, i64, i64, i64, i64,
                                                       dbl, ci, i64, i64, vp, vp]
            lib.oracle_softmax_bwd.argtypes = [ci, vp, vp, vp, vp, i64, i64, i64, i64, dbl,
                                               ci, i64, i64, i64, i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_chain_fwd.argtypes = [ci, vp, vp, vp, i64, i64, i64, i64, ci, dbl,
                                             i64, vp, vp]
            lib.oracle_chain_bwd.argtypes = [ci, vp, vp, vp, vp, i64, i64, i64, i64, ci, i64, vp,
                                             i64, vp, vp, vp, vp]
            lib.oracle_relayout.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp]
            lib.oracle_e4m3_decode.argtypes = [vp, i64, vp]
            lib.oracle_e4m3_decode.restype = None
            lib.oracle_relayout_inverse.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp]
            for fn in ("oracle_softmax_fwd", "oracle_softmax_fwd_blocked", "oracle_softmax_bwd",
                       "oracle_chain_fwd", "oracle_chain_bwd", "oracle_relayout",
                       "oracle_relayout_inverse"):
                getattr(lib, fn).restype = ci
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _raw(x):
    """Return (contiguous numpy array holding the stored bits, dtype code)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy(), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy(), E4M3
            raise TypeError(f"oracle: unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    raise TypeError(f"oracle: unsupported dtype {x.dtype}")


def _same(*arrs):
    codes = {c for _, c in arrs}
    if len(codes) != 1:
        raise TypeError("oracle: all inputs must share one dtype")
    return codes.pop()


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (uint8 array or torch float8_e4m3fn)."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().contiguous()
            if codes.dtype == torch.float8_e4m3fn:
                codes = codes.view(torch.uint8)
            codes = codes.numpy()
    except ImportError:  # pragma: no cover
        pass
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode(_p(c), int(c.size), _p(out))
    return out


def softmax_fwd(Q, K, V, scale: float, causal: bool, rows=None):
    """Plain softmax attention forward.

    Q, K: [BH, n, d]; V: [BH, n, dv].  ``rows`` is None for every (bh, i), or
    an int array of shape [R, 2] of (bh, i) pairs.  Returns (O, LSE): O has
    shape [BH, n, dv] / LSE [BH, n] for all rows, else [R, dv] / [R].
    """
    q, k, v = _raw(Q), _raw(K), _raw(V)
    dt = _same(q, k, v)
    BH, n, d = q[0].shape
    dv = v[0].shape[-1]
    if rows is None:
        bh = np.repeat(np.arange(BH, dtype=np.int64), n)
        ii = np.tile(np.arange(n, dtype=np.int64), BH)
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        bh, ii = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
    R = bh.shape[0]
    O = np.empty((R, dv), np.float64)
    L = np.empty((R,), np.float64)
    rc = _load().oracle_softmax_fwd(dt, _p(q[0]), _p(k[0]), _p(v[0]), BH, n, d, dv,
                                    float(scale), int(bool(causal)), R, _p(bh), _p(ii),
                                    _p(O), _p(L))
    if rc != 0:
        raise RuntimeError(f"oracle_softmax_fwd failed ({rc})")
    if rows is None:
        return O.reshape(BH, n, dv), L.reshape(BH, n)
    return O, L


def softmax_fwd_blocked(Q, K, V, scale: float, causal: bool, pq: int, pk: int):
    """pq x pk block decomposition with the online (max, sum) merge."""
    q, k, v = _raw(Q), _raw(K), _raw(V)
    dt = _same(q, k, v)
    BH, n, d = q[0].shape
    dv = v[0].shape[-1]
    O = np.empty((BH, n, dv), np.float64)
    L = np.empty((BH, n), np.float64)
    rc = _load().oracle_softmax_fwd_blocked(dt, _p(q[0]), _p(k[0]), _p(v[0]), BH, n, d, dv,
                                            float(scale), int(bool(causal)), pq, pk,
                                            _p(O), _p(L))
    if rc != 0:
        raise RuntimeError(f"oracle_softmax_fwd_blocked failed ({rc})")
    return O, L


def softmax_bwd(Q, K, V, dO, scale: float, causal: bool, heads=None, row_range=None,
                col_range=None):
    """Textbook softmax-attention backward.

    ``heads`` = (bh0, bh1), ``row_range`` = (i0, i1), ``col_range`` = (j0, j1);
    defaults cover everything.  Returns (dQ [nh, i1-i0, d], dK [nh, j1-j0, d],
    dV [nh, j1-j0, dv], D [nh, i1-i0]).  dK/dV hold the contributions of the
    requested rows only.
    """
    q, k, v, g = _raw(Q), _raw(K), _raw(V), _raw(dO)
    dt = _same(q, k, v, g)
    BH, n, d = q[0].shape
    dv = v[0].shape[-1]
    bh0, bh1 = heads if heads is not None else (0, BH)
    i0, i1 = row_range if row_range is not None else (0, n)
    j0, j1 = col_range if col_range is not None else (0, n)
    nh, nr, nc = bh1 - bh0, i1 - i0, j1 - j0
    dQ = np.empty((nh, nr, d), np.float64)
    dK = np.empty((nh, nc, d), np.float64)
    dV = np.empty((nh, nc, dv), np.float64)
    D = np.empty((nh, nr), np.float64)
    rc = _load().oracle_softmax_bwd(dt, _p(q[0]), _p(k[0]), _p(v[0]), _p(g[0]), BH, n, d, dv,
                                    float(scale), int(bool(causal)), bh0, bh1, i0, i1, j0, j1,
                                    _p(dQ), _p(dK), _p(dV), _p(D))
    if rc != 0:
        raise RuntimeError(f"oracle_softmax_bwd failed ({rc})")
    return dQ, dK, dV, D


def chain_fwd(A, B, C, f: int, scale: float = 1.0, rows=None):
    """General O = f(A B) C for requested rows (None = all).  A [M,K], B [K,N], C [N,P]."""
    a, b, c = _raw(A), _raw(B), _raw(C)
    dt = _same(a, b, c)
    M, K = a[0].shape
    K2, N = b[0].shape
    N2, P = c[0].shape
    if K2 != K or N2 != N:
        raise ValueError("oracle.chain_fwd: inner dimensions differ")
    r = (np.arange(M, dtype=np.int64) if rows is None
         else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    O = np.empty((r.shape[0], P), np.float64)
    rc = _load().oracle_chain_fwd(dt, _p(a[0]), _p(b[0]), _p(c[0]), M, K, N, P, int(f),
                                  float(scale), r.shape[0], _p(r), _p(O))
    if rc != 0:
        raise RuntimeError(f"oracle_chain_fwd failed ({rc})")
    return O


def chain_bwd(A, B, C, dO, f: int, rows=None, hidden=None):
    """Backward of O = f(A B) C (f identity or gelu_tanh), the intermediate
    recomputed.  A [M,K], B [K,N], C [N,P], dO [M,P].

    Returns (dA_rows [R,K], dB_cols [RH,K], dC_rows [RH,P]): rows `rows` of
    dA (None = all) and, for hidden units `hidden` (None = all), column h of
    dB (stored as a row) and row h of dC."""
    a, b, c, g = _raw(A), _raw(B), _raw(C), _raw(dO)
    dt = _same(a, b, c, g)
    M, K = a[0].shape
    K2, N = b[0].shape
    N2, P = c[0].shape
    if K2 != K or N2 != N or g[0].shape != (M, P):
        raise ValueError("oracle.chain_bwd: shapes differ")
    ra = (np.arange(M, dtype=np.int64) if rows is None
          else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    rh = (np.arange(N, dtype=np.int64) if hidden is None
          else np.ascontiguousarray(np.asarray(hidden, dtype=np.int64)))
    dA = np.empty((ra.shape[0], K), np.float64)
    dB = np.empty((rh.shape[0], K), np.float64)
    dC = np.empty((rh.shape[0], P), np.float64)
    rc = _load().oracle_chain_bwd(dt, _p(a[0]), _p(b[0]), _p(c[0]), _p(g[0]), M, K, N, P, int(f),
                                  ra.shape[0], _p(ra), rh.shape[0], _p(rh), _p(dA), _p(dB), _p(dC))
    if rc != 0:
        raise RuntimeError(f"oracle_chain_bwd failed ({rc})")
    return dA, dB, dC


def _bytes_view(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            return x.view(torch.uint8).numpy().reshape(-1), x.element_size(), tuple(x.shape)
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    return x.view(np.uint8).reshape(-1), x.itemsize, x.shape


def relayout(shards, p: int, g: int):
    """Sequence shards [p, n_loc, H, d] -> head-major [H/p, p*n_loc, d] for group g.

    Returns a uint8 numpy array of the output bytes and the output shape."""
    raw, esz, shp = _bytes_view(shards)
    p_, n_loc, H, d = shp
    if p_ != p:
        raise ValueError("oracle.relayout: leading dim must equal p")
    out = np.zeros(((H // p) * p * n_loc * d * esz,), np.uint8)
    rc = _load().oracle_relayout(_p(raw), esz, p, n_loc, H, d, g, _p(out))
    if rc != 0:
        raise RuntimeError(f"oracle_relayout failed ({rc})")
    return out, (H // p, p * n_loc, d)


def relayout_inverse(headmajor, p: int, n_loc: int, H: int, g: int, into=None):
    """Head-major [H/p, p*n_loc, d] -> the group-g heads of shards [p, n_loc, H, d].

    ``into``: optional uint8 array of the full shard bytes to update in place."""
    raw, esz, shp = _bytes_view(headmajor)
    Hl, n, d = shp
    out = (np.zeros((p * n_loc * H * d * esz,), np.uint8) if into is None else into)
    rc = _load().oracle_relayout_inverse(_p(raw), esz, p, n_loc, H, d, g, _p(out))
    if rc != 0:
        raise RuntimeError(f"oracle_relayout_inverse failed ({rc})")
    return out
