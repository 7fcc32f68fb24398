"""chain_gb300 -- Python binding of the sm_103a C-ABI library for O = f(A.B).C.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libchain_gb300.so`` (see ``include/chain.h``).  PyTorch is used
for device memory and streams.  There is no fallback: if the library is
missing or cannot be built, importing the binding's functions raises.

Entry points (same names as the C ABI):
  chain_fwd(A, B, C, f, mask, scale, O, LSE=None, stream=None)
  chain_bwd(dO, A, B, C, O, LSE, f, mask, scale, dA, dB, dC, workspace, stream=None)
  chain_bwd_workspace_size(A, C)
  sp_relayout(shards, p, head_group, out, stream=None)
  sp_relayout_inverse(inp, p, head_group, shards, stream=None)
  chain_check(stream=None)
plus allocating conveniences ``attention_fwd``, ``attention_bwd``,
``mlp_chain_fwd`` and ``relayout``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

F_IDENTITY, F_SOFTMAX, F_GELU_TANH = 0, 1, 2
MASK_NONE, MASK_CAUSAL = 0, 1
BF16, F32, E4M3 = 0, 1, 2

OK, ERR_ARG, ERR_DTYPE, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
ERR_SCRATCH_LIMIT = -7
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # CHAIN_NOALLOC_SCRATCH_BYTES

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libchain_gb300.so")
_lock = threading.Lock()
_lib = None


class ChainError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _load().chain_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cuda error {_load().chain_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{status}]")


class TensorDesc(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                build()
            lib = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER(TensorDesc)
            vp, ci, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.chain_fwd.argtypes = [P, P, P, ci, ci, fl, P, P, vp]
            lib.chain_bwd.argtypes = [P, P, P, P, P, P, ci, ci, fl, P, P, P, vp, ctypes.c_size_t, vp]
            lib.chain_bwd_noalloc.argtypes = [P, P, P, P, P, P, ci, ci, fl, P, P, P, vp]
            lib.chain_bwd_workspace_size.argtypes = [P, P]
            lib.chain_bwd_workspace_size.restype = ctypes.c_size_t
            lib.chain_bwd_workspace_size_f.argtypes = [P, P, ci]
            lib.chain_bwd_workspace_size_f.restype = ctypes.c_size_t
            lib.chain_fwd_sp.argtypes = [P, P, P, ci, ci, ci, fl, P, P, vp]
            lib.chain_fwd_varlen.argtypes = [P, P, P, vp, ci, ci, ci, fl, P, P, vp]
            lib.chain_bwd_varlen.argtypes = [P, P, P, P, P, P, vp, ci, ci, ci, fl, P, P, P, vp,
                                             ctypes.c_size_t, vp]
            lib.chain_fwd_fp8.argtypes = [P, P, P, ci, fl, fl, P, P, vp, ctypes.c_size_t, vp]
            lib.chain_fwd_f16pv.argtypes = [P, P, P, ci, fl, P, P, vp, ctypes.c_size_t, vp]
            lib.chain_fwd_f16pv_workspace_size.argtypes = [P, P]
            lib.chain_fwd_sp_f16pv.argtypes = [P, P, P, ci, ci, ci, fl, P, P, vp, ctypes.c_size_t,
                                               vp]
            lib.chain_fwd_f16h.argtypes = [P, P, P, ci, P, vp, ctypes.c_size_t, vp]
            lib.chain_fwd_f16h_workspace_size.argtypes = [P]
            lib.chain_fwd_f16h_workspace_size.restype = ctypes.c_size_t
            lib.chain_fwd_varlen_f16pv.argtypes = [P, P, P, vp, ci, ci, ci, fl, P, P, vp,
                                                   ctypes.c_size_t, vp]
            lib.chain_fwd_varlen_f16pv_workspace_size.argtypes = [P]
            lib.chain_fwd_varlen_f16pv_workspace_size.restype = ctypes.c_size_t
            lib.chain_fwd_sp_f16pv_workspace_size.argtypes = [P, ci]
            lib.chain_fwd_sp_f16pv_workspace_size.restype = ctypes.c_size_t
            lib.chain_fwd_f16pv_workspace_size.restype = ctypes.c_size_t
            lib.chain_fwd_fp8_workspace_size.argtypes = [P]
            lib.chain_fwd_fp8_workspace_size.restype = ctypes.c_size_t
            lib.sp_relayout.argtypes = [P, ci, ci, P, vp]
            lib.sp_relayout_inverse.argtypes = [P, ci, ci, P, vp]
            lib.chain_check.argtypes = [vp, ctypes.POINTER(ci)]
            lib.chain_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.chain_set_wait_limit_ns.restype = None
            lib.chain_set_timing_events.argtypes = [ctypes.POINTER(vp), ci]
            lib.chain_set_timing_events.restype = None
            lib.chain_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
            lib.chain_umma_selftest.argtypes = [vp, vp, vp, ci, ci, ci, vp]
            lib.chain_status_string.argtypes = [ci]
            lib.chain_status_string.restype = ctypes.c_char_p
            for fn in ("chain_fwd", "chain_fwd_sp", "chain_fwd_varlen", "chain_bwd", "chain_bwd_varlen",
                       "chain_bwd_noalloc", "chain_fwd_fp8", "chain_fwd_f16pv",
                       "chain_fwd_sp_f16pv",
                       "sp_relayout",
                       "sp_relayout_inverse",
                       "chain_check", "chain_selftest_wait_timeout", "chain_umma_selftest",
                       "chain_last_cuda_error"):
                getattr(lib, fn).restype = ci
            _lib = lib
    return _lib


def lib():
    return _load()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.int16 or t.dtype == torch.float16:
        return BF16  # 2-byte payload (relayout moves bits only)
    if t.dtype == torch.int32:
        return F32  # 4-byte payload
    if t.dtype == torch.float8_e4m3fn:
        return E4M3
    if t.dtype == torch.uint8 or t.dtype == torch.int8:
        return E4M3  # 1-byte payload (relayout moves bits only)
    raise TypeError(f"chain_gb300: unsupported dtype {t.dtype}")


def desc(t: torch.Tensor | None):
    if t is None:
        return None
    if t.dim() < 1 or t.dim() > 4:
        raise ValueError("chain_gb300: tensors must have 1 to 4 dimensions")
    d = TensorDesc()
    d.ptr = t.data_ptr()
    d.dtype = _dt(t)
    d.ndim = t.dim()
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = s
        d.stride[i] = st
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ok(rc: int, what: str):
    if rc != OK:
        raise ChainError(rc, what)


# ------------------------------------------------------------- C-ABI calls
def chain_fwd(A, B, C, f, mask, scale, O, LSE=None, stream=None):
    """O = f(A B) C; see include/chain.h for shapes per f."""
    _ok(_load().chain_fwd(_ref(desc(A)), _ref(desc(B)), _ref(desc(C)), int(f), int(mask),
                          float(scale), _ref(desc(O)), _ref(desc(LSE)), _stream(stream)),
        "chain_fwd")


def chain_fwd_f16h(A, B, C, f, O, workspace, stream=None):
    """MLP chain O = f(A B) C with the intermediate as one f16 tile; see include/chain.h."""
    _ok(_load().chain_fwd_f16h(_ref(desc(A)), _ref(desc(B)), _ref(desc(C)), int(f), _ref(desc(O)),
                               ctypes.c_void_p(workspace.data_ptr()),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
        "chain_fwd_f16h")


def chain_fwd_f16h_workspace_size(C) -> int:
    return int(_load().chain_fwd_f16h_workspace_size(_ref(desc(C))))


def chain_fwd_fp8(Q, K, V, mask, scale, v_scale, O, LSE, workspace, stream=None):
    """Attention on e4m3 Q, K, V (d = 128) into bf16 O; see include/chain.h."""
    _ok(_load().chain_fwd_fp8(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)), int(mask), float(scale),
                              float(v_scale), _ref(desc(O)), _ref(desc(LSE)),
                              ctypes.c_void_p(workspace.data_ptr()),
                              workspace.numel() * workspace.element_size(), _stream(stream)),
        "chain_fwd_fp8")


def chain_fwd_f16pv(Q, K, V, mask, scale, O, LSE, workspace, stream=None):
    """Softmax attention, bf16, P V as one f16 product; see include/chain.h."""
    _ok(_load().chain_fwd_f16pv(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)), int(mask),
                                float(scale), _ref(desc(O)), _ref(desc(LSE)),
                                ctypes.c_void_p(workspace.data_ptr()),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
        "chain_fwd_f16pv")


def chain_fwd_sp_f16pv(Q, K, V, p, head_group, mask, scale, O, LSE, workspace, stream=None):
    """chain_fwd_sp with P V as one f16 product; see include/chain.h."""
    _ok(_load().chain_fwd_sp_f16pv(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)), int(p),
                                   int(head_group), int(mask), float(scale), _ref(desc(O)),
                                   _ref(desc(LSE)), ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
        "chain_fwd_sp_f16pv")


def chain_fwd_sp_f16pv_workspace_size(V, p) -> int:
    return int(_load().chain_fwd_sp_f16pv_workspace_size(_ref(desc(V)), int(p)))


def chain_fwd_f16pv_workspace_size(Q, V) -> int:
    return int(_load().chain_fwd_f16pv_workspace_size(_ref(desc(Q)), _ref(desc(V))))


def chain_fwd_fp8_workspace_size(V) -> int:
    return int(_load().chain_fwd_fp8_workspace_size(_ref(desc(V))))


def chain_fwd_sp(Q, K, V, p, head_group, mask, scale, O, LSE, stream=None):
    """Attention of one head group read from and written to sequence shards
    [p][n_loc][H][d]; see include/chain.h."""
    _ok(_load().chain_fwd_sp(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)), int(p), int(head_group),
                             int(mask), float(scale), _ref(desc(O)), _ref(desc(LSE)),
                             _stream(stream)), "chain_fwd_sp")


def chain_fwd_varlen(Q, K, V, cu_seqlens, batch, max_seqlen, mask, scale, O, LSE, stream=None):
    """Attention over sequences packed end to end; cu_seqlens is a device
    int32 tensor [batch + 1]; see include/chain.h."""
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a CUDA int32 tensor")
    _ok(_load().chain_fwd_varlen(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)),
                                 ctypes.c_void_p(cu_seqlens.data_ptr()), int(batch), int(max_seqlen),
                                 int(mask), float(scale), _ref(desc(O)), _ref(desc(LSE)),
                                 _stream(stream)), "chain_fwd_varlen")


def chain_fwd_varlen_f16pv(Q, K, V, cu_seqlens, batch, max_seqlen, mask, scale, O, LSE, workspace,
                           stream=None):
    """chain_fwd_varlen with P V as one f16 product; see include/chain.h."""
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a CUDA int32 tensor")
    _ok(_load().chain_fwd_varlen_f16pv(_ref(desc(Q)), _ref(desc(K)), _ref(desc(V)),
                                       ctypes.c_void_p(cu_seqlens.data_ptr()), int(batch),
                                       int(max_seqlen), int(mask), float(scale), _ref(desc(O)),
                                       _ref(desc(LSE)), ctypes.c_void_p(workspace.data_ptr()),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "chain_fwd_varlen_f16pv")


def chain_fwd_varlen_f16pv_workspace_size(V) -> int:
    return int(_load().chain_fwd_varlen_f16pv_workspace_size(_ref(desc(V))))


def chain_bwd_varlen(dO, Q, K, V, O, LSE, cu_seqlens, batch, max_seqlen, mask, scale, dQ, dK, dV,
                     workspace, stream=None):
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a CUDA int32 tensor")
    _ok(_load().chain_bwd_varlen(_ref(desc(dO)), _ref(desc(Q)), _ref(desc(K)), _ref(desc(V)),
                                 _ref(desc(O)), _ref(desc(LSE)), ctypes.c_void_p(cu_seqlens.data_ptr()),
                                 int(batch), int(max_seqlen), int(mask), float(scale),
                                 _ref(desc(dQ)), _ref(desc(dK)), _ref(desc(dV)),
                                 ctypes.c_void_p(workspace.data_ptr()),
                                 ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                 _stream(stream)), "chain_bwd_varlen")


def chain_bwd_workspace_size(A, C) -> int:
    return int(_load().chain_bwd_workspace_size(_ref(desc(A)), _ref(desc(C))))


def chain_bwd_workspace_size_f(A, C, f) -> int:
    return int(_load().chain_bwd_workspace_size_f(_ref(desc(A)), _ref(desc(C)), int(f)))


def chain_bwd(dO, A, B, C, O, LSE, f, mask, scale, dA, dB, dC, workspace, stream=None):
    _ok(_load().chain_bwd(_ref(desc(dO)), _ref(desc(A)), _ref(desc(B)), _ref(desc(C)),
                          _ref(desc(O)), _ref(desc(LSE)), int(f), int(mask), float(scale),
                          _ref(desc(dA)), _ref(desc(dB)), _ref(desc(dC)),
                          ctypes.c_void_p(workspace.data_ptr()),
                          ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                          _stream(stream)), "chain_bwd")


def chain_bwd_noalloc(dO, A, B, C, O, LSE, f, mask, scale, dA, dB, dC, stream=None):
    """chain_bwd without a workspace argument: the library's fixed scratch
    array is used instead (see include/chain.h for the limit and the rules
    on overlapping calls)."""
    _ok(_load().chain_bwd_noalloc(_ref(desc(dO)), _ref(desc(A)), _ref(desc(B)), _ref(desc(C)),
                                  _ref(desc(O)), _ref(desc(LSE)), int(f), int(mask), float(scale),
                                  _ref(desc(dA)), _ref(desc(dB)), _ref(desc(dC)), _stream(stream)),
        "chain_bwd_noalloc")


def sp_relayout(shards, p, head_group, out, stream=None):
    _ok(_load().sp_relayout(_ref(desc(shards)), int(p), int(head_group), _ref(desc(out)),
                            _stream(stream)), "sp_relayout")


def sp_relayout_inverse(inp, p, head_group, shards, stream=None):
    _ok(_load().sp_relayout_inverse(_ref(desc(inp)), int(p), int(head_group), _ref(desc(shards)),
                                    _stream(stream)), "sp_relayout_inverse")


def chain_check(stream=None) -> tuple[int, int]:
    site = ctypes.c_int(0)
    rc = _load().chain_check(_stream(stream), ctypes.byref(site))
    return rc, site.value


def set_wait_limit_ns(ns: int):
    _load().chain_set_wait_limit_ns(int(ns))


def set_timing_events(*events):
    """Record torch.cuda.Event objects at the main-kernel boundaries of
    subsequent calls from this thread (events[0] before the first main
    kernel, events[k] after the k-th); no arguments clears."""
    for ev in events:
        if ev.cuda_event == 0:
            ev.record()  # torch creates the underlying event on first record
    arr = (ctypes.c_void_p * max(1, len(events)))(*[ev.cuda_event for ev in events])
    _load().chain_set_timing_events(arr if events else None, len(events))


def selftest_wait_timeout(limit_ns: int, stream=None):
    _ok(_load().chain_selftest_wait_timeout(int(limit_ns), _stream(stream)),
        "chain_selftest_wait_timeout")


def umma_selftest(A, B, D, N, K, b_mn_major, a_in_tmem=False, stream=None):
    flags = int(bool(b_mn_major)) | (2 if a_in_tmem else 0)
    _ok(_load().chain_umma_selftest(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                    ctypes.c_void_p(D.data_ptr()), int(N), int(K), flags,
                                    _stream(stream)), "chain_umma_selftest")


# --------------------------------------------------- allocating helpers
def attention_fwd(q, k, v, causal: bool, scale: float | None = None, stream=None):
    """Returns (O, LSE) for q, k, v [BH, n, d] (or [B, H, n, d])."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    chain_fwd(q, k, v, F_SOFTMAX, MASK_CAUSAL if causal else MASK_NONE, scale, o, lse, stream)
    return o, lse


def attention_fwd_f16pv(q, k, v, causal: bool, scale: float | None = None, workspace=None,
                        stream=None):
    """Returns (O, LSE) for bf16 q [BH, n, d], k, v [BHkv, n, d]; P V in f16."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(chain_fwd_f16pv_workspace_size(q, v), 16), dtype=torch.uint8,
                                device=q.device)
    chain_fwd_f16pv(q, k, v, MASK_CAUSAL if causal else MASK_NONE, scale, o, lse, workspace, stream)
    return o, lse


def attention_fwd_fp8(q, k, v, causal: bool, scale: float | None = None, v_scale: float = 1.0,
                      workspace=None, stream=None):
    """Returns (O bf16, LSE) for e4m3 q [BH, n, 128], k, v [BHkv, n, 128]."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(chain_fwd_fp8_workspace_size(v), 16), dtype=torch.uint8,
                                device=q.device)
    chain_fwd_fp8(q, k, v, MASK_CAUSAL if causal else MASK_NONE, scale, v_scale, o, lse, workspace,
                  stream)
    return o, lse


def attention_fwd_sp(q, k, v, p: int, head_group: int, causal: bool, scale: float | None = None,
                     o=None, stream=None):
    """Shards q, k, v [p][n_loc][H][d] -> (O shards, LSE [H/p][p*n_loc]).  Only
    the heads of `head_group` are written into `o` (a new zeroed tensor if
    None)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    P, n_loc, H, d = q.shape
    if o is None:
        o = torch.zeros_like(q)
    lse = torch.empty(H // p, p * n_loc, dtype=torch.float32, device=q.device)
    chain_fwd_sp(q, k, v, p, head_group, MASK_CAUSAL if causal else MASK_NONE, scale, o, lse, stream)
    return o, lse


def attention_fwd_sp_f16pv(q, k, v, p: int, head_group: int, causal: bool,
                           scale: float | None = None, o=None, workspace=None, stream=None):
    """attention_fwd_sp with P V as one f16 product."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    P, n_loc, H, d = q.shape
    if o is None:
        o = torch.zeros_like(q)
    lse = torch.empty(H // p, p * n_loc, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(chain_fwd_sp_f16pv_workspace_size(v, p), 16),
                                dtype=torch.uint8, device=q.device)
    chain_fwd_sp_f16pv(q, k, v, p, head_group, MASK_CAUSAL if causal else MASK_NONE, scale, o, lse,
                       workspace, stream)
    return o, lse


def attention_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool,
                         scale: float | None = None, stream=None):
    """q [total, H, d], k, v [total, Hkv, d]; cu_seqlens a CUDA int32 tensor
    [batch + 1].  Returns (O [total, H, d], LSE [H, total])."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    chain_fwd_varlen(q, k, v, cu_seqlens, cu_seqlens.numel() - 1, max_seqlen,
                     MASK_CAUSAL if causal else MASK_NONE, scale, o, lse, stream)
    return o, lse


def attention_fwd_varlen_f16pv(q, k, v, cu_seqlens, max_seqlen: int, causal: bool,
                               scale: float | None = None, workspace=None, stream=None):
    """attention_fwd_varlen with P V as one f16 product: returns (O, LSE)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(max(chain_fwd_varlen_f16pv_workspace_size(v), 16),
                                dtype=torch.uint8, device=q.device)
    chain_fwd_varlen_f16pv(q, k, v, cu_seqlens, cu_seqlens.numel() - 1, max_seqlen,
                           MASK_CAUSAL if causal else MASK_NONE, scale, o, lse, workspace, stream)
    return o, lse


def attention_bwd_varlen(do, q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool,
                         scale: float | None = None, stream=None):
    """Gradients of attention_fwd_varlen: returns (dQ, dK, dV), packed like q, k, v."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    ws = torch.empty(chain_bwd_workspace_size(q, q), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    chain_bwd_varlen(do, q, k, v, o, lse, cu_seqlens, cu_seqlens.numel() - 1, max_seqlen,
                     MASK_CAUSAL if causal else MASK_NONE, scale, dq, dk, dv, ws, stream)
    return dq, dk, dv


def attention_bwd(do, q, k, v, o, lse, causal: bool, scale: float | None = None,
                  workspace=None, stream=None):
    """Returns (dQ, dK, dV)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    if workspace is None:
        nbytes = chain_bwd_workspace_size(q, v)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    chain_bwd(do, q, k, v, o, lse, F_SOFTMAX, MASK_CAUSAL if causal else MASK_NONE, scale,
              dq, dk, dv, workspace, stream)
    return dq, dk, dv


def mlp_chain_fwd_f16h(x, w1, w2, gelu: bool = True, workspace=None, stream=None):
    """O = gelu_tanh(x w1) w2 (or (x w1) w2) with the intermediate as one f16 tile."""
    o = torch.empty(x.shape[0], w2.shape[1], dtype=x.dtype, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(chain_fwd_f16h_workspace_size(w2), 16), dtype=torch.uint8,
                                device=x.device)
    chain_fwd_f16h(x, w1, w2, F_GELU_TANH if gelu else F_IDENTITY, o, workspace, stream)
    return o


def mlp_chain_fwd(x, w1, w2, gelu: bool = True, stream=None):
    """O = gelu_tanh(x w1) w2 (or (x w1) w2 with gelu=False)."""
    o = torch.empty(x.shape[0], w2.shape[1], dtype=x.dtype, device=x.device)
    chain_fwd(x, w1, w2, F_GELU_TANH if gelu else F_IDENTITY, MASK_NONE, 1.0, o, None, stream)
    return o


def mlp_chain_bwd(do, x, w1, w2, gelu: bool = True, workspace=None, stream=None):
    """Returns (dX, dW1, dW2) of O = gelu_tanh(x w1) w2 (or identity)."""
    f = F_GELU_TANH if gelu else F_IDENTITY
    if workspace is None:
        workspace = torch.empty(chain_bwd_workspace_size_f(x, w2, f), dtype=torch.uint8,
                                device=x.device)
    dx, dw1, dw2 = torch.empty_like(x), torch.empty_like(w1), torch.empty_like(w2)
    chain_bwd(do, x, w1, w2, None, None, f, MASK_NONE, 1.0, dx, dw1, dw2, workspace, stream)
    return dx, dw1, dw2


def relayout(shards, p: int, head_group: int, stream=None):
    P, n_loc, H, d = shards.shape
    out = torch.empty(H // p, p * n_loc, d, dtype=shards.dtype, device=shards.device)
    sp_relayout(shards, p, head_group, out, stream)
    return out
