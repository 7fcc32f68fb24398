"""Host-side argument checking of every C-ABI entry point, on the CPU.

Every entry point validates its descriptors, sizes and flags on the host
before its first device call, and returns a negative status for a bad
argument.  These tests pass descriptors that hold dummy, never-dereferenced
addresses and check the status each call returns.  A fully valid call is
also made: on a machine without a GPU it must get past every argument check
and fail only at the device query (CHAIN_ERR_CUDA or CHAIN_ERR_DEVICE).
They run only where no GPU is visible, so a missing check can never send a
dummy address to a device."""
import ctypes
import math

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host-side argument checks only; never run with a device present")


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


_next_addr = [0x10000000]


def D(cg, shape, dtype=None, strides=None, ptr=None):
    """A descriptor of a dense (or explicitly strided) tensor at a dummy,
    16-byte aligned address."""
    d = cg.TensorDesc()
    if ptr is None:
        ptr = _next_addr[0]
        _next_addr[0] += 1 << 24
    d.ptr = ptr
    d.dtype = cg.BF16 if dtype is None else dtype
    d.ndim = len(shape)
    if strides is None:
        strides, st = [], 1
        for s in reversed(shape):
            strides.insert(0, st)
            st *= s
    for i, (s, t) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = t
    return d


def R(x):
    return None if x is None else ctypes.byref(x)


def no_device(cg):
    """Statuses a valid call may return on a machine without a GPU."""
    return (cg.ERR_CUDA, cg.ERR_DEVICE)


# ------------------------------------------------------------------ chain_fwd
def fwd(cg, A, B, C, f, mask, scale, O, L):
    return cg.lib().chain_fwd(R(A), R(B), R(C), f, mask, ctypes.c_float(scale), R(O), R(L), None)


def attn(cg, BH=2, n=256, d=128, BHkv=None, dtype=None):
    BHkv = BH if BHkv is None else BHkv
    q, o = D(cg, (BH, n, d), dtype), D(cg, (BH, n, d), dtype)
    k, v = D(cg, (BHkv, n, d), dtype), D(cg, (BHkv, n, d), dtype)
    lse = D(cg, (BH, n), cg.F32)
    return q, k, v, o, lse


def test_chain_fwd_attention_args(cg):
    S, C = cg.F_SOFTMAX, cg.MASK_CAUSAL
    q, k, v, o, lse = attn(cg)
    assert fwd(cg, q, k, v, S, C, 0.088, o, lse) in no_device(cg)
    assert fwd(cg, None, k, v, S, C, 0.088, o, lse) == cg.ERR_ARG
    assert fwd(cg, q, k, v, 7, C, 0.088, o, lse) == cg.ERR_ARG           # unknown f
    assert fwd(cg, q, k, v, S, 2, 0.088, o, lse) == cg.ERR_ARG           # unknown mask
    for bad in (0.0, -1.0, math.nan, math.inf):
        assert fwd(cg, q, k, v, S, C, bad, o, lse) == cg.ERR_ARG         # scale
    assert fwd(cg, q, k, v, S, C, 0.088, o, None) == cg.ERR_ARG          # LSE missing
    assert fwd(cg, q, k, v, S, C, 0.088, o, D(cg, (2, 256))) == cg.ERR_DTYPE  # LSE not fp32
    assert fwd(cg, q, k, v, S, C, 0.088, o, D(cg, (2, 255), cg.F32)) == cg.ERR_ARG
    q96, k96, v96, o96, l96 = attn(cg, d=96)
    assert fwd(cg, q96, k96, v96, S, C, 0.1, o96, l96) == cg.ERR_ARG    # head dimension
    q2, k3, v3, o2, l2 = attn(cg, BH=2, BHkv=3)
    assert fwd(cg, q2, k3, v3, S, C, 0.088, o2, l2) == cg.ERR_ARG       # K/V heads do not divide
    assert fwd(cg, q, D(cg, (2, 256, 128), cg.F32), v, S, C, 0.088, o, lse) == cg.ERR_DTYPE
    q8, k8, v8, o8, l8 = attn(cg, dtype=cg.E4M3)
    assert fwd(cg, q8, k8, v8, S, C, 0.088, o8, l8) == cg.ERR_DTYPE      # 8-bit: chain_fwd_fp8
    misaligned = D(cg, (2, 256, 128), ptr=0x20000008)
    assert fwd(cg, misaligned, k, v, S, C, 0.088, o, lse) == cg.ERR_ARG
    pitch = D(cg, (2, 256, 128), strides=(256 * 132, 132, 1))          # 264-byte rows
    assert fwd(cg, pitch, k, v, S, C, 0.088, o, lse) == cg.ERR_ARG
    inner = D(cg, (2, 256, 128), strides=(256 * 256, 256, 2))          # innermost stride 2
    assert fwd(cg, inner, k, v, S, C, 0.088, o, lse) == cg.ERR_ARG
    unfold = D(cg, (2, 1, 256, 128), strides=(1 << 20, 256 * 128, 128, 1))
    q4 = D(cg, (2, 2, 256, 128), strides=(3 * 256 * 128, 256 * 128, 128, 1))  # B, H do not fold
    assert fwd(cg, q4, q4, q4, S, C, 0.088, q4, D(cg, (2, 2, 256), cg.F32)) == cg.ERR_ARG
    assert fwd(cg, unfold, unfold, unfold, S, C, 0.088, unfold,
               D(cg, (2, 1, 256), cg.F32)) in no_device(cg)            # size-1 head dim: any stride


def test_chain_fwd_mlp_args(cg):
    G, N0 = cg.F_GELU_TANH, cg.MASK_NONE
    x, w1, w2, o = D(cg, (128, 64)), D(cg, (64, 128)), D(cg, (128, 256)), D(cg, (128, 256))
    assert fwd(cg, x, w1, w2, G, N0, 1.0, o, None) in no_device(cg)
    assert fwd(cg, x, w1, w2, cg.F_IDENTITY, N0, 1.0, o, None) in no_device(cg)
    assert fwd(cg, x, w1, w2, G, cg.MASK_CAUSAL, 1.0, o, None) == cg.ERR_ARG   # no mask on an MLP
    assert fwd(cg, x, w1, w2, G, N0, 1.0, o, D(cg, (128,), cg.F32)) == cg.ERR_ARG
    assert fwd(cg, x, D(cg, (32, 128)), w2, G, N0, 1.0, o, None) == cg.ERR_ARG  # inner dims
    assert fwd(cg, x, w1, w2, G, N0, 1.0, D(cg, (128, 128)), None) == cg.ERR_ARG
    x100, o100 = D(cg, (100, 64)), D(cg, (100, 256))
    assert fwd(cg, x100, w1, w2, G, N0, 1.0, o100, None) == cg.ERR_UNSUPPORTED  # M % 128


def test_chain_fwd_f16h_args(cg):
    lib = cg.lib()
    x, w1, w2, o = D(cg, (128, 64)), D(cg, (64, 64)), D(cg, (64, 512)), D(cg, (128, 512))
    need = lib.chain_fwd_f16h_workspace_size(ctypes.byref(w2))
    assert need >= 64 * 512 * 2
    ws = ctypes.c_void_p(0x70000000)

    def call(f, X, W1, W2, O, nbytes):
        return lib.chain_fwd_f16h(R(X), R(W1), R(W2), f, R(O), ws, ctypes.c_size_t(nbytes), None)

    assert call(cg.F_GELU_TANH, x, w1, w2, o, need) in no_device(cg)
    assert call(cg.F_GELU_TANH, x, w1, w2, o, need - 16) == cg.ERR_ARG           # short workspace
    assert call(cg.F_SOFTMAX, x, w1, w2, o, need) == cg.ERR_ARG                  # MLP only
    w2s, os_ = D(cg, (64, 256)), D(cg, (128, 256))
    assert call(cg.F_GELU_TANH, x, w1, w2s, os_, 1 << 30) == cg.ERR_UNSUPPORTED  # P < 512
    assert lib.chain_fwd_f16h_workspace_size(None) == 0


# ------------------------------------------------------------------ chain_bwd
def bwd(cg, g, q, k, v, o, lse, f, mask, scale, dq, dk, dv, ws, nbytes):
    return cg.lib().chain_bwd(R(g), R(q), R(k), R(v), R(o), R(lse), f, mask, ctypes.c_float(scale),
                              R(dq), R(dk), R(dv), ctypes.c_void_p(ws), ctypes.c_size_t(nbytes), None)


def test_chain_bwd_attention_args(cg):
    lib = cg.lib()
    S, C = cg.F_SOFTMAX, cg.MASK_CAUSAL
    q, k, v, o, lse = attn(cg)
    g, dq, dk, dv = (D(cg, (2, 256, 128)) for _ in range(4))
    need = lib.chain_bwd_workspace_size(ctypes.byref(q), ctypes.byref(v))
    assert need == ((2 * 256 * 4 + 255) // 256) * 256
    assert lib.chain_bwd_workspace_size_f(ctypes.byref(q), ctypes.byref(v), S) == need
    assert bwd(cg, g, q, k, v, o, lse, S, C, 0.088, dq, dk, dv, 0x70000000, need) in no_device(cg)
    assert bwd(cg, g, q, k, v, o, lse, S, C, 0.088, dq, dk, dv, 0x70000000, need - 256) == cg.ERR_ARG
    assert bwd(cg, g, q, k, v, o, lse, S, C, 0.088, dq, dk, dv, 0, need) == cg.ERR_ARG
    assert bwd(cg, g, q, k, v, o, lse, 7, C, 0.088, dq, dk, dv, 0x70000000, need) == cg.ERR_ARG
    assert bwd(cg, g, q, k, v, o, lse, S, 2, 0.088, dq, dk, dv, 0x70000000, need) == cg.ERR_ARG
    assert bwd(cg, g, q, k, v, o, lse, S, C, 0.0, dq, dk, dv, 0x70000000, need) == cg.ERR_ARG
    padded = D(cg, (2, 256, 128), strides=(256 * 192, 192, 1))  # the backward takes packed tensors
    assert bwd(cg, g, padded, k, v, o, lse, S, C, 0.088, dq, dk, dv, 0x70000000, need) == cg.ERR_ARG
    assert bwd(cg, g, q, k, v, o, D(cg, (2, 256), cg.F32, strides=(512, 1)), S, C, 0.088,
               dq, dk, dv, 0x70000000, need) == cg.ERR_ARG               # LSE rows not packed
    assert bwd(cg, g, q, k, v, o, lse, S, C, 0.088, dq, D(cg, (2, 256, 128), cg.F32), dv,
               0x70000000, need) == cg.ERR_DTYPE


def test_chain_bwd_mlp_args(cg):
    lib = cg.lib()
    G, N0 = cg.F_GELU_TANH, cg.MASK_NONE
    x, w1, w2, g = D(cg, (128, 256)), D(cg, (256, 512)), D(cg, (512, 256)), D(cg, (128, 256))
    dx, dw1, dw2 = D(cg, (128, 256)), D(cg, (256, 512)), D(cg, (512, 256))
    need = lib.chain_bwd_workspace_size_f(ctypes.byref(x), ctypes.byref(w2), G)
    assert need == 128 * 512 * 4
    assert lib.chain_bwd_workspace_size_f(ctypes.byref(x), ctypes.byref(w2), 7) == 0
    assert bwd(cg, g, x, w1, w2, None, None, G, N0, 1.0, dx, dw1, dw2, 0x70000000, need) in no_device(cg)
    assert bwd(cg, g, x, w1, w2, None, None, G, N0, 1.0, dx, dw1, dw2, 0x70000000, need - 1) == cg.ERR_ARG
    assert bwd(cg, g, x, w1, w2, None, None, G, cg.MASK_CAUSAL, 1.0, dx, dw1, dw2, 0x70000000,
               need) == cg.ERR_ARG
    x192, w192, dx192, dw192 = D(cg, (128, 192)), D(cg, (192, 512)), D(cg, (128, 192)), D(cg, (192, 512))
    assert bwd(cg, g, x192, w192, w2, None, None, G, N0, 1.0, dx192, dw192, dw2, 0x70000000,
               1 << 30) == cg.ERR_UNSUPPORTED                            # K % 256
    # X and W2 of one shape: only f tells the MLP apart from attention
    xs, w2s = D(cg, (4096, 1024)), D(cg, (4096, 1024))
    assert lib.chain_bwd_workspace_size_f(ctypes.byref(xs), ctypes.byref(w2s), G) == 4096 * 4096 * 4


def test_chain_bwd_noalloc_limits(cg):
    lib = cg.lib()
    G, N0 = cg.F_GELU_TANH, cg.MASK_NONE
    xs, w1, w2s, g = D(cg, (4096, 1024)), D(cg, (1024, 4096)), D(cg, (4096, 1024)), D(cg, (4096, 1024))
    dx, dw1, dw2 = D(cg, (4096, 1024)), D(cg, (1024, 4096)), D(cg, (4096, 1024))
    f = ctypes.c_float(1.0)
    assert lib.chain_bwd_noalloc(R(g), R(xs), R(w1), R(w2s), None, None, G, N0, f,
                                 R(dx), R(dw1), R(dw2), None) == cg.ERR_SCRATCH_LIMIT
    assert lib.chain_bwd_noalloc(R(g), R(xs), R(w1), R(w2s), None, None, 7, N0, f,
                                 R(dx), R(dw1), R(dw2), None) == cg.ERR_ARG
    q, k, v, o, lse = attn(cg, BH=9, n=1 << 20)
    assert lib.chain_bwd_noalloc(R(q), R(q), R(k), R(v), R(o), R(lse), cg.F_SOFTMAX, cg.MASK_CAUSAL,
                                 ctypes.c_float(0.088), R(q), R(k), R(v), None) == cg.ERR_SCRATCH_LIMIT


# ------------------------------------------------------------ other forwards
def test_chain_fwd_f16pv_and_fp8_args(cg):
    lib = cg.lib()
    q, k, v, o, lse = attn(cg)
    need = lib.chain_fwd_f16pv_workspace_size(ctypes.byref(q), ctypes.byref(v))
    assert need > 2 * 256 * 128 * 2

    def f16pv(Q, K, V, O, L, nbytes, scale=0.088):
        return lib.chain_fwd_f16pv(R(Q), R(K), R(V), cg.MASK_CAUSAL, ctypes.c_float(scale), R(O), R(L),
                                   ctypes.c_void_p(0x70000000), ctypes.c_size_t(nbytes), None)

    assert f16pv(q, k, v, o, lse, need) in no_device(cg)
    assert f16pv(q, k, v, o, lse, need - 16) == cg.ERR_ARG
    qf, kf, vf, of_, lf = attn(cg, dtype=cg.F32)
    assert f16pv(qf, kf, vf, of_, lf, need) == cg.ERR_DTYPE
    assert f16pv(q, k, v, o, lse, need, scale=-1.0) == cg.ERR_ARG

    def fp8(Q, K, V, O, L, nbytes, v_scale=1.0):
        return lib.chain_fwd_fp8(R(Q), R(K), R(V), cg.MASK_CAUSAL, ctypes.c_float(0.088),
                                 ctypes.c_float(v_scale), R(O), R(L), ctypes.c_void_p(0x70000000),
                                 ctypes.c_size_t(nbytes), None)

    q8, k8, v8 = (D(cg, (2, 256, 128), cg.E4M3) for _ in range(3))
    need8 = lib.chain_fwd_fp8_workspace_size(ctypes.byref(v8))
    assert need8 == 2 * 256 * 128 * 2
    assert fp8(q8, k8, v8, o, lse, need8) in no_device(cg)
    assert fp8(q8, k8, v8, o, lse, need8 - 256) == cg.ERR_ARG
    assert fp8(q8, k8, v8, o, lse, need8, v_scale=math.nan) == cg.ERR_ARG
    assert fp8(q8, k8, v8, D(cg, (2, 256, 128), cg.F32), lse, need8) == cg.ERR_DTYPE
    q64, k64, v64 = (D(cg, (2, 256, 64), cg.E4M3) for _ in range(3))
    assert fp8(q64, k64, v64, D(cg, (2, 256, 64)), lse, 1 << 30) == cg.ERR_UNSUPPORTED
    q96, k96, v96 = (D(cg, (2, 256, 96), cg.E4M3) for _ in range(3))
    assert fp8(q96, k96, v96, D(cg, (2, 256, 96)), lse, 1 << 30) == cg.ERR_ARG


def test_sharded_and_relayout_args(cg):
    lib = cg.lib()
    p, n_loc, H, d = 4, 256, 8, 128
    sh = [D(cg, (p, n_loc, H, d)) for _ in range(4)]
    lse = D(cg, (H // p, p * n_loc), cg.F32)

    def sp(Q, p_, g, L, mask=cg.MASK_CAUSAL):
        return lib.chain_fwd_sp(R(Q), R(sh[1]), R(sh[2]), p_, g, mask, ctypes.c_float(0.088),
                                R(sh[3]), R(L), None)

    assert sp(sh[0], p, 0, lse) in no_device(cg)
    for p_, g in ((p, p), (p, -1), (0, 0), (3, 0)):
        assert sp(sh[0], p_, g, lse) == cg.ERR_ARG                       # group / divisibility
    assert sp(D(cg, (2, 256, 128)), p, 0, lse) == cg.ERR_ARG              # not [p][n_loc][H][d]
    ragged = [D(cg, (p, 100, H, d)) for _ in range(4)]
    assert lib.chain_fwd_sp(R(ragged[0]), R(ragged[1]), R(ragged[2]), p, 0, cg.MASK_CAUSAL,
                            ctypes.c_float(0.088), R(ragged[3]),
                            R(D(cg, (H // p, p * 100), cg.F32)), None) == cg.ERR_UNSUPPORTED
    hm = D(cg, (H // p, p * n_loc, d))

    def rel(S, p_, g, O):
        return lib.sp_relayout(R(S), p_, g, R(O), None)

    assert rel(sh[0], p, 1, hm) in no_device(cg)
    assert lib.sp_relayout_inverse(R(hm), p, 1, R(sh[0]), None) in no_device(cg)
    assert rel(sh[0], p, p, hm) == cg.ERR_ARG
    assert rel(sh[0], 3, 0, D(cg, (2, 3 * n_loc, d))) == cg.ERR_ARG       # H % p
    assert rel(sh[0], p, 0, D(cg, (H // p, p * n_loc, d), cg.F32)) == cg.ERR_DTYPE
    assert rel(sh[0], p, 0, D(cg, (H // p, p * n_loc, d), strides=(p * n_loc * 256, 256, 1))) == cg.ERR_ARG
    assert rel(D(cg, (p, n_loc, H, 4)), p, 0, D(cg, (H // p, p * n_loc, 4))) == cg.ERR_ARG  # 8-byte rows
    assert rel(None, p, 0, hm) == cg.ERR_ARG


def test_varlen_args(cg):
    lib = cg.lib()
    total, H, d = 1000, 4, 128
    q, k, v, o = (D(cg, (total, H, d)) for _ in range(4))
    lse = D(cg, (H, total), cg.F32)
    cu = ctypes.c_void_p(0x60000000)

    def fv(cu_, batch, maxlen, K=k):
        return lib.chain_fwd_varlen(R(q), R(K), R(v), cu_, batch, maxlen, cg.MASK_CAUSAL,
                                    ctypes.c_float(0.088), R(o), R(lse), None)

    assert fv(cu, 3, 500) in no_device(cg)
    assert fv(None, 3, 500) == cg.ERR_ARG                                   # no cu_seqlens
    assert fv(ctypes.c_void_p(0x60000002), 3, 500) == cg.ERR_ARG            # misaligned
    assert fv(cu, 0, 500) == cg.ERR_ARG
    assert fv(cu, 3, total + 1) == cg.ERR_ARG                                # max_seqlen > total
    assert fv(cu, 3, 500, K=D(cg, (total, 3, d))) == cg.ERR_ARG              # K/V heads do not divide
    g, dq, dk, dv = (D(cg, (total, H, d)) for _ in range(4))
    need = ((H * total * 4 + 255) // 256) * 256

    def bv(nbytes, dK=dk):
        return lib.chain_bwd_varlen(R(g), R(q), R(k), R(v), R(o), R(lse), cu, 3, 500, cg.MASK_CAUSAL,
                                    ctypes.c_float(0.088), R(dq), R(dK), R(dv),
                                    ctypes.c_void_p(0x70000000), ctypes.c_size_t(nbytes), None)

    assert bv(need) in no_device(cg)
    assert bv(need - 256) == cg.ERR_ARG
    other = D(cg, (total, H, d), strides=(H * d * 2, d, 1))                 # a second stride pair
    assert bv(need, dK=other) == cg.ERR_ARG


def test_status_and_check_without_device(cg):
    lib = cg.lib()
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.chain_status_string(s)
    assert b"unknown" not in lib.chain_status_string(-7)
    site = ctypes.c_int(0)
    assert lib.chain_check(None, ctypes.byref(site)) in no_device(cg)
