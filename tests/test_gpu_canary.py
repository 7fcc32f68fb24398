"""GPU: canary regions around every output and workspace.

Each output (and each workspace) is a view into a larger device buffer
whose bytes before and after it (and, for row-strided outputs, the gap
between rows) hold a fixed pattern.  After calls on ragged shapes (n = 1,
127, 129, 300; an odd number of heads) the pattern must be intact: no
tensor-memory-accelerator store, vector store or epilogue writes outside the
tensor it was given.  This stands in for a memory checker, which this
library's test runs do not have."""
import math

import numpy as np
import pytest
import torch

import chain_synth as cs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PAT = 0xA5


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


class Guarded:
    """A tensor of `shape`/`dtype` inside a pattern-filled byte buffer.

    With `pad` > 0 the innermost dimension has `pad` extra elements of row
    pitch (a strided view), and those gap elements are checked too."""

    def __init__(self, shape, dtype, pad=0):
        esz = torch.empty((), dtype=dtype).element_size()
        inner = shape[-1] + pad
        full = tuple(shape[:-1]) + (inner,)
        self.nbytes = math.prod(full) * esz
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), PAT, dtype=torch.uint8,
                              device="cuda")
        base = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(full)
        self.t = base[..., :shape[-1]] if pad else base
        self.pad, self.esz, self.full = pad, esz, full

    def check(self, what):
        b = self.buf.cpu().numpy()
        assert np.all(b[:GUARD] == PAT), f"{what}: bytes before the tensor were written"
        assert np.all(b[GUARD + self.nbytes:] == PAT), f"{what}: bytes after the tensor were written"
        if self.pad:
            body = b[GUARD:GUARD + self.nbytes].reshape(-1, self.full[-1] * self.esz)
            gap = body[:, (self.full[-1] - self.pad) * self.esz:]
            assert np.all(gap == PAT), f"{what}: the gap between rows was written"


def _ok(cg):
    rc, site = cg.chain_check()
    assert rc == 0, (rc, hex(site))


RAGGED = [1, 127, 129, 300]


@pytest.mark.parametrize("n", RAGGED)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_canary_attention_forward(cg, n, d, causal):
    BH = 3
    q, k, v = (t.cuda() for t in cs.attn_inputs(BH, n, d, seed=15000 + n + d))
    mask = cg.MASK_CAUSAL if causal else cg.MASK_NONE
    # chain_fwd: O with a row gap, LSE dense
    O = Guarded((BH, n, d), torch.bfloat16, pad=64)
    L = Guarded((BH, n), torch.float32)
    cg.chain_fwd(q, k, v, cg.F_SOFTMAX, mask, d ** -0.5, O.t, L.t)
    _ok(cg)
    O.check("chain_fwd O")
    L.check("chain_fwd LSE")
    # chain_fwd_f16pv: O, LSE and the workspace
    O = Guarded((BH, n, d), torch.bfloat16)
    L = Guarded((BH, n), torch.float32)
    W = Guarded((cg.chain_fwd_f16pv_workspace_size(q, v),), torch.uint8)
    cg.chain_fwd_f16pv(q, k, v, mask, d ** -0.5, O.t, L.t, W.t)
    _ok(cg)
    O.check("chain_fwd_f16pv O")
    L.check("chain_fwd_f16pv LSE")
    W.check("chain_fwd_f16pv workspace")


@pytest.mark.parametrize("n", RAGGED)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_canary_attention_backward(cg, n, d, causal):
    BH = 3
    q, k, v, do = (t.cuda() for t in cs.attn_inputs(BH, n, d, seed=15100 + n + d, with_do=True))
    o, lse = cg.attention_fwd(q, k, v, causal)
    outs = [Guarded((BH, n, d), torch.bfloat16) for _ in range(3)]
    W = Guarded((cg.chain_bwd_workspace_size(q, v),), torch.uint8)
    cg.chain_bwd(do, q, k, v, o, lse, cg.F_SOFTMAX, cg.MASK_CAUSAL if causal else cg.MASK_NONE,
                 d ** -0.5, *(g.t for g in outs), W.t)
    _ok(cg)
    for name, g in zip(("dQ", "dK", "dV"), outs):
        g.check(f"chain_bwd {name}")
    W.check("chain_bwd workspace")


@pytest.mark.parametrize("n", RAGGED)
def test_canary_attention_fp32(cg, n):
    BH, d = 3, 64
    q, k, v = (t.cuda() for t in cs.attn_inputs(BH, n, d, seed=15200 + n, dtype=torch.float32))
    O = Guarded((BH, n, d), torch.float32)
    L = Guarded((BH, n), torch.float32)
    cg.chain_fwd(q, k, v, cg.F_SOFTMAX, cg.MASK_CAUSAL, 0.125, O.t, L.t)
    _ok(cg)
    O.check("fp32 O")
    L.check("fp32 LSE")


@pytest.mark.parametrize("n", [1, 129, 300])
def test_canary_attention_e4m3(cg, n):
    BH = 3
    q, k, v = (t.float().to(torch.float8_e4m3fn).cuda()
               for t in cs.attn_inputs(BH, n, 128, seed=15300 + n, dtype=torch.float32))
    O = Guarded((BH, n, 128), torch.bfloat16)
    L = Guarded((BH, n), torch.float32)
    W = Guarded((cg.chain_fwd_fp8_workspace_size(v),), torch.uint8)
    cg.chain_fwd_fp8(q, k, v, cg.MASK_CAUSAL, 128 ** -0.5, 1.0, O.t, L.t, W.t)
    _ok(cg)
    O.check("e4m3 O")
    L.check("e4m3 LSE")
    W.check("e4m3 workspace")


def test_canary_varlen(cg):
    lens = RAGGED
    total, H, d = sum(lens), 3, 128
    q = cs.normal((total, H, d), 15400).cuda()
    k = cs.normal((total, H, d), 15401).cuda()
    v = cs.normal((total, H, d), 15402).cuda()
    do = cs.normal((total, H, d), 15403).cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
    for f16pv in (False, True):
        O = Guarded((total, H, d), torch.bfloat16)
        L = Guarded((H, total), torch.float32)
        if f16pv:
            W = Guarded((cg.chain_fwd_varlen_f16pv_workspace_size(v),), torch.uint8)
            cg.chain_fwd_varlen_f16pv(q, k, v, cu, len(lens), max(lens), cg.MASK_CAUSAL,
                                      d ** -0.5, O.t, L.t, W.t)
        else:
            cg.chain_fwd_varlen(q, k, v, cu, len(lens), max(lens), cg.MASK_CAUSAL, d ** -0.5,
                                O.t, L.t)
        _ok(cg)
        O.check(f"varlen O (f16pv={f16pv})")
        L.check(f"varlen LSE (f16pv={f16pv})")
        if f16pv:
            W.check("varlen f16pv workspace")
    o, lse = cg.attention_fwd_varlen(q, k, v, cu, max(lens), True)
    outs = [Guarded((total, H, d), torch.bfloat16) for _ in range(3)]
    W = Guarded((cg.chain_bwd_workspace_size(q, q),), torch.uint8)
    cg.chain_bwd_varlen(do, q, k, v, o, lse, cu, len(lens), max(lens), cg.MASK_CAUSAL, d ** -0.5,
                        *(g.t for g in outs), W.t)
    _ok(cg)
    for name, g in zip(("dQ", "dK", "dV"), outs):
        g.check(f"varlen backward {name}")
    W.check("varlen backward workspace")


@pytest.mark.parametrize("n_loc", [1, 3, 127])
def test_canary_relayout(cg, n_loc):
    p, H, d = 4, 12, 64  # three heads per group
    x = cs.iota16((p, n_loc, H, d)).view(torch.bfloat16).cuda()
    out = Guarded((H // p, p * n_loc, d), torch.bfloat16)
    cg.sp_relayout(x, p, 2, out.t)
    _ok(cg)
    out.check("sp_relayout out")
    back = Guarded((p, n_loc, H, d), torch.bfloat16)
    back.t.copy_(x)
    cg.sp_relayout_inverse(out.t, p, 2, back.t)
    _ok(cg)
    back.check("sp_relayout_inverse shards")
    assert torch.equal(back.t.view(torch.int16), x.view(torch.int16))


def test_canary_attention_sp(cg):
    p, n_loc, H, d, g = 4, 128, 12, 128, 1
    q, k, v = (cs.normal((p, n_loc, H, d), seed=15500 + i).cuda() for i in range(3))
    O = Guarded((p, n_loc, H, d), torch.bfloat16)
    O.t.zero_()
    L = Guarded((H // p, p * n_loc), torch.float32)
    cg.chain_fwd_sp(q, k, v, p, g, cg.MASK_CAUSAL, d ** -0.5, O.t, L.t)
    _ok(cg)
    O.check("chain_fwd_sp O")
    L.check("chain_fwd_sp LSE")
    O = Guarded((p, n_loc, H, d), torch.bfloat16)
    L = Guarded((H // p, p * n_loc), torch.float32)
    W = Guarded((cg.chain_fwd_sp_f16pv_workspace_size(v, p),), torch.uint8)
    cg.chain_fwd_sp_f16pv(q, k, v, p, g, cg.MASK_CAUSAL, d ** -0.5, O.t, L.t, W.t)
    _ok(cg)
    O.check("chain_fwd_sp_f16pv O")
    L.check("chain_fwd_sp_f16pv LSE")
    W.check("chain_fwd_sp_f16pv workspace")


def test_canary_mlp(cg):
    M, K, N, P = 128, 64, 128, 256
    x, w1, w2 = (t.cuda() for t in cs.mlp_inputs(M, K, N, P, seed=15600))
    O = Guarded((M, P), torch.bfloat16)
    cg.chain_fwd(x, w1, w2, cg.F_GELU_TANH, cg.MASK_NONE, 1.0, O.t)
    _ok(cg)
    O.check("MLP chain_fwd O")
    M, K, N, P = 128, 64, 64, 512
    x, w1, w2 = (t.cuda() for t in cs.mlp_inputs(M, K, N, P, seed=15610))
    O = Guarded((M, P), torch.bfloat16)
    W = Guarded((cg.chain_fwd_f16h_workspace_size(w2),), torch.uint8)
    cg.chain_fwd_f16h(x, w1, w2, cg.F_GELU_TANH, O.t, W.t)
    _ok(cg)
    O.check("chain_fwd_f16h O")
    W.check("chain_fwd_f16h workspace")
    M, K, N, P = 128, 256, 256, 256
    x, w1, w2 = (t.cuda() for t in cs.mlp_inputs(M, K, N, P, seed=15620))
    do = cs.normal((M, P), 15623).cuda()
    outs = [Guarded(tuple(t.shape), torch.bfloat16) for t in (x, w1, w2)]
    W = Guarded((cg.chain_bwd_workspace_size_f(x, w2, cg.F_GELU_TANH),), torch.uint8)
    cg.chain_bwd(do, x, w1, w2, None, None, cg.F_GELU_TANH, cg.MASK_NONE, 1.0,
                 *(g.t for g in outs), W.t)
    _ok(cg)
    for name, g in zip(("dX", "dW1", "dW2"), outs):
        g.check(f"MLP backward {name}")
    W.check("MLP backward workspace")
