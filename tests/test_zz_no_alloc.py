"""GPU: chain_bwd_noalloc, the backward entry point for callers that cannot
allocate device memory, against the existing chain_bwd entry point and
against the fp64 oracle.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It passes alone in a fresh
process and after the other tests (the scratch array keeps whatever the last
call left there; every call must re-initialise what it reads)."""
import ctypes
import math

import pytest
import torch

import chain_synth as cs
from tol import assert_grad_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


def test_noalloc_matches_chain_bwd_and_oracle_on_two_calls(cg, orc):
    # Two attention backwards in a row through the fixed scratch array, one
    # causal and one not, each against chain_bwd with a caller workspace and
    # against the oracle's textbook chain rule.
    for call, (BH, n, d, causal) in enumerate([(2, 1000, 128, True), (3, 520, 64, False)]):
        qc, kc, vc, doc = cs.attn_inputs(BH, n, d, seed=12000 + call, with_do=True)
        q, k, v, do = (t.cuda() for t in (qc, kc, vc, doc))
        scale = 1.0 / math.sqrt(d)
        o, lse = cg.attention_fwd(q, k, v, causal, scale)
        ref = cg.attention_bwd(do, q, k, v, o, lse, causal, scale)  # caller-provided workspace
        got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        cg.chain_bwd_noalloc(do, q, k, v, o, lse, cg.F_SOFTMAX,
                             cg.MASK_CAUSAL if causal else cg.MASK_NONE, scale, *got)
        rc, site = cg.chain_check()
        assert rc == 0, (rc, hex(site))
        orc_ref = orc.softmax_bwd(qc, kc, vc, doc, scale, causal)[:3]
        for name, g_, r_, o_ in zip(("dQ", "dK", "dV"), got, ref, orc_ref):
            assert_grad_close(g_.cpu(), r_.cpu(), f"{name} call {call} vs chain_bwd")
            assert_grad_close(g_.cpu(), o_, f"{name} call {call} vs oracle")


@pytest.mark.parametrize("gelu", [True, False])
def test_noalloc_mlp_matches_chain_bwd_and_oracle(cg, orc, gelu):
    # The MLP backward keeps H and dT in the scratch array; two calls in a row
    # on different inputs, each against chain_bwd and the oracle.
    f = cg.F_GELU_TANH if gelu else cg.F_IDENTITY
    for call in range(2):
        M, K, N, P = 256, 256, 256, 256
        xc, w1c, w2c = cs.mlp_inputs(M, K, N, P, seed=12100 + 10 * call + gelu)
        doc = cs.normal((M, P), 12150 + 10 * call + gelu)
        x, w1, w2, do = (t.cuda() for t in (xc, w1c, w2c, doc))
        ref = cg.mlp_chain_bwd(do, x, w1, w2, gelu=gelu)
        got = [torch.empty_like(x), torch.empty_like(w1), torch.empty_like(w2)]
        cg.chain_bwd_noalloc(do, x, w1, w2, None, None, f, cg.MASK_NONE, 1.0, *got)
        rc, site = cg.chain_check()
        assert rc == 0, (rc, hex(site))
        rA, rB, rC = orc.chain_bwd(xc, w1c, w2c, doc, orc.F_GELU_TANH if gelu else orc.F_IDENTITY)
        for name, g_, r_, o_ in zip(("dX", "dW1", "dW2"), got, ref, (rA, rB.T, rC)):
            assert_grad_close(g_.cpu(), r_.cpu(), f"{name} call {call} vs chain_bwd")
            assert_grad_close(g_.cpu(), o_, f"{name} call {call} vs oracle")


def _desc_3d(cg, t, BH, n, d):
    # A descriptor of [BH][n][d] over a small buffer: the size checks run on
    # the host before any memory is touched, so it may describe more rows
    # than the buffer holds.
    x = cg.desc(t)
    x.ndim = 3
    x.shape[0], x.shape[1], x.shape[2] = BH, n, d
    x.stride[0], x.stride[1], x.stride[2] = n * d, d, 1
    return x


def test_noalloc_rejects_attention_beyond_scratch(cg):
    # 9 * 2^20 query rows need a 36 MiB row term: more than the 32 MiB array.
    q = torch.zeros(1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 128, dtype=torch.float32, device="cuda")
    BH, n = 9, 1 << 20
    ds = [_desc_3d(cg, q, BH, n, 128) for _ in range(8)]
    dl = cg.desc(lse)
    dl.ndim, dl.shape[0], dl.shape[1], dl.stride[0], dl.stride[1] = 2, BH, n, n, 1
    assert cg.lib().chain_bwd_workspace_size(ctypes.byref(ds[1]), ctypes.byref(ds[3])) > \
        cg.NOALLOC_SCRATCH_BYTES
    rc = cg.lib().chain_bwd_noalloc(*(ctypes.byref(d) for d in ds[:5]), ctypes.byref(dl),
                                    cg.F_SOFTMAX, cg.MASK_CAUSAL, ctypes.c_float(0.1),
                                    *(ctypes.byref(d) for d in ds[5:]), None)
    assert rc == cg.ERR_SCRATCH_LIMIT


def test_noalloc_rejects_mlp_beyond_scratch(cg):
    # The GeLU MLP workload's shapes: X and W2 are both [4096][1024], so only
    # f tells it from attention.  Its H and dT need 4096 * 4096 * 4 bytes =
    # 64 MiB, more than the array: refused before anything is enqueued.
    x = torch.zeros(4096, 1024, dtype=torch.bfloat16, device="cuda")
    w1 = torch.zeros(1024, 4096, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(4096, 1024, dtype=torch.bfloat16, device="cuda")
    do = torch.zeros(4096, 1024, dtype=torch.bfloat16, device="cuda")
    assert cg.chain_bwd_workspace_size_f(x, w2, cg.F_GELU_TANH) > cg.NOALLOC_SCRATCH_BYTES
    dx, dw1, dw2 = torch.empty_like(x), torch.empty_like(w1), torch.empty_like(w2)
    for f in (cg.F_GELU_TANH, cg.F_IDENTITY):
        with pytest.raises(cg.ChainError) as e:
            cg.chain_bwd_noalloc(do, x, w1, w2, None, None, f, cg.MASK_NONE, 1.0, dx, dw1, dw2)
        assert e.value.status == cg.ERR_SCRATCH_LIMIT
