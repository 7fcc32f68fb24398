"""GPU: chain_bwd_noalloc, the backward entry point for callers that cannot
allocate device memory, against the existing chain_bwd entry point.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It passes alone in a fresh
process and after the other tests (the scratch array keeps whatever the last
call left there; every call must re-initialise what it reads)."""
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


def test_noalloc_matches_chain_bwd_on_two_calls(cg):
    for call, (BH, n, d, causal) in enumerate([(2, 1000, 128, True), (3, 520, 64, False)]):
        q, k, v, do = (t.cuda() for t in cs.attn_inputs(BH, n, d, seed=12000 + call, with_do=True))
        scale = 1.0 / math.sqrt(d)
        o, lse = cg.attention_fwd(q, k, v, causal, scale)
        ref = cg.attention_bwd(do, q, k, v, o, lse, causal, scale)  # caller-provided workspace
        got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        cg.chain_bwd_noalloc(do, q, k, v, o, lse, cg.F_SOFTMAX,
                             cg.MASK_CAUSAL if causal else cg.MASK_NONE, scale, *got)
        rc, site = cg.chain_check()
        assert rc == 0, (rc, hex(site))
        for name, g_, r_ in zip(("dQ", "dK", "dV"), got, ref):
            assert_grad_close(g_.cpu(), r_.cpu(), f"{name} call {call}")


def test_noalloc_rejects_problem_beyond_scratch(cg):
    # A problem whose row term needs more than the fixed scratch: 9 * 2^20
    # rows of d = 128 (the descriptors are checked before any memory is
    # touched, so they may describe more rows than the buffers hold).
    import ctypes
    q = torch.zeros(1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 128, dtype=torch.float32, device="cuda")
    BH, n = 9, 1 << 20

    def big(t, lse_like=False):
        d = cg.desc(t)
        if lse_like:
            d.ndim, d.shape[0], d.shape[1], d.stride[0], d.stride[1] = 2, BH, n, n, 1
        else:
            d.ndim = 3
            d.shape[0], d.shape[1], d.shape[2] = BH, n, 128
            d.stride[0], d.stride[1], d.stride[2] = n * 128, 128, 1
        return d

    ds = [big(q) for _ in range(8)]
    dl = big(lse, lse_like=True)
    assert cg.lib().chain_bwd_workspace_size(ctypes.byref(ds[1]), ctypes.byref(ds[3])) > \
        cg.NOALLOC_SCRATCH_BYTES
    rc = cg.lib().chain_bwd_noalloc(*(ctypes.byref(d) for d in ds[:5]), ctypes.byref(dl),
                                    cg.F_SOFTMAX, cg.MASK_CAUSAL, ctypes.c_float(0.1),
                                    *(ctypes.byref(d) for d in ds[5:]), None)
    assert rc == cg.ERR_SCRATCH_LIMIT
