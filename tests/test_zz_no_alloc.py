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
    BH, n, d = 16, 8192, 128  # needs 16*8192*(128+1)*4 bytes > 32 MiB
    q = torch.zeros(BH, n, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(BH, n, dtype=torch.float32, device="cuda")
    assert cg.chain_bwd_workspace_size(q, q) > cg.NOALLOC_SCRATCH_BYTES
    out = [torch.empty_like(q) for _ in range(3)]
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_bwd_noalloc(q, q, q, q, q, lse, cg.F_SOFTMAX, cg.MASK_CAUSAL, 0.1, *out)
    assert ei.value.status == cg.ERR_SCRATCH_LIMIT
