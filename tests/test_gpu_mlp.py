"""GPU: the MLP instance of O = f(A B) C (GeLU tanh and identity) against
the fp64 oracle."""
import numpy as np
import pytest
import torch

import chain_synth as cs
from tol import assert_fwd_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


CASES = [(128, 64, 128, 256), (256, 128, 256, 256), (384, 192, 384, 512), (256, 1024, 640, 768)]


@pytest.mark.parametrize("gelu", [True, False])
@pytest.mark.parametrize("M,K,N,P", CASES)
def test_mlp_small_vs_oracle(cg, orc, M, K, N, P, gelu):
    x, w1, w2 = cs.mlp_inputs(M, K, N, P, seed=2000 + M + K + N + P)
    o = cg.mlp_chain_fwd(x.cuda(), w1.cuda(), w2.cuda(), gelu=gelu)
    assert cg.chain_check()[0] == 0
    ref = orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH if gelu else orc.F_IDENTITY)
    assert_fwd_close(o, ref, f"mlp {M}x{K}x{N}x{P} gelu={gelu}")


def test_identity_chain_associativity(cg, orc):
    # f = identity: the fused (A B) C equals A (B C) computed by the oracle
    # in the other association.
    x, w1, w2 = cs.mlp_inputs(256, 128, 384, 256, seed=2100)
    o = cg.mlp_chain_fwd(x.cuda(), w1.cuda(), w2.cuda(), gelu=False)
    bc = orc.chain_fwd(w1, w2, torch.eye(256, dtype=torch.bfloat16), orc.F_IDENTITY)
    ref = x.double().numpy() @ bc
    assert_fwd_close(o, ref, "A(BC)")


def test_gelu_chain_with_identity_c(cg, orc):
    # C = I: O = GeLU(A B) elementwise (then rounded to bf16).
    x, w1, _ = cs.mlp_inputs(128, 256, 256, 256, seed=2200)
    eye = torch.eye(256, dtype=torch.bfloat16)
    o = cg.mlp_chain_fwd(x.cuda(), w1.cuda(), eye.cuda(), gelu=True)
    t = x.double() @ w1.double()
    ref = torch.nn.functional.gelu(t, approximate="tanh").numpy()
    assert_fwd_close(o, ref, "gelu(AB)")


def test_mlp_full_size_sampled(cg, orc):
    wl = cs.WORKLOADS["gelu_mlp"]
    dm = wl.dims
    x, w1, w2 = cs.mlp_inputs(dm["M"], dm["K"], dm["N"], dm["P"], seed=wl.seed)
    o = cg.mlp_chain_fwd(x.cuda(), w1.cuda(), w2.cuda(), gelu=True)
    assert cg.chain_check()[0] == 0
    g = torch.Generator().manual_seed(5)
    rows = sorted(set([0, 1, 127, 128, dm["M"] - 1] + torch.randint(0, dm["M"], (123,), generator=g).tolist()))
    ref = orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH, rows=rows)
    assert_fwd_close(o.cpu()[rows], ref, "mlp 4096 sampled")


def test_mlp_rejects_unsupported_shapes(cg):
    x = torch.zeros(100, 64, dtype=torch.bfloat16, device="cuda")
    w1 = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.mlp_chain_fwd(x, w1, w2)
    assert ei.value.status == cg.ERR_UNSUPPORTED
