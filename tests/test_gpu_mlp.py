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


# ------------------------------------------------- f16 intermediate (f16h)
F16H_CASES = [(128, 64, 64, 512), (256, 128, 320, 768), (384, 192, 384, 1024), (256, 1024, 640, 768)]


@pytest.mark.parametrize("gelu", [True, False])
@pytest.mark.parametrize("M,K,N,P", F16H_CASES)
def test_mlp_f16h_small_vs_oracle(cg, orc, M, K, N, P, gelu):
    x, w1, w2 = cs.mlp_inputs(M, K, N, P, seed=2300 + M + K + N + P)
    o = cg.mlp_chain_fwd_f16h(x.cuda(), w1.cuda(), w2.cuda(), gelu=gelu)
    assert cg.chain_check()[0] == 0
    ref = orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH if gelu else orc.F_IDENTITY)
    assert_fwd_close(o, ref, f"f16h {M}x{K}x{N}x{P} gelu={gelu}")


def test_mlp_f16h_full_size_sampled(cg, orc):
    wl = cs.WORKLOADS["gelu_mlp"]
    dm = wl.dims
    x, w1, w2 = cs.mlp_inputs(dm["M"], dm["K"], dm["N"], dm["P"], seed=wl.seed)
    o = cg.mlp_chain_fwd_f16h(x.cuda(), w1.cuda(), w2.cuda(), gelu=True)
    assert cg.chain_check()[0] == 0
    g = torch.Generator().manual_seed(6)
    rows = sorted(set([0, 1, 127, 128, dm["M"] - 1] + torch.randint(0, dm["M"], (123,), generator=g).tolist()))
    ref = orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH, rows=rows)
    assert_fwd_close(o.cpu()[rows], ref, "f16h 4096 sampled")


@pytest.mark.parametrize("w2_scale", [2.0 ** 30, 2.0 ** -40])
def test_mlp_f16h_c_far_from_f16_range(cg, orc, w2_scale):
    # C scaled far outside f16's range (2^30 x): its copy takes its own power
    # of two, so the result stays within the forward bound
    x, w1, w2 = cs.mlp_inputs(256, 128, 256, 512, seed=2400)
    w2 = (w2.float() * w2_scale).to(torch.bfloat16)
    o = cg.mlp_chain_fwd_f16h(x.cuda(), w1.cuda(), w2.cuda(), gelu=True)
    assert cg.chain_check()[0] == 0
    ref = orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH)
    assert_fwd_close(o, ref, f"f16h C x {w2_scale}")


def test_mlp_f16h_back_to_back_calls_share_a_workspace(cg, orc):
    # A call's main kernel overlaps its own pre-pass; the next call's pre-pass
    # rewrites the same f16 copy and scale.  Two calls issued back to back
    # (no synchronisation between them), with C differing by 2^10, must each
    # match the oracle.
    x, w1, w2 = cs.mlp_inputs(256, 128, 512, 512, seed=2450)
    w2b = (w2.float() * 1024.0).to(torch.bfloat16)
    xd, w1d = x.cuda(), w1.cuda()
    w2d, w2bd = w2.cuda(), w2b.cuda()
    ws = torch.empty(cg.chain_fwd_f16h_workspace_size(w2d), dtype=torch.uint8, device="cuda")
    oa = torch.empty(256, 512, dtype=torch.bfloat16, device="cuda")
    ob = torch.empty_like(oa)
    for _ in range(3):
        cg.chain_fwd_f16h(xd, w1d, w2d, cg.F_GELU_TANH, oa, ws)
        cg.chain_fwd_f16h(xd, w1d, w2bd, cg.F_GELU_TANH, ob, ws)
    assert cg.chain_check()[0] == 0
    assert_fwd_close(oa, orc.chain_fwd(x, w1, w2, orc.F_GELU_TANH), "first call")
    assert_fwd_close(ob, orc.chain_fwd(x, w1, w2b, orc.F_GELU_TANH), "second call")


def test_mlp_f16h_matches_compensated_form(cg):
    # the two forms of the same chain agree to within their rounding
    x, w1, w2 = cs.mlp_inputs(512, 256, 512, 1024, seed=2500)
    xd, w1d, w2d = x.cuda(), w1.cuda(), w2.cuda()
    a = cg.mlp_chain_fwd_f16h(xd, w1d, w2d, gelu=True).float()
    b = cg.mlp_chain_fwd(xd, w1d, w2d, gelu=True).float()
    assert float((a - b).abs().max()) <= 1e-2 * float(b.abs().max())


def test_mlp_f16h_intermediate_beyond_f16_is_reported(cg):
    # X W1 of about 1e5: GeLU of it is beyond f16's largest finite value
    x, w1, w2 = cs.mlp_inputs(128, 64, 64, 512, seed=2600)
    x = torch.full_like(x, 64.0)
    w1 = torch.full_like(w1, 32.0)  # T = 64 * 32 * 64 = 131072
    cg.mlp_chain_fwd_f16h(x.cuda(), w1.cuda(), w2.cuda(), gelu=False)
    rc, _ = cg.chain_check()
    assert rc == cg.ERR_ARG
    assert cg.chain_check()[0] == 0


def test_mlp_f16h_rejects_bad_args(cg):
    x = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    w1 = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")  # P = 256: no cluster
    with pytest.raises(cg.ChainError) as ei:
        cg.mlp_chain_fwd_f16h(x, w1, w2)
    assert ei.value.status == cg.ERR_UNSUPPORTED
    w2 = torch.zeros(128, 512, dtype=torch.bfloat16, device="cuda")
    need = cg.chain_fwd_f16h_workspace_size(w2)
    assert need >= 128 * 512 * 2
    o = torch.empty(128, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_f16h(x, w1, w2, cg.F_GELU_TANH, o,
                          torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == cg.ERR_ARG
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_f16h(x, w1, w2, cg.F_SOFTMAX, o, ws)
    assert ei.value.status == cg.ERR_ARG
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_f16h(x.float(), w1, w2, cg.F_GELU_TANH, o, ws)
    assert ei.value.status == cg.ERR_DTYPE
