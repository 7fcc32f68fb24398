"""GPU: backward of the MLP chain O = f(X W1) W2 (GeLU tanh and identity),
the intermediate recomputed, against the fp64 oracle."""
import numpy as np
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


def _inputs(M, K, N, P, seed):
    x, w1, w2 = cs.mlp_inputs(M, K, N, P, seed=seed)
    do = cs.normal((M, P), seed + 3)
    return x, w1, w2, do


CASES = [(128, 256, 256, 256), (256, 256, 512, 256), (384, 512, 256, 512)]


@pytest.mark.parametrize("gelu", [True, False])
@pytest.mark.parametrize("M,K,N,P", CASES)
def test_mlp_bwd_small_vs_oracle(cg, orc, M, K, N, P, gelu):
    x, w1, w2, do = _inputs(M, K, N, P, seed=3000 + M + K + N + P)
    dx, dw1, dw2 = cg.mlp_chain_bwd(do.cuda(), x.cuda(), w1.cuda(), w2.cuda(), gelu=gelu)
    assert cg.chain_check()[0] == 0
    rA, rB, rC = orc.chain_bwd(x, w1, w2, do, orc.F_GELU_TANH if gelu else orc.F_IDENTITY)
    tag = f"{M}x{K}x{N}x{P} gelu={gelu}"
    assert_grad_close(dx, rA, "dX " + tag)
    assert_grad_close(dw1, rB.T, "dW1 " + tag)
    assert_grad_close(dw2, rC, "dW2 " + tag)


def test_mlp_bwd_identity_vs_fp32_products(cg):
    # f = identity: dX = dO W2^T W1^T, dW1 = X^T dO W2^T, dW2 = (X W1)^T dO,
    # formed here with fp32 products on the GPU in the other association.
    x, w1, w2, do = (t.cuda() for t in _inputs(256, 512, 512, 256, seed=3100))
    dx, dw1, dw2 = cg.mlp_chain_bwd(do, x, w1, w2, gelu=False)
    xf, w1f, w2f, dof = (t.float() for t in (x, w1, w2, do))
    assert_grad_close(dx, dof @ w2f.T @ w1f.T, "dX")
    assert_grad_close(dw1, xf.T @ (dof @ w2f.T), "dW1")
    assert_grad_close(dw2, (xf @ w1f).T @ dof, "dW2")


def test_mlp_bwd_twice_same_result(cg):
    # deterministic: no atomics, the same bits on a second call
    x, w1, w2, do = (t.cuda() for t in _inputs(256, 256, 256, 256, seed=3200))
    a = cg.mlp_chain_bwd(do, x, w1, w2)
    b = cg.mlp_chain_bwd(do, x, w1, w2)
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


def test_mlp_bwd_rejects_bad_args(cg):
    x = torch.zeros(128, 192, dtype=torch.bfloat16, device="cuda")   # K % 256
    w1 = torch.zeros(192, 256, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    do = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as e:
        cg.mlp_chain_bwd(do, x, w1, w2)
    assert e.value.status == cg.ERR_UNSUPPORTED
    x = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    w1 = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")             # too small
    with pytest.raises(cg.ChainError) as e:
        cg.mlp_chain_bwd(do, x, w1, w2, workspace=ws)
    assert e.value.status == cg.ERR_ARG
    dx, dw1, dw2 = torch.empty_like(x), torch.empty_like(w1), torch.empty_like(w2)
    big = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError) as e:                             # causal mask
        cg.chain_bwd(do, x, w1, w2, None, None, cg.F_GELU_TANH, cg.MASK_CAUSAL, 1.0,
                     dx, dw1, dw2, big)
    assert e.value.status == cg.ERR_ARG


def test_mlp_bwd_full_size_sampled(cg, orc):
    # The GeLU MLP workload, X [4096][1024], W1 [1024][4096], W2 [4096][1024],
    # dO [4096][1024] ~ N(0,1): sampled rows of dX and hidden units of dW1, dW2.
    wl = cs.WORKLOADS["gelu_mlp"]
    dm = wl.dims
    M, K, N, P = dm["M"], dm["K"], dm["N"], dm["P"]
    x, w1, w2 = cs.mlp_inputs(M, K, N, P, seed=wl.seed)
    do = cs.normal((M, P), wl.seed + 3)
    dx, dw1, dw2 = cg.mlp_chain_bwd(do.cuda(), x.cuda(), w1.cuda(), w2.cuda())
    assert cg.chain_check()[0] == 0
    g = np.random.default_rng(77)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M - 1], g.integers(0, M, 27)]))
    hid = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 12)]))
    rA, rB, rC = orc.chain_bwd(x, w1, w2, do, orc.F_GELU_TANH, rows=rows, hidden=hid)
    assert_grad_close(dx.cpu()[rows], rA, "dX rows")
    assert_grad_close(dw1.cpu()[:, hid].T, rB, "dW1 columns")
    assert_grad_close(dw2.cpu()[hid], rC, "dW2 rows")
