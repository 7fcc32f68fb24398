"""GPU: the tensor-core building block and the bounded-wait failure path."""
import numpy as np
import pytest
import torch

import chain_synth as cs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


@pytest.mark.parametrize("a_tmem", [False, True])
@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("K", [64, 128, 256])
@pytest.mark.parametrize("b_mn", [0, 1])
def test_umma_building_block(cg, orc, N, K, b_mn, a_tmem):
    # D = A B^T (B given [N][K]) or D = A B (B given [K][N]); checked against
    # the oracle's identity chain with C = I.
    A = cs.normal((128, K), seed=500 + K)
    Bs = cs.normal((K, N) if b_mn else (N, K), seed=600 + N)
    D = torch.full((128, N), float("nan"), device="cuda")
    cg.umma_selftest(A.cuda(), Bs.cuda(), D, N, K, b_mn, a_tmem)
    assert cg.chain_check()[0] == 0
    Bkn = Bs if b_mn else Bs.t().contiguous()
    ref = orc.chain_fwd(A, Bkn, torch.eye(N, dtype=torch.bfloat16), orc.F_IDENTITY)
    got = D.cpu().double().numpy()
    # exact bf16 products summed in fp32: tiny relative error
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


def test_bounded_wait_expires_and_reports(cg):
    cg.selftest_wait_timeout(5_000_000)  # 5 ms
    rc, site = cg.chain_check()
    assert rc == cg.ERR_TIMEOUT and site == 0x901
    # the status word is cleared and the context stays usable
    assert cg.chain_check()[0] == 0
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
