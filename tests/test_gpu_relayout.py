"""GPU: Ulysses relayout, bit-exact against the oracle."""
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


@pytest.mark.parametrize("p,n_loc,H,d,g", [
    (4, 37, 8, 128, 0), (4, 37, 8, 128, 3), (2, 5, 6, 64, 1), (4, 1, 4, 8, 2), (1, 19, 3, 128, 0),
    # more positions than one grid pass, 2 KB rows, a group of 512 heads
    (4, 300, 8, 128, 1), (2, 16, 4, 1024, 1), (1, 7, 512, 8, 0)])
def test_relayout_iota_bit_exact(cg, orc, p, n_loc, H, d, g):
    x = cs.iota16((p, n_loc, H, d))
    out = cg.relayout(x.cuda(), p, g)
    assert cg.chain_check()[0] == 0
    ref, shape = orc.relayout(x, p, g)
    assert tuple(out.shape) == shape
    assert np.array_equal(out.cpu().view(torch.uint8).numpy().reshape(-1), ref)


def test_relayout_fp32_payload(cg, orc):
    x = cs.normal((4, 33, 8, 32), seed=7, dtype=torch.float32)
    out = cg.relayout(x.cuda(), 4, 1)
    ref, _ = orc.relayout(x, 4, 1)
    assert np.array_equal(out.cpu().view(torch.uint8).numpy().reshape(-1), ref)


def test_relayout_inverse_round_trip(cg, orc):
    p, n_loc, H, d = 4, 64, 8, 128
    x = cs.normal((p, n_loc, H, d), seed=8)
    xd = x.cuda()
    back = torch.zeros_like(xd)
    for g in range(p):
        hm = cg.relayout(xd, p, g)
        cg.sp_relayout_inverse(hm, p, g, back)
        ref = orc.relayout_inverse(hm.cpu(), p, n_loc, H, g)
        # the oracle writes group g only; compare those heads
        got = back.cpu().view(torch.uint8).numpy().reshape(p, n_loc, H, d * 2)
        r = ref.reshape(p, n_loc, H, d * 2)
        Hl = H // p
        assert np.array_equal(got[:, :, g * Hl:(g + 1) * Hl], r[:, :, g * Hl:(g + 1) * Hl])
    assert torch.equal(back.view(torch.int16), xd.view(torch.int16))


def test_relayout_rejects_bad_args(cg):
    x = torch.zeros(4, 8, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(3, 32, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.sp_relayout(x, 4, 0, out)  # wrong head count in out (8/4 = 2 expected)
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.sp_relayout(x, 4, 4, out)  # group out of range
    odd = torch.zeros(4, 8, 8, 4, dtype=torch.bfloat16, device="cuda")  # 8-byte rows
    with pytest.raises(cg.ChainError):
        cg.sp_relayout(odd, 4, 0, torch.empty(2, 32, 4, dtype=torch.bfloat16, device="cuda"))


def test_relayout_ulysses_full_size_bit_exact(cg, orc):
    # 4 shards [32768][32][128] bf16 -> [8][131072][128], group 0 (and 3).
    wl = cs.WORKLOADS["ulysses_128k"].dims
    x = cs.shard_inputs(wl["p"], wl["n_loc"], wl["H"], wl["d"], seed=4000)
    xd = x.cuda()
    for g in (0, 3):
        out = cg.relayout(xd, wl["p"], g)
        assert cg.chain_check()[0] == 0
        ref, shape = orc.relayout(x, wl["p"], g)
        assert np.array_equal(out.cpu().view(torch.uint8).numpy().reshape(-1), ref)
