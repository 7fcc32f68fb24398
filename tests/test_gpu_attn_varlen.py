"""GPU: attention over sequences of different lengths packed end to end
(chain_fwd_varlen), against chain_fwd on each sequence alone (bit for bit)
and the oracle."""
import numpy as np
import pytest
import torch

import chain_synth as cs
from tol import assert_fwd_close, assert_grad_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


LENS = [300, 1, 129, 512, 77, 256]


def _packed(lens, H, Hkv, d, seed):
    total = sum(lens)
    q = cs.normal((total, H, d), seed)
    k = cs.normal((total, Hkv, d), seed + 1)
    v = cs.normal((total, Hkv, d), seed + 2)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return q, k, v, cu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 128), (4, 2, 64), (6, 3, 128)])
def test_varlen_matches_each_sequence_alone(cg, H, Hkv, d, causal):
    q, k, v, cu = _packed(LENS, H, Hkv, d, seed=8400 + H + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cg.attention_fwd_varlen(qd, kd, vd, cu.cuda(), max(LENS), causal)
    assert cg.chain_check()[0] == 0
    for b, L in enumerate(LENS):
        lo, hi = int(cu[b]), int(cu[b + 1])
        # the same sequence alone, head-major [H][L][d]
        oa, la = cg.attention_fwd(qd[lo:hi].transpose(0, 1).contiguous(),
                                  kd[lo:hi].transpose(0, 1).contiguous(),
                                  vd[lo:hi].transpose(0, 1).contiguous(), causal)
        assert torch.equal(o[lo:hi].transpose(0, 1).contiguous().view(torch.int16),
                           oa.view(torch.int16)), f"O of sequence {b}"
        assert torch.equal(lse[:, lo:hi].contiguous().view(torch.int32),
                           la.view(torch.int32)), f"LSE of sequence {b}"


def test_varlen_vs_oracle(cg, orc):
    H, Hkv, d = 4, 2, 128
    q, k, v, cu = _packed(LENS, H, Hkv, d, seed=8500)
    o, lse = cg.attention_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(LENS), True)
    assert cg.chain_check()[0] == 0
    G = H // Hkv
    for b in range(len(LENS)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        qs = q[lo:hi].transpose(0, 1).contiguous()
        ks = k[lo:hi].transpose(0, 1).repeat_interleave(G, 0).contiguous()
        vs = v[lo:hi].transpose(0, 1).repeat_interleave(G, 0).contiguous()
        ro, rl = orc.softmax_fwd(qs, ks, vs, d ** -0.5, True)
        assert_fwd_close(o.cpu()[lo:hi].transpose(0, 1), ro, f"varlen O seq {b}")
        assert_lse_close(lse.cpu()[:, lo:hi], rl, f"varlen LSE seq {b}")


def test_varlen_sequence_longer_than_max_is_reported(cg):
    q, k, v, cu = _packed([300, 40], 2, 2, 128, seed=8600)
    cg.attention_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), 256, True)
    rc, _ = cg.chain_check()
    assert rc == cg.ERR_ARG
    assert cg.chain_check()[0] == 0  # the report is cleared


def test_varlen_offsets_clamped_to_the_tensor(cg):
    # offsets past the packed rows are clamped on the device: no access
    # outside the tensors, and the in-range sequence is still right
    q, k, v, _ = _packed([128, 128], 2, 2, 128, seed=8700)
    cu = torch.tensor([0, 128, 999], dtype=torch.int32, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, _ = cg.attention_fwd_varlen(qd, kd, vd, cu, 256, False)
    assert cg.chain_check()[0] == 0
    oa, _ = cg.attention_fwd(qd[:128].transpose(0, 1).contiguous(), kd[:128].transpose(0, 1).contiguous(),
                             vd[:128].transpose(0, 1).contiguous(), False)
    assert torch.equal(o[:128].transpose(0, 1).contiguous().view(torch.int16), oa.view(torch.int16))


def test_varlen_rejects_bad_args(cg):
    q = torch.zeros(64, 2, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.attention_fwd_varlen(q, q, q, cu, 65, True)       # max_seqlen > total
    k = torch.zeros(64, 3, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.attention_fwd_varlen(q, k, k, cu, 64, True)        # 2 % 3 != 0


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 128), (4, 2, 64)])
def test_varlen_bwd_matches_each_sequence_alone(cg, H, Hkv, d, causal):
    q, k, v, cu = _packed(LENS, H, Hkv, d, seed=8800 + H + d)
    do = cs.normal(tuple(q.shape), 8899)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    o, lse = cg.attention_fwd_varlen(qd, kd, vd, cud, max(LENS), causal)
    dq, dk, dv = cg.attention_bwd_varlen(dod, qd, kd, vd, o, lse, cud, max(LENS), causal)
    assert cg.chain_check()[0] == 0
    hm = lambda x, lo, hi: x[lo:hi].transpose(0, 1).contiguous()
    for b, L in enumerate(LENS):
        lo, hi = int(cu[b]), int(cu[b + 1])
        oa, la = cg.attention_fwd(hm(qd, lo, hi), hm(kd, lo, hi), hm(vd, lo, hi), causal)
        ga = cg.attention_bwd(hm(dod, lo, hi), hm(qd, lo, hi), hm(kd, lo, hi), hm(vd, lo, hi), oa, la,
                              causal)
        for name, got, ref in (("dQ", dq, ga[0]), ("dK", dk, ga[1]), ("dV", dv, ga[2])):
            assert torch.equal(hm(got, lo, hi).view(torch.int16), ref.view(torch.int16)), \
                f"{name} of sequence {b}"


def test_varlen_bwd_vs_oracle(cg, orc):
    H, Hkv, d = 4, 2, 128
    lens = [200, 64, 333]
    q, k, v, cu = _packed(lens, H, Hkv, d, seed=8900)
    do = cs.normal(tuple(q.shape), 8999)
    o, lse = cg.attention_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(lens), True)
    dq, dk, dv = cg.attention_bwd_varlen(do.cuda(), q.cuda(), k.cuda(), v.cuda(), o, lse, cu.cuda(),
                                         max(lens), True)
    assert cg.chain_check()[0] == 0
    G = H // Hkv
    for b in range(len(lens)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        hm = lambda x: x[lo:hi].transpose(0, 1).contiguous()
        rq, rk, rv, _ = orc.softmax_bwd(hm(q), hm(k).repeat_interleave(G, 0), hm(v).repeat_interleave(G, 0),
                                        hm(do), d ** -0.5, True)
        n = hi - lo
        rk = np.asarray(rk).reshape(Hkv, G, n, d).sum(1)
        rv = np.asarray(rv).reshape(Hkv, G, n, d).sum(1)
        assert_grad_close(hm(dq.cpu()), rq, f"varlen dQ seq {b}")
        assert_grad_close(hm(dk.cpu()), rk, f"varlen dK seq {b}")
        assert_grad_close(hm(dv.cpu()), rv, f"varlen dV seq {b}")


# ---------------------------------------------------------------- f16 P V
def _flush_tiny(v):
    # no nonzero |v| below 2^-31 of its head's largest: the per-head
    # power-of-two scale of the f16 copy then changes no rounding, so the
    # packed batch and each sequence alone give the same bits
    return torch.where(v.float().abs() < 1e-6, torch.zeros_like(v), v)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 128), (4, 2, 64), (6, 3, 128)])
def test_varlen_f16pv_matches_each_sequence_alone(cg, H, Hkv, d, causal):
    q, k, v, cu = _packed(LENS, H, Hkv, d, seed=9400 + H + d)
    v = _flush_tiny(v)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cg.attention_fwd_varlen_f16pv(qd, kd, vd, cu.cuda(), max(LENS), causal)
    assert cg.chain_check()[0] == 0
    hm = lambda x, lo, hi: x[lo:hi].transpose(0, 1).contiguous()
    for b, L in enumerate(LENS):
        lo, hi = int(cu[b]), int(cu[b + 1])
        oa, la = cg.attention_fwd_f16pv(hm(qd, lo, hi), hm(kd, lo, hi), hm(vd, lo, hi), causal)
        assert torch.equal(hm(o, lo, hi).view(torch.int16), oa.view(torch.int16)), f"O of sequence {b}"
        assert torch.equal(lse[:, lo:hi].contiguous().view(torch.int32), la.view(torch.int32)), \
            f"LSE of sequence {b}"


def test_varlen_f16pv_vs_oracle(cg, orc):
    H, Hkv, d = 4, 2, 128
    q, k, v, cu = _packed(LENS, H, Hkv, d, seed=9500)
    o, lse = cg.attention_fwd_varlen_f16pv(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(LENS), True)
    assert cg.chain_check()[0] == 0
    G = H // Hkv
    for b in range(len(LENS)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        qs = q[lo:hi].transpose(0, 1).contiguous()
        ks = k[lo:hi].transpose(0, 1).repeat_interleave(G, 0).contiguous()
        vs = v[lo:hi].transpose(0, 1).repeat_interleave(G, 0).contiguous()
        ro, rl = orc.softmax_fwd(qs, ks, vs, d ** -0.5, True)
        assert_fwd_close(o.cpu()[lo:hi].transpose(0, 1), ro, f"varlen f16pv O seq {b}")
        assert_lse_close(lse.cpu()[:, lo:hi], rl, f"varlen f16pv LSE seq {b}")


def test_varlen_f16pv_heads_of_very_different_scale(cg, orc):
    # one K/V head scaled by 2^40, another by 2^-40: each head's copy takes
    # its own power of two, so both stay within the forward bound
    H, Hkv, d = 4, 2, 64
    lens = [130, 257, 64]
    q, k, v, cu = _packed(lens, H, Hkv, d, seed=9550)
    v = v.float()
    v[:, 0] *= 2.0 ** 40
    v[:, 1] *= 2.0 ** -40
    v = v.to(torch.bfloat16)
    o, lse = cg.attention_fwd_varlen_f16pv(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max(lens), False)
    assert cg.chain_check()[0] == 0
    G = H // Hkv
    for b in range(len(lens)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            qs = q[lo:hi, h:h + 1].transpose(0, 1).contiguous()
            ks = k[lo:hi, h // G:h // G + 1].transpose(0, 1).contiguous()
            vs = v[lo:hi, h // G:h // G + 1].transpose(0, 1).contiguous()
            ro, _ = orc.softmax_fwd(qs, ks, vs, d ** -0.5, False)
            assert_fwd_close(o.cpu()[lo:hi, h:h + 1].transpose(0, 1), ro, f"seq {b} head {h}")


def test_varlen_f16pv_then_bwd(cg, orc):
    # O and LSE of the f16 P V forward feed chain_bwd_varlen
    H, Hkv, d = 4, 2, 128
    lens = [200, 64, 333]
    q, k, v, cu = _packed(lens, H, Hkv, d, seed=9600)
    do = cs.normal(tuple(q.shape), 9699)
    qd, kd, vd, cud = q.cuda(), k.cuda(), v.cuda(), cu.cuda()
    o, lse = cg.attention_fwd_varlen_f16pv(qd, kd, vd, cud, max(lens), True)
    dq, dk, dv = cg.attention_bwd_varlen(do.cuda(), qd, kd, vd, o, lse, cud, max(lens), True)
    assert cg.chain_check()[0] == 0
    G = H // Hkv
    for b in range(len(lens)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        hm = lambda x: x[lo:hi].transpose(0, 1).contiguous()
        rq, rk, rv, _ = orc.softmax_bwd(hm(q), hm(k).repeat_interleave(G, 0), hm(v).repeat_interleave(G, 0),
                                        hm(do), d ** -0.5, True)
        n = hi - lo
        rk = np.asarray(rk).reshape(Hkv, G, n, d).sum(1)
        rv = np.asarray(rv).reshape(Hkv, G, n, d).sum(1)
        assert_grad_close(hm(dq.cpu()), rq, f"dQ seq {b}")
        assert_grad_close(hm(dk.cpu()), rk, f"dK seq {b}")
        assert_grad_close(hm(dv.cpu()), rv, f"dV seq {b}")


def test_varlen_f16pv_rejects_bad_args(cg):
    q = torch.zeros(64, 2, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    need = cg.chain_fwd_varlen_f16pv_workspace_size(q)
    assert need >= 2 * 64 * 2 * 128
    o = torch.empty_like(q)
    lse = torch.empty(2, 64, dtype=torch.float32, device="cuda")
    short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_varlen_f16pv(q, q, q, cu, 1, 64, cg.MASK_CAUSAL, 0.1, o, lse, short)
    assert ei.value.status == cg.ERR_ARG
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.chain_fwd_varlen_f16pv(q, q, q, cu, 1, 65, cg.MASK_CAUSAL, 0.1, o, lse, ws)
    k = torch.zeros(64, 3, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.chain_fwd_varlen_f16pv(q, k, k, cu, 1, 64, cg.MASK_CAUSAL, 0.1, o, lse, ws)
    assert cg.chain_fwd_varlen_f16pv_workspace_size(q[:, :, :96]) == 0  # d = 96


def test_varlen_grid_beyond_its_extent_is_unsupported(cg):
    # 2^20 sequences (all but one empty) with max_seqlen 2^20: one block per
    # head, sequence and query tile would need more than 2^31 - 1 blocks;
    # refused before any launch
    total, H, d = 1 << 20, 1, 64
    q = torch.zeros(total, H, d, dtype=torch.bfloat16, device="cuda")
    cu = torch.full((total + 1,), total, dtype=torch.int32, device="cuda")
    cu[0] = 0
    batch = total
    o = torch.empty_like(q)
    lse = torch.empty(H, total, dtype=torch.float32, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_varlen(q, q, q, cu, batch, total, cg.MASK_CAUSAL, 0.125, o, lse)
    assert ei.value.status == cg.ERR_UNSUPPORTED
    ws = torch.empty(cg.chain_fwd_varlen_f16pv_workspace_size(q), dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_fwd_varlen_f16pv(q, q, q, cu, batch, total, cg.MASK_CAUSAL, 0.125, o, lse, ws)
    assert ei.value.status == cg.ERR_UNSUPPORTED
    wsb = torch.empty(cg.chain_bwd_workspace_size(q, q), dtype=torch.uint8, device="cuda")
    g = torch.empty_like(q)
    with pytest.raises(cg.ChainError) as ei:
        cg.chain_bwd_varlen(q, q, q, q, q, lse, cu, batch, total, cg.MASK_CAUSAL, 0.125, g, g, g, wsb)
    assert ei.value.status == cg.ERR_UNSUPPORTED
    del ws, wsb
    torch.cuda.synchronize()
    assert cg.chain_check()[0] == 0


def test_varlen_bwd_sequence_longer_than_max_is_reported(cg):
    # the 300-row sequence exceeds max_seqlen = 256: reported, and the other
    # sequence's gradients are still those of it alone
    lens = [300, 40]
    q, k, v, cu = _packed(lens, 2, 2, 128, seed=8650)
    do = cs.normal(tuple(q.shape), 8651)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    o, lse = cg.attention_fwd_varlen(qd, kd, vd, cud, 300, True)
    assert cg.chain_check()[0] == 0
    dq, dk, dv = cg.attention_bwd_varlen(dod, qd, kd, vd, o, lse, cud, 256, True)
    rc, _ = cg.chain_check()
    assert rc == cg.ERR_ARG
    assert cg.chain_check()[0] == 0
    hm = lambda x: x[300:340].transpose(0, 1).contiguous()
    oa, la = cg.attention_fwd(hm(qd), hm(kd), hm(vd), True)
    ga = cg.attention_bwd(hm(dod), hm(qd), hm(kd), hm(vd), oa, la, True)
    for name, got, ref in (("dQ", dq, ga[0]), ("dK", dk, ga[1]), ("dV", dv, ga[2])):
        assert torch.equal(hm(got).view(torch.int16), ref.view(torch.int16)), name
