"""GPU: the grouped-query and packed-sequence workloads at full size, through
the calls bench.py times beside the step, against the oracle on sampled rows
and on exact tails (the last 256 queries of a sequence and the key columns
they complete)."""
import math

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


def test_gqa_32q8kv_full_size(cg, orc):
    wl = cs.WORKLOADS["gqa_32k"]
    dm = wl.dims
    BH, BHkv, n, d = dm["BH"], dm["BHkv"], dm["n"], dm["d"]
    G = BH // BHkv
    q, _, _, do = cs.attn_inputs(BH, n, d, seed=wl.seed, with_do=True)
    k = cs.normal((BHkv, n, d), wl.seed + cs.OFF_K)
    v = cs.normal((BHkv, n, d), wl.seed + cs.OFF_V)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cg.attention_fwd_f16pv(qd, kd, vd, True, scale)
    dq, dk, dv = cg.attention_bwd(dod, qd, kd, vd, o, lse, True, scale)
    assert cg.chain_check()[0] == 0
    o, lse, dq, dk, dv = o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()
    kr, vr = k.repeat_interleave(G, 0), v.repeat_interleave(G, 0)
    rows = cs.sample_rows(BH, n, 12, seed=71)
    ro, rl = orc.softmax_fwd(q, kr, vr, scale, True, rows=rows)
    r = rows.numpy()
    assert_fwd_close(o[r[:, 0], r[:, 1]], ro, "GQA sampled O")
    assert_lse_close(lse[r[:, 0], r[:, 1]], rl, "GQA sampled LSE")
    # exact tails: dQ of the last 256 queries of a head; dK, dV of the last
    # 256 keys of a K/V head, summed over its group's query heads
    i0 = n - 256
    for hkv in (0, BHkv - 1):
        sk = np.zeros((256, d))
        sv = np.zeros((256, d))
        for h in range(hkv * G, (hkv + 1) * G):
            rq, rk, rv, _ = orc.softmax_bwd(q, kr, vr, do, scale, True, heads=(h, h + 1),
                                            row_range=(i0, n), col_range=(i0, n))
            sk += rk[0]
            sv += rv[0]
            if h == hkv * G:
                assert_grad_close(dq[h, i0:], rq[0], f"GQA dQ tail head {h}")
        assert_grad_close(dk[hkv, i0:], sk, f"GQA dK tail K/V head {hkv}")
        assert_grad_close(dv[hkv, i0:], sv, f"GQA dV tail K/V head {hkv}")
    # key block 0 of K/V head 0 in full: the dK/dV kernel accumulates it over
    # every query tile of all G query heads of the group
    sk = np.zeros((128, d))
    sv = np.zeros((128, d))
    for h in range(G):
        _, rk, rv, _ = orc.softmax_bwd(q, kr, vr, do, scale, True, heads=(h, h + 1),
                                       row_range=(0, n), col_range=(0, 128))
        sk += rk[0]
        sv += rv[0]
    assert_grad_close(dk[0, :128], sk, "GQA dK key block 0, K/V head 0")
    assert_grad_close(dv[0, :128], sv, "GQA dV key block 0, K/V head 0")
    # over every K/V head: the key-sum of dK vanishes; the key-sum of dV
    # equals the query-sum of its group's dO
    dk64 = dk.double()
    ksum = dk64.sum(1).norm(dim=-1) / dk64.norm(dim=(1, 2))
    assert float(ksum.max()) < 1e-2, float(ksum.max())
    gs = do.double().reshape(BHkv, G, n, d).sum(dim=(1, 2))
    rel = (dv.double().sum(1) - gs).norm(dim=-1) / gs.norm(dim=-1)
    assert float(rel.max()) < 2e-2, float(rel.max())


def test_varlen_128k_full_size(cg, orc):
    wl = cs.WORKLOADS["varlen_128k"]
    dm = wl.dims
    total, H, d = dm["total"], dm["H"], dm["d"]
    lens = cs.varlen_lengths(total, dm["min_len"], dm["max_len"], wl.seed)
    q = cs.normal((total, H, d), wl.seed + cs.OFF_Q)
    k = cs.normal((total, H, d), wl.seed + cs.OFF_K)
    v = cs.normal((total, H, d), wl.seed + cs.OFF_V)
    do = cs.normal((total, H, d), wl.seed + cs.OFF_DO)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    o, lse = cg.attention_fwd_varlen_f16pv(qd, kd, vd, cud, max(lens), True, scale)
    dq, dk, dv = cg.attention_bwd_varlen(dod, qd, kd, vd, o, lse, cud, max(lens), True, scale)
    assert cg.chain_check()[0] == 0
    o, lse, dq, dk, dv = o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()
    hm = lambda x, lo, hi: x[lo:hi].transpose(0, 1).contiguous()
    # the shortest, a middle and the longest sequence
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    for b in (order[0], order[len(order) // 2], order[-1]):
        lo, hi = int(cu[b]), int(cu[b + 1])
        nb = hi - lo
        qs, ks, vs, gs = hm(q, lo, hi), hm(k, lo, hi), hm(v, lo, hi), hm(do, lo, hi)
        rows = cs.sample_rows(H, nb, 8, seed=90 + b)
        ro, rl = orc.softmax_fwd(qs, ks, vs, scale, True, rows=rows)
        r = rows.numpy()
        assert_fwd_close(hm(o, lo, hi)[r[:, 0], r[:, 1]], ro, f"sequence {b} sampled O")
        assert_lse_close(lse[:, lo:hi][r[:, 0], r[:, 1]], rl, f"sequence {b} sampled LSE")
        i0 = nb - 256
        for h in (0, H - 1):
            rq, rk, rv, _ = orc.softmax_bwd(qs, ks, vs, gs, scale, True, heads=(h, h + 1),
                                            row_range=(i0, nb), col_range=(i0, nb))
            assert_grad_close(dq[lo + i0:hi, h], rq[0], f"sequence {b} dQ tail head {h}")
            assert_grad_close(dk[lo + i0:hi, h], rk[0], f"sequence {b} dK tail head {h}")
            assert_grad_close(dv[lo + i0:hi, h], rv[0], f"sequence {b} dV tail head {h}")
