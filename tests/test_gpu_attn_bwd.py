"""GPU: attention backward with recompute against the fp64 oracle.

The forward saves only O and LSE (produced by this library's own forward);
the backward recomputes S and P per tile.  Gradients are compared with the
textbook chain rule of the oracle in relative Frobenius norm."""
import math

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


def run_bwd(cg, q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = cg.attention_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = cg.attention_bwd(dod, qd, kd, vd, o, lse, causal, scale)
    rc, site = cg.chain_check()
    assert rc == 0, (rc, hex(site))
    return dq.cpu(), dk.cpu(), dv.cpu()


CASES = [(2, 256, 128), (1, 300, 128), (2, 129, 64), (1, 1, 128), (3, 520, 64), (1, 1024, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,n,d", CASES)
def test_bwd_small_vs_oracle(cg, orc, BH, n, d, causal):
    q, k, v, do = cs.attn_inputs(BH, n, d, seed=9000 + n + d, with_do=True)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = run_bwd(cg, q, k, v, do, causal, scale)
    rq, rk, rv, _ = orc.softmax_bwd(q, k, v, do, scale, causal)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_bwd_causal_64k_full_size(cg, orc):
    wl = cs.WORKLOADS["causal_bwd_64k"]
    dm = wl.dims
    BH, n, d = dm["BH"], dm["n"], dm["d"]
    q, k, v, do = cs.attn_inputs(BH, n, d, seed=wl.seed, with_do=True)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = run_bwd(cg, q, k, v, do, True, scale)
    # exact rows: the last 256 queries (and the key columns they complete)
    # plus two interior query windows, for the first and last head.
    for h in (0, BH - 1):
        i0 = n - 256
        rq, rk, rv, _ = orc.softmax_bwd(q, k, v, do, scale, True, heads=(h, h + 1),
                                        row_range=(i0, n), col_range=(i0, n))
        assert_grad_close(dq[h, i0:], rq[0], f"dQ tail head {h}")
        assert_grad_close(dk[h, i0:], rk[0], f"dK tail head {h}")
        assert_grad_close(dv[h, i0:], rv[0], f"dV tail head {h}")
        for a in (0, n // 2 + 77):
            rq, _, _, _ = orc.softmax_bwd(q, k, v, do, scale, True, heads=(h, h + 1),
                                          row_range=(a, a + 64), col_range=(a, a + 1))
            assert_grad_close(dq[h, a:a + 64], rq[0], f"dQ rows {a} head {h}")
    # key block 0 of head 0 in full: every one of the n queries attends to
    # it, so the dK/dV kernel accumulates it over all n/128 query tiles.
    rq, rk, rv, _ = orc.softmax_bwd(q, k, v, do, scale, True, heads=(0, 1),
                                    row_range=(0, n), col_range=(0, 128))
    assert_grad_close(dk[0, :128], rk[0], "dK key block 0 head 0")
    assert_grad_close(dv[0, :128], rv[0], "dV key block 0 head 0")
    assert_grad_close(dq[0], rq[0], "dQ head 0, every row")
    # invariants over every tile of every head: the key-sum of dK vanishes,
    # the key-sum of dV equals the query-sum of dO.
    dk64 = dk.double()
    dv64 = dv.double()
    ksum = dk64.sum(1).norm(dim=-1) / dk64.norm(dim=(1, 2))
    assert float(ksum.max()) < 1e-2, float(ksum.max())
    vs, gs = dv64.sum(1), do.double().sum(1)
    rel = (vs - gs).norm(dim=-1) / gs.norm(dim=-1)
    assert float(rel.max()) < 2e-2, float(rel.max())


def test_bwd_rejects_small_workspace(cg):
    q = torch.zeros(1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 128, dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.attention_bwd(q, q, q, q, q, lse, True, workspace=ws)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,BHkv,n,d", [(8, 2, 256, 128), (6, 3, 300, 64), (4, 1, 129, 128)])
def test_bwd_grouped_query_vs_oracle(cg, orc, BH, BHkv, n, d, causal):
    # Grouped-query attention: the oracle sees K and V repeated over each
    # group; dK and dV of a K/V head are the sums over its group.
    q, _, _, do = cs.attn_inputs(BH, n, d, seed=7600 + BH + n, with_do=True)
    _, k, v = cs.attn_inputs(BHkv, n, d, seed=7700 + BHkv + n)
    G = BH // BHkv
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cg.attention_fwd(qd, kd, vd, causal)
    dq, dk, dv = cg.attention_bwd(dod, qd, kd, vd, o, lse, causal)
    assert cg.chain_check()[0] == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    rq, rk, rv, _ = orc.softmax_bwd(q, k.repeat_interleave(G, 0), v.repeat_interleave(G, 0), do,
                                    d ** -0.5, causal)
    rk = np.asarray(rk).reshape(BHkv, G, n, d).sum(1)
    rv = np.asarray(rv).reshape(BHkv, G, n, d).sum(1)
    assert_grad_close(dq, rq, "GQA dQ")
    assert_grad_close(dk, rk, "GQA dK")
    assert_grad_close(dv, rv, "GQA dV")


def test_bwd_causal_16k_one_head_complete(cg, orc):
    # One causal head at n = 16384, d = 128: every element of dQ, dK and dV
    # against the oracle (128 query tiles, 128 key blocks).
    q, k, v, do = cs.attn_inputs(1, 16384, 128, seed=9400, with_do=True)
    scale = 128 ** -0.5
    dq, dk, dv = run_bwd(cg, q, k, v, do, True, scale)
    rq, rk, rv, _ = orc.softmax_bwd(q, k, v, do, scale, True)
    assert_grad_close(dq, rq, "dQ n=16384")
    assert_grad_close(dk, rk, "dK n=16384")
    assert_grad_close(dv, rv, "dV n=16384")
    # and per key block, so an error confined to one block is not averaged away
    for j in range(0, 16384, 128):
        assert_grad_close(dk[0, j:j + 128], rk[0, j:j + 128], f"dK block {j // 128}")
        assert_grad_close(dv[0, j:j + 128], rv[0, j:j + 128], f"dV block {j // 128}")
        assert_grad_close(dq[0, j:j + 128], rq[0, j:j + 128], f"dQ tile {j // 128}")
