"""GPU: softmax attention forward with P V as one f16 product
(chain_fwd_f16pv) against the fp64 oracle, including V of wide dynamic
range (the per-head power-of-two scale of its f16 copy)."""
import math

import numpy as np
import pytest
import torch

import chain_synth as cs
from tol import assert_fwd_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


CASES = [(2, 256, 128), (3, 300, 128), (1, 1, 128), (2, 129, 64), (1, 640, 64), (4, 1000, 128),
         (1, 127, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,n,d", CASES)
def test_f16pv_small_vs_oracle(cg, orc, BH, n, d, causal):
    q, k, v = cs.attn_inputs(BH, n, d, seed=9500 + n + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = cg.attention_fwd_f16pv(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert cg.chain_check()[0] == 0
    ro, rl = orc.softmax_fwd(q, k, v, scale, causal)
    assert_fwd_close(o, ro, f"f16pv O {BH}x{n}x{d} causal={causal}")
    assert_lse_close(lse, rl, "f16pv LSE")


@pytest.mark.parametrize("causal", [False, True])
def test_f16pv_grouped_query_vs_oracle(cg, orc, causal):
    BH, BHkv, n, d = 8, 2, 300, 128
    q, _, _ = cs.attn_inputs(BH, n, d, seed=9600)
    _, k, v = cs.attn_inputs(BHkv, n, d, seed=9610)
    o, lse = cg.attention_fwd_f16pv(q.cuda(), k.cuda(), v.cuda(), causal)
    assert cg.chain_check()[0] == 0
    G = BH // BHkv
    ro, rl = orc.softmax_fwd(q, k.repeat_interleave(G, 0), v.repeat_interleave(G, 0), d ** -0.5,
                             causal)
    assert_fwd_close(o, ro, "f16pv GQA O")
    assert_lse_close(lse, rl, "f16pv GQA LSE")


def test_f16pv_wide_range_values(cg, orc):
    # Heads of V at 2^40, 2^-60, 1e30 (beyond f16's range) and all zeros, and
    # a head whose values span 2^-20 .. 2^10: each head's f16 copy carries its
    # own scale, so all match the oracle.
    BH, n, d = 5, 384, 128
    q, k, v = cs.attn_inputs(BH, n, d, seed=9700)
    vf = v.float()
    vf[0] *= 2.0 ** 40
    vf[1] *= 2.0 ** -60
    vf[2] *= 1e30
    vf[3] = 0.0
    vf[4] *= torch.exp2(torch.linspace(-20, 10, n)).reshape(n, 1)
    v = vf.to(torch.bfloat16)
    o, lse = cg.attention_fwd_f16pv(q.cuda(), k.cuda(), v.cuda(), True)
    assert cg.chain_check()[0] == 0
    ro, rl = orc.softmax_fwd(q, k, v, d ** -0.5, True)
    for h in (0, 1, 2, 4):
        assert_fwd_close(o[h], ro[h], f"head {h}")
    assert torch.count_nonzero(o[3]) == 0
    assert_lse_close(lse, rl, "wide-range LSE")


def test_f16pv_matches_compensated_path(cg):
    # The same S, the same softmax: LSE agrees with chain_fwd's to fp32
    # rounding of the row sums, O within the rounding of the two forms.
    q, k, v = (t.cuda() for t in cs.attn_inputs(4, 1024, 128, seed=9800))
    o1, l1 = cg.attention_fwd(q, k, v, True)
    o2, l2 = cg.attention_fwd_f16pv(q, k, v, True)
    assert (l1 - l2).abs().max().item() < 1e-5
    d = (o1.float() - o2.float()).abs()
    assert d.sum().item() / o1.float().abs().sum().item() < 2e-3


def test_f16pv_strided_4d_and_caller_workspace(cg, orc):
    B, H, n, d = 2, 2, 200, 64
    base = cs.normal((3, B, H, n, 128), seed=9900).cuda()
    q, k, v = (base[i, ..., :d] for i in range(3))
    o = torch.empty(B, H, n, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    ws = torch.empty(cg.chain_fwd_f16pv_workspace_size(q, v), dtype=torch.uint8, device="cuda")
    cg.chain_fwd_f16pv(q, k, v, cg.MASK_CAUSAL, d ** -0.5, o, lse, ws)
    assert cg.chain_check()[0] == 0
    fl = lambda x: x.reshape(B * H, n, d).cpu()
    ro, rl = orc.softmax_fwd(fl(q), fl(k), fl(v), d ** -0.5, True)
    assert_fwd_close(o.reshape(B * H, n, d), ro, "f16pv 4-D")
    assert_lse_close(lse.reshape(B * H, n), rl, "f16pv 4-D LSE")


def test_f16pv_rejects_bad_args(cg):
    q = torch.zeros(1, 128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as e:  # workspace too small
        cg.attention_fwd_f16pv(q, q, q, True, workspace=torch.empty(64, dtype=torch.uint8,
                                                                       device="cuda"))
    assert e.value.status == cg.ERR_ARG
    qf = torch.zeros(1, 128, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_f16pv(qf, qf, qf, True)
    assert e.value.status == cg.ERR_DTYPE
    q96 = torch.zeros(1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_f16pv(q96, q96, q96, True)
    assert e.value.status == cg.ERR_ARG


def test_f16pv_full_size_sampled(cg, orc):
    wl = cs.WORKLOADS["causal_attn_32k"]
    dm = wl.dims
    q, k, v = cs.attn_inputs(dm["BH"], dm["n"], dm["d"], seed=wl.seed)
    scale = dm["d"] ** -0.5
    o, lse = cg.attention_fwd_f16pv(q.cuda(), k.cuda(), v.cuda(), True, scale)
    assert cg.chain_check()[0] == 0
    rows = cs.sample_rows(dm["BH"], dm["n"], 16, seed=5)
    ro, rl = orc.softmax_fwd(q, k, v, scale, True, rows=rows)
    r = rows.numpy()
    assert_fwd_close(o.cpu()[r[:, 0], r[:, 1]], ro, "f16pv sampled O")
    assert_lse_close(lse.cpu()[r[:, 0], r[:, 1]], rl, "f16pv sampled LSE")
