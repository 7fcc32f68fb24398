"""GPU: softmax attention forward against the fp64 oracle."""
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


CASES = [  # BH, n, d
    (2, 256, 128), (3, 300, 128), (1, 1, 128), (2, 129, 64), (1, 640, 64), (4, 1000, 128),
    (1, 127, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,n,d", CASES)
def test_fwd_small_vs_oracle(cg, orc, BH, n, d, causal):
    q, k, v = cs.attn_inputs(BH, n, d, seed=7000 + n + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert cg.chain_check()[0] == 0
    ro, rl = orc.softmax_fwd(q, k, v, scale, causal)
    assert_fwd_close(o, ro, f"O {BH}x{n}x{d} causal={causal}")
    assert_lse_close(lse, rl, "LSE")


def test_fwd_4d_layout_and_strided_rows(cg, orc):
    # [B][H][n][d] with a padded row pitch (d=64 inside rows of 128).
    B, H, n, d = 2, 2, 200, 64
    base = cs.normal((3, B, H, n, 128), seed=99)
    q, k, v = (base[i, ..., :d] for i in range(3))
    based = base.cuda()
    qd, kd, vd = (based[i, ..., :d] for i in range(3))
    assert qd.stride(-2) == 128
    o = torch.empty(B, H, n, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    cg.chain_fwd(qd, kd, vd, cg.F_SOFTMAX, cg.MASK_CAUSAL, d ** -0.5, o, lse)
    assert cg.chain_check()[0] == 0
    ro, rl = orc.softmax_fwd(q.reshape(B * H, n, d).contiguous(), k.reshape(B * H, n, d).contiguous(),
                             v.reshape(B * H, n, d).contiguous(), d ** -0.5, True)
    assert_fwd_close(o.reshape(B * H, n, d), ro, "4-D strided")
    assert_lse_close(lse.reshape(B * H, n), rl, "4-D LSE")


def test_fwd_uniform_scores_closed_form(cg):
    # Q = 0: O_i = mean of V over the allowed keys, LSE_i = ln(#keys).
    BH, n, d = 1, 384, 128
    q = torch.zeros(BH, n, d, dtype=torch.bfloat16)
    _, k, v = cs.attn_inputs(BH, n, d, seed=71)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), True)
    cnt = torch.arange(1, n + 1, dtype=torch.float64)
    ref = v.double().cumsum(1) / cnt.reshape(1, n, 1)
    assert_fwd_close(o, ref, "uniform")
    assert np.abs(lse.cpu().double().numpy() - np.log(cnt.numpy())).max() < 1e-3


def test_fwd_large_scores_stable(cg, orc):
    # |scores| ~ 1e3: no inf/NaN, still matches.
    q, k, v = cs.attn_inputs(2, 256, 64, seed=72)
    q = (q.float() * 30).to(torch.bfloat16)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), True, 1.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    ro, rl = orc.softmax_fwd(q, k, v, 1.0, True)
    assert_fwd_close(o, ro, "large scores")
    assert_lse_close(lse, rl, "large scores LSE")


def test_fwd_rejects_bad_args(cg):
    q = torch.zeros(1, 64, 96, dtype=torch.bfloat16, device="cuda")  # d=96 unsupported
    with pytest.raises(cg.ChainError):
        cg.attention_fwd(q, q, q, True)
    q = torch.zeros(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError):
        cg.chain_fwd(q, q, q, cg.F_SOFTMAX, 0, 0.1, torch.empty_like(q), None)  # LSE missing


def _sampled_check(cg, orc, q, k, v, causal, seed, per_head):
    BH, n, d = q.shape
    scale = 1.0 / math.sqrt(d)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert cg.chain_check()[0] == 0
    rows = cs.sample_rows(BH, n, per_head, seed=seed)
    ro, rl = orc.softmax_fwd(q, k, v, scale, causal, rows=rows)
    r = rows.numpy()
    oc = o.cpu()[r[:, 0], r[:, 1]]
    lc = lse.cpu()[r[:, 0], r[:, 1]]
    assert_fwd_close(oc, ro, "sampled O")
    assert_lse_close(lc, rl, "sampled LSE")
    return o, lse


def test_fwd_causal_32k_full_size_sampled(cg, orc):
    wl = cs.WORKLOADS["causal_attn_32k"]
    dm = wl.dims
    q, k, v = cs.attn_inputs(dm["BH"], dm["n"], dm["d"], seed=wl.seed)
    _sampled_check(cg, orc, q, k, v, True, seed=3, per_head=24)


# ------------------------------------------------------- fp32 (3xTF32) path
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,n", [(1, 256), (2, 300), (1, 1), (3, 129)])
def test_fwd_fp32_vs_oracle(cg, orc, BH, n, causal):
    q, k, v = cs.attn_inputs(BH, n, 64, seed=1000 + n, dtype=torch.float32)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal, 0.125)
    assert cg.chain_check()[0] == 0
    assert o.dtype == torch.float32
    ro, rl = orc.softmax_fwd(q, k, v, 0.125, causal)
    mx, mean = assert_fwd_close(o, ro, f"fp32 {BH}x{n} causal={causal}")
    assert mean < 1e-5, mean  # full fp32 accuracy from the split tf32 products
    assert_lse_close(lse, rl, "fp32 LSE")


def test_fwd_fp32_tiny_workload(cg, orc):
    # 1 head, n = 256, d = 64, fp32 N(0,1), scale 1/8, non-causal
    wl = cs.WORKLOADS["tiny_attn_fp32"]
    dm = wl.dims
    q, k, v = cs.attn_inputs(dm["BH"], dm["n"], dm["d"], seed=wl.seed, dtype=torch.float32)
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), False, 1.0 / math.sqrt(dm["d"]))
    ro, rl = orc.softmax_fwd(q, k, v, 1.0 / math.sqrt(dm["d"]), False)
    assert_fwd_close(o, ro, "tiny fp32 workload")
    assert_lse_close(lse, rl, "tiny fp32 LSE")


def test_fwd_fp32_rejects_d128(cg):
    q = torch.zeros(1, 64, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(cg.ChainError) as ei:
        cg.attention_fwd(q, q, q, False)
    assert ei.value.status == cg.ERR_UNSUPPORTED


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,BHkv,n,d", [(8, 2, 300, 128), (6, 3, 256, 64), (4, 1, 129, 128)])
def test_fwd_grouped_query_vs_oracle(cg, orc, BH, BHkv, n, d, causal):
    # Grouped-query attention: query head h reads K/V head h // (BH // BHkv).
    # The oracle sees K and V repeated over each group.
    q, _, _ = cs.attn_inputs(BH, n, d, seed=7400 + BH + n)
    _, k, v = cs.attn_inputs(BHkv, n, d, seed=7500 + BHkv + n)
    G = BH // BHkv
    o, lse = cg.attention_fwd(q.cuda(), k.cuda(), v.cuda(), causal)
    assert cg.chain_check()[0] == 0
    ro, rl = orc.softmax_fwd(q, k.repeat_interleave(G, 0), v.repeat_interleave(G, 0), d ** -0.5,
                             causal)
    assert_fwd_close(o, ro, f"GQA O {BH}/{BHkv}x{n}x{d}")
    assert_lse_close(lse, rl, "GQA LSE")


def test_fwd_grouped_query_bad_ratio(cg):
    q = torch.zeros(6, 128, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(4, 128, 128, dtype=torch.bfloat16, device="cuda")  # 6 % 4 != 0
    with pytest.raises(cg.ChainError):
        cg.attention_fwd(q, k, k, True)
