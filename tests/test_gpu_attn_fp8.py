"""GPU: softmax attention on e4m3 Q, K, V (chain_fwd_fp8) against the fp64
oracle fed the same e4m3 codes (their exact values)."""
import math

import numpy as np
import pytest
import torch

import chain_synth as cs
from tol import assert_fwd_close, assert_lse_close

pytestmark = pytest.mark.gpu
E4M3 = torch.float8_e4m3fn


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


def _fp8_inputs(BH, n, seed, BHkv=None):
    q, _, _ = cs.attn_inputs(BH, n, 128, seed=seed, dtype=E4M3)
    _, k, v = cs.attn_inputs(BHkv or BH, n, 128, seed=seed + 10, dtype=E4M3)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,n", [(2, 256), (3, 300), (1, 1), (1, 127), (4, 1000), (2, 129)])
def test_fp8_small_vs_oracle(cg, orc, BH, n, causal):
    q, k, v = _fp8_inputs(BH, n, seed=9000 + n)
    scale = 1.0 / math.sqrt(128)
    o, lse = cg.attention_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert cg.chain_check()[0] == 0
    assert o.dtype == torch.bfloat16
    ro, rl = orc.softmax_fwd(q, k, v, scale, causal)
    assert_fwd_close(o, ro, f"fp8 O {BH}x{n} causal={causal}")
    assert_lse_close(lse, rl, "fp8 LSE")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_grouped_query_vs_oracle(cg, orc, causal):
    BH, BHkv, n = 8, 2, 384
    q, k, v = _fp8_inputs(BH, n, seed=9100, BHkv=BHkv)
    o, lse = cg.attention_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), causal)
    assert cg.chain_check()[0] == 0
    G = BH // BHkv
    ro, rl = orc.softmax_fwd(q, k.repeat_interleave(G, 0), v.repeat_interleave(G, 0), 128 ** -0.5,
                             causal)
    assert_fwd_close(o, ro, "fp8 GQA O")
    assert_lse_close(lse, rl, "fp8 GQA LSE")


def test_fp8_every_value_of_v_passes_exactly(cg, orc):
    # Hard attention: K_j = 16 e_j, Q_i = 16 e_pi(i), scale 1, so S_ij = 256
    # for j = pi(i) and 0 otherwise; exp(-256) vanishes in fp32 and f16, so
    # O_i = V_pi(i) exactly.  V holds every finite e4m3 code (subnormals,
    # 448, negative zero), so each passes the f16 re-encoding unchanged.
    n = 128
    perm = torch.from_numpy(np.random.default_rng(5).permutation(n))
    eye = torch.eye(n, dtype=torch.float32) * 16.0
    k = eye.to(E4M3).reshape(1, n, 128)
    q = eye[perm].to(E4M3).reshape(1, n, 128)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    codes = np.resize(finite, n * 128).reshape(1, n, 128)
    codes = codes[:, np.random.default_rng(6).permutation(n)]
    v = torch.from_numpy(codes.copy()).view(E4M3)
    o, lse = cg.attention_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), False, 1.0)
    assert cg.chain_check()[0] == 0
    want = orc.e4m3_decode(v)[0][perm.numpy()]
    np.testing.assert_array_equal(o.float().cpu().numpy()[0], want)
    assert np.abs(lse.cpu().numpy() - 256.0).max() < 1e-3


def test_fp8_v_scale(cg, orc):
    q, k, v = _fp8_inputs(2, 300, seed=9200)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = cg.attention_fwd_fp8(qd, kd, vd, True)
    o2, l2 = cg.attention_fwd_fp8(qd, kd, vd, True, v_scale=2.0)
    # a power of two scales exactly, before the one rounding of O
    assert torch.equal(o2.float(), 2.0 * o1.float())
    assert torch.equal(l1, l2)
    # any factor: against the oracle on the scaled values (and Q, K scales
    # folded into the score scale)
    vs, qs, ks = 0.37, 0.5, 1.25
    o3, l3 = cg.attention_fwd_fp8(qd, kd, vd, True, scale=qs * ks * 128 ** -0.5, v_scale=vs)
    assert cg.chain_check()[0] == 0
    dq, dk, dv = (torch.from_numpy(orc.e4m3_decode(x)) for x in (q, k, v))
    ro, rl = orc.softmax_fwd(dq * qs, dk * ks, dv * vs, 128 ** -0.5, True)
    assert_fwd_close(o3, ro, "fp8 scaled O")
    assert_lse_close(l3, rl, "fp8 scaled LSE")


def test_fp8_strided_4d_and_caller_workspace(cg, orc):
    # [B][H][n][d] views with a padded row pitch (rows 256 bytes apart), a
    # caller-owned workspace
    B, H, n = 2, 2, 200
    base = cs.normal((3, B, H, n, 256), seed=9300).to(E4M3).cuda()
    q, k, v = (base[i, ..., :128] for i in range(3))
    assert q.stride(-2) == 256
    o = torch.empty(B, H, n, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, n, dtype=torch.float32, device="cuda")
    ws = torch.empty(cg.chain_fwd_fp8_workspace_size(v), dtype=torch.uint8, device="cuda")
    assert ws.numel() == 2 * B * H * n * 128
    cg.chain_fwd_fp8(q, k, v, cg.MASK_CAUSAL, 128 ** -0.5, 1.0, o, lse, ws)
    assert cg.chain_check()[0] == 0
    fl = lambda x: x.reshape(B * H, n, 128).cpu()
    ro, rl = orc.softmax_fwd(fl(q), fl(k), fl(v), 128 ** -0.5, True)
    assert_fwd_close(o.reshape(B * H, n, 128), ro, "fp8 4-D")
    assert_lse_close(lse.reshape(B * H, n), rl, "fp8 4-D LSE")


def test_fp8_rejects_bad_args(cg):
    z = lambda *s, dt=E4M3: torch.zeros(*s, device="cuda").to(dt)
    q = z(1, 128, 64)  # d = 64
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_fp8(q, q, q, True)
    assert e.value.status == cg.ERR_UNSUPPORTED
    qb = z(1, 128, 128, dt=torch.bfloat16)
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_fp8(qb, qb, qb, True)
    assert e.value.status == cg.ERR_DTYPE
    q = z(1, 128, 128)
    with pytest.raises(cg.ChainError) as e:  # workspace too small
        cg.attention_fwd_fp8(q, q, q, True, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == cg.ERR_ARG
    with pytest.raises(cg.ChainError) as e:  # e4m3 through the bf16 entry point
        cg.attention_fwd(q, q, q, True)
    assert e.value.status == cg.ERR_DTYPE
    with pytest.raises(cg.ChainError) as e:  # K heads not dividing Q heads
        cg.attention_fwd_fp8(z(3, 128, 128), q.expand(2, 128, 128).contiguous(),
                             q.expand(2, 128, 128).contiguous(), True)
    assert e.value.status == cg.ERR_ARG


def test_fp8_relayout_moves_bytes(cg, orc):
    # the Ulysses relayout is a bit copy: e4m3 shards move like any 1-byte type
    p, n_loc, H, g = 4, 64, 8, 1
    x = cs.normal((p, n_loc, H, 128), seed=9400).to(E4M3)
    out = cg.relayout(x.cuda(), p, g)
    raw, shape = orc.relayout(x.view(torch.uint8), p, g)
    assert np.array_equal(out.view(torch.uint8).cpu().numpy().reshape(-1), raw.reshape(-1))


def test_fp8_full_size_sampled(cg, orc):
    # the causal 32 x 32768 x 128 workload with e4m3 inputs: sampled rows
    wl = cs.WORKLOADS["causal_attn_32k_e4m3"]
    dm = wl.dims
    q, k, v = cs.attn_inputs(dm["BH"], dm["n"], dm["d"], seed=wl.seed, dtype=E4M3)
    scale = dm["d"] ** -0.5
    o, lse = cg.attention_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), True, scale)
    assert cg.chain_check()[0] == 0
    rows = cs.sample_rows(dm["BH"], dm["n"], 16, seed=4)
    ro, rl = orc.softmax_fwd(q, k, v, scale, True, rows=rows)
    r = rows.numpy()
    assert_fwd_close(o.cpu()[r[:, 0], r[:, 1]], ro, "fp8 sampled O")
    assert_lse_close(lse.cpu()[r[:, 0], r[:, 1]], rl, "fp8 sampled LSE")
