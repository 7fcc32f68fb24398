"""GPU: attention read from and written back to Ulysses sequence shards
(chain_fwd_sp), against the unfused GPU path (bit for bit) and the oracle."""
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


def _unfused(cg, q, k, v, p, g, causal, scale, o_init):
    """sp_relayout of Q, K, V, head-major attention, inverse relayout of O."""
    qh, kh, vh = (cg.relayout(x, p, g) for x in (q, k, v))
    oh, lse = cg.attention_fwd(qh, kh, vh, causal, scale)
    o = o_init.clone()
    cg.sp_relayout_inverse(oh, p, g, o)
    return o, lse


def _bits(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


@pytest.mark.parametrize("p,n_loc,H,d,g,causal", [
    (4, 256, 8, 128, 0, True), (4, 256, 8, 128, 3, False), (2, 384, 4, 64, 1, True),
    (1, 512, 2, 128, 0, True), (4, 128, 4, 128, 2, True)])
def test_sp_matches_unfused_bit_exact(cg, p, n_loc, H, d, g, causal):
    q, k, v = (cs.normal((p, n_loc, H, d), seed=8100 + i).cuda() for i in range(3))
    scale = 1.0 / math.sqrt(d)
    o_init = cs.iota16((p, n_loc, H, d)).view(torch.bfloat16).cuda()
    o = o_init.clone()
    o, lse = cg.attention_fwd_sp(q, k, v, p, g, causal, scale, o=o)
    assert cg.chain_check()[0] == 0
    ro, rl = _unfused(cg, q, k, v, p, g, causal, scale, o_init)
    assert np.array_equal(_bits(o), _bits(ro)), "O differs from the unfused path"
    assert np.array_equal(_bits(lse), _bits(rl)), "LSE differs from the unfused path"


def test_sp_vs_oracle(cg, orc):
    p, n_loc, H, d, g = 4, 128, 8, 128, 2
    q, k, v = (cs.normal((p, n_loc, H, d), seed=8200 + i) for i in range(3))
    scale = d ** -0.5
    o, lse = cg.attention_fwd_sp(q.cuda(), k.cuda(), v.cuda(), p, g, True, scale)
    assert cg.chain_check()[0] == 0
    heads = []
    for x in (q, k, v):
        raw, shape = orc.relayout(x, p, g)
        heads.append(torch.from_numpy(raw).view(torch.bfloat16).reshape(shape))
    ro, rl = orc.softmax_fwd(heads[0], heads[1], heads[2], scale, True)
    raw, shape = orc.relayout(o.cpu(), p, g)
    oh = torch.from_numpy(raw).view(torch.bfloat16).reshape(shape)
    assert_fwd_close(oh, ro, "sharded O vs oracle")
    assert_lse_close(lse, rl, "sharded LSE vs oracle")


def test_sp_leaves_other_heads_untouched(cg):
    p, n_loc, H, d, g = 4, 128, 8, 64, 1
    q, k, v = (cs.normal((p, n_loc, H, d), seed=8300 + i).cuda() for i in range(3))
    o_init = cs.iota16((p, n_loc, H, d)).view(torch.bfloat16).cuda()
    o, _ = cg.attention_fwd_sp(q, k, v, p, g, True, o=o_init.clone())
    Hl = H // p
    mine = torch.zeros(H, dtype=torch.bool)
    mine[g * Hl:(g + 1) * Hl] = True
    assert torch.equal(o[:, :, ~mine].view(torch.int16), o_init[:, :, ~mine].view(torch.int16))
    assert not torch.equal(o[:, :, mine].view(torch.int16), o_init[:, :, mine].view(torch.int16))


def test_sp_rejects_bad_args(cg):
    q = torch.zeros(4, 100, 8, 128, dtype=torch.bfloat16, device="cuda")  # n_loc % 128
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_sp(q, q, q, 4, 0, True)
    assert e.value.status == cg.ERR_UNSUPPORTED
    q = torch.zeros(4, 128, 8, 128, dtype=torch.bfloat16, device="cuda")
    for p, g in ((4, 4), (4, -1), (3, 0)):  # group out of range, H % p != 0
        with pytest.raises(cg.ChainError) as e:
            cg.attention_fwd_sp(q, q, q, p, g, True)
        assert e.value.status == cg.ERR_ARG
    qf = torch.zeros(4, 128, 8, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_sp(qf, qf, qf, 4, 0, True)
    assert e.value.status == cg.ERR_DTYPE


def test_sp_full_size_matches_unfused(cg):
    # The Ulysses workload: shards 4 x [32768][32][128], head group 0 (8 heads
    # over 131072 positions), causal.
    dm = cs.WORKLOADS["ulysses_128k"].dims
    p, n_loc, H, d = dm["p"], dm["n_loc"], dm["H"], dm["d"]
    gen = torch.Generator(device="cuda").manual_seed(84)
    q, k, v = (torch.randn(p, n_loc, H, d, device="cuda", generator=gen).to(torch.bfloat16)
               for _ in range(3))
    o_init = torch.zeros_like(q)
    o, lse = cg.attention_fwd_sp(q, k, v, p, 0, True, o=o_init.clone())
    assert cg.chain_check()[0] == 0
    ro, rl = _unfused(cg, q, k, v, p, 0, True, d ** -0.5, o_init)
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))


# ------------------------------------------- f16 P V form (chain_fwd_sp_f16pv)
def _unfused_f16pv(cg, q, k, v, p, g, causal, scale, o_init):
    """sp_relayout of Q, K, V, chain_fwd_f16pv, inverse relayout of O."""
    qh, kh, vh = (cg.relayout(x, p, g) for x in (q, k, v))
    oh, lse = cg.attention_fwd_f16pv(qh, kh, vh, causal, scale)
    o = o_init.clone()
    cg.sp_relayout_inverse(oh, p, g, o)
    return o, lse


@pytest.mark.parametrize("p,n_loc,H,d,g,causal", [
    (4, 256, 8, 128, 0, True), (4, 256, 8, 128, 3, False), (2, 384, 4, 64, 1, True),
    (1, 512, 2, 128, 0, True), (4, 128, 4, 128, 2, True)])
def test_sp_f16pv_matches_unfused_bit_exact(cg, p, n_loc, H, d, g, causal):
    q, k, v = (cs.normal((p, n_loc, H, d), seed=8500 + i).cuda() for i in range(3))
    scale = 1.0 / math.sqrt(d)
    o_init = cs.iota16((p, n_loc, H, d)).view(torch.bfloat16).cuda()
    o, lse = cg.attention_fwd_sp_f16pv(q, k, v, p, g, causal, scale, o=o_init.clone())
    assert cg.chain_check()[0] == 0
    ro, rl = _unfused_f16pv(cg, q, k, v, p, g, causal, scale, o_init)
    assert np.array_equal(_bits(o), _bits(ro)), "O differs from the unfused path"
    assert np.array_equal(_bits(lse), _bits(rl)), "LSE differs from the unfused path"


def test_sp_f16pv_vs_oracle(cg, orc):
    p, n_loc, H, d, g = 4, 128, 8, 128, 1
    q, k, v = (cs.normal((p, n_loc, H, d), seed=8600 + i) for i in range(3))
    scale = d ** -0.5
    o, lse = cg.attention_fwd_sp_f16pv(q.cuda(), k.cuda(), v.cuda(), p, g, True, scale)
    assert cg.chain_check()[0] == 0
    heads = []
    for x in (q, k, v):
        raw, shape = orc.relayout(x, p, g)
        heads.append(torch.from_numpy(raw).view(torch.bfloat16).reshape(shape))
    ro, rl = orc.softmax_fwd(heads[0], heads[1], heads[2], scale, True)
    raw, shape = orc.relayout(o.cpu(), p, g)
    oh = torch.from_numpy(raw).view(torch.bfloat16).reshape(shape)
    assert_fwd_close(oh, ro, "sharded f16 P V O vs oracle")
    assert_lse_close(lse, rl, "sharded f16 P V LSE vs oracle")


def test_sp_f16pv_rejects_short_workspace(cg):
    q = torch.zeros(4, 128, 8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.ChainError) as e:
        cg.attention_fwd_sp_f16pv(q, q, q, 4, 0, True,
                                  workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == cg.ERR_ARG


def test_sp_f16pv_full_size_matches_unfused(cg):
    dm = cs.WORKLOADS["ulysses_128k"].dims
    p, n_loc, H, d = dm["p"], dm["n_loc"], dm["H"], dm["d"]
    gen = torch.Generator(device="cuda").manual_seed(85)
    q, k, v = (torch.randn(p, n_loc, H, d, device="cuda", generator=gen).to(torch.bfloat16)
               for _ in range(3))
    o_init = torch.zeros_like(q)
    o, lse = cg.attention_fwd_sp_f16pv(q, k, v, p, 0, True, o=o_init.clone())
    assert cg.chain_check()[0] == 0
    ro, rl = _unfused_f16pv(cg, q, k, v, p, 0, True, d ** -0.5, o_init)
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))


# --------------------- the Ulysses workload at full size against the oracle
def _ulysses_rows(Hl, n, seed):
    """(head, row) pairs: per head rows 0, 1, 127, 128, n-2, n-1, three rows
    of the last 256-query block (whose causal rows span every key tile) and
    seeded rows elsewhere, at least 16 per head."""
    g = np.random.default_rng(seed)
    out = []
    for h in range(Hl):
        fixed = {0, 1, 127, 128, n - 2, n - 1}
        fixed |= set(int(r) for r in g.integers(n - 256, n, 3))
        fixed |= set(int(r) for r in g.integers(0, n, 12))
        out.extend((h, r) for r in sorted(fixed))
    return np.asarray(out, dtype=np.int64)


def test_ulysses_128k_full_size_vs_oracle(cg, orc):
    # The Ulysses workload as the benchmark runs it: shards 4 x [32768][32][128]
    # bf16 ~ N(0,1) (seeds of the workload), head group 0 relayouted to
    # [8][131072][128], causal attention on those heads through
    # chain_fwd_f16pv; then the same heads straight from the shards through
    # chain_fwd_sp_f16pv and chain_fwd_sp.  The oracle attends the heads its
    # own relayout produced, on sampled rows.
    wl = cs.WORKLOADS["ulysses_128k"]
    dm = wl.dims
    p, n_loc, H, d, g = dm["p"], dm["n_loc"], dm["H"], dm["d"], dm["g"]
    Hl, n = H // p, p * n_loc
    scale = d ** -0.5
    shards = [cs.shard_inputs(p, n_loc, H, d, seed=wl.seed + t) for t in range(3)]
    heads = []
    for x in shards:
        raw, shape = orc.relayout(x, p, g)
        heads.append(torch.from_numpy(raw).view(torch.bfloat16).reshape(shape))
    rows = _ulysses_rows(Hl, n, seed=41)
    ro, rl = orc.softmax_fwd(heads[0], heads[1], heads[2], scale, True, rows=rows)

    def check(o_hm, lse, what):
        o_hm, lse = o_hm.cpu(), lse.cpu()
        assert_fwd_close(o_hm[rows[:, 0], rows[:, 1]], ro, f"{what} sampled O")
        assert_lse_close(lse[rows[:, 0], rows[:, 1]], rl, f"{what} sampled LSE")

    sd = [x.cuda() for x in shards]
    # the step's calls: sp_relayout of Q, K, V, then chain_fwd_f16pv
    hm = [cg.relayout(x, p, g) for x in sd]
    o, lse = cg.attention_fwd_f16pv(hm[0], hm[1], hm[2], True, scale)
    assert cg.chain_check()[0] == 0
    check(o, lse, "relayout + chain_fwd_f16pv")
    del hm, o
    # fused: read from and written back to the shards
    for name, fn in (("chain_fwd_sp_f16pv", cg.attention_fwd_sp_f16pv),
                     ("chain_fwd_sp", cg.attention_fwd_sp)):
        o_sh, lse = fn(sd[0], sd[1], sd[2], p, g, True, scale)
        assert cg.chain_check()[0] == 0
        raw, shape = orc.relayout(o_sh.cpu(), p, g)
        check(torch.from_numpy(raw).view(torch.bfloat16).reshape(shape), lse, name)
        del o_sh
