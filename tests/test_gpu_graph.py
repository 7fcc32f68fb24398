"""GPU: the entry points inside a CUDA graph.

One call of each kind (the f16 P V forward with its V pre-pass, the
backward reading that forward's O and LSE, the f16-intermediate MLP with its
W2 pre-pass and its programmatically chained launches, and the relayout) is
captured into one graph.  Two replays must reproduce the results of the same
calls run eagerly, bit for bit: every kernel here is deterministic (no
atomics, fixed reduction orders)."""
import pytest
import torch

import chain_synth as cs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    import chain_gb300
    chain_gb300.lib()
    return chain_gb300


def test_graph_replay_matches_eager(cg):
    dev = "cuda"
    BH, n, d = 2, 1024, 128
    scale = d ** -0.5
    q, k, v, do = (t.to(dev) for t in cs.attn_inputs(BH, n, d, seed=16000, with_do=True))
    x, w1, w2 = (t.to(dev) for t in cs.mlp_inputs(256, 128, 512, 512, seed=16010))
    p, n_loc, H = 4, 256, 8
    shards = cs.shard_inputs(p, n_loc, H, d, seed=16020).to(dev)

    o = torch.empty_like(q)
    lse = torch.empty(BH, n, dtype=torch.float32, device=dev)
    ws_f = torch.empty(cg.chain_fwd_f16pv_workspace_size(q, v), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_b = torch.empty(cg.chain_bwd_workspace_size(q, v), dtype=torch.uint8, device=dev)
    om = torch.empty(256, 512, dtype=torch.bfloat16, device=dev)
    ws_m = torch.empty(cg.chain_fwd_f16h_workspace_size(w2), dtype=torch.uint8, device=dev)
    hm = torch.empty(H // p, p * n_loc, d, dtype=torch.bfloat16, device=dev)
    outs = (o, lse, dq, dk, dv, om, hm)

    def calls():
        cg.chain_fwd_f16pv(q, k, v, cg.MASK_CAUSAL, scale, o, lse, ws_f)
        cg.chain_bwd(do, q, k, v, o, lse, cg.F_SOFTMAX, cg.MASK_CAUSAL, scale, dq, dk, dv, ws_b)
        cg.chain_fwd_f16h(x, w1, w2, cg.F_GELU_TANH, om, ws_m)
        cg.sp_relayout(shards, p, 1, hm)

    calls()
    torch.cuda.synchronize()
    assert cg.chain_check()[0] == 0
    ref = [t.clone() for t in outs]

    # warm up on a side stream, then capture (the usual order for graphs)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for _ in range(2):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert cg.chain_check()[0] == 0
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV", "MLP O", "relayout"), outs, ref):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{name} differs after replay"
