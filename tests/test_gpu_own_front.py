"""The one-launch layer for at most eight tokens: the decode kernel routes its tokens and
builds the plan itself.  Checked bit for bit against the split steps (router, plan, forward
as separate calls), against the oracle, and for the plan it leaves in the workspace."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_helpers import assert_parity, bf16_tensor, device_weights
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(T, d, F, E, k, seed, tag):
    cfg = mi.CONFIGS["tiny"].replace(name=f"own{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=tag)
    return cfg, mi.gen_layer(cfg, seed=seed)


def _one_launch_applies(moe, shape):
    return shape.T <= 8 and moe.auto_algo(shape) == 3 and moe.unroute_fused(shape, 0)


# (T, d, F, E, k): one token; the headline shape; the largest route count (8 x 32); E above 512
# (32 logits per lane in the router); every token on every expert (E = k); small experts
@pytest.mark.parametrize("T,d,F,E,k", [(1, 2048, 512, 512, 10), (4, 2048, 512, 512, 10), (8, 2048, 512, 512, 32),
                                       (8, 256, 256, 1000, 32), (5, 512, 256, 64, 8), (8, 256, 256, 8, 8),
                                       (2, 1024, 2048, 16, 16), (7, 256, 1024, 40, 3)])
def test_one_launch_layer_matches_split_steps_and_oracle(T, d, F, E, k):
    import routed_moe_decode_gb300 as moe
    cfg, inp = _inputs(T, d, F, E, k, seed=11, tag=400 + T)
    one = moe.MoeLayer(T, d, F, E, k)
    assert _one_launch_applies(moe, one.shape)
    w = device_weights(inp, "cuda")
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    outs = [one(logits, hidden, w, res) for _ in range(3)]  # the counter sets alternate
    split = moe.MoeLayer(T, d, F, E, k, algo=3)  # router, plan, forward as separate calls
    ref = split(logits, hidden, w, res)
    torch.cuda.synchronize()
    assert one.status() == 0 and split.status() == 0
    assert torch.equal(one.ids, split.ids) and torch.equal(one.weights, split.weights)
    for o in outs:
        assert torch.equal(o, ref)
    ids_ref, w_ref = O.route_topk(inp["logits"], k)
    np.testing.assert_array_equal(one.ids.cpu().numpy(), ids_ref)
    oref = O.moe_experts((T, d, F, E, k), inp["hidden"], ids_ref, w_ref, inp, inp["residual"], None)
    assert_parity(outs[0].float().cpu().numpy(), oref, cfg.name)


@pytest.mark.parametrize("T,E,k", [(4, 512, 10), (8, 8, 8), (3, 1000, 32)])
def test_one_launch_layer_leaves_the_plan(T, E, k):
    # the workspace holds the same buckets as moe_plan writes; positions within a bucket may
    # differ (route order here, arrival order there) but must be a valid bucketing
    import routed_moe_decode_gb300 as moe
    d, F = 256, 256
    cfg, inp = _inputs(T, d, F, E, k, seed=12, tag=420 + T)
    one = moe.MoeLayer(T, d, F, E, k)
    assert _one_launch_applies(moe, one.shape)
    w = device_weights(inp, "cuda")
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    out = one(logits, hidden, w, None)
    split = moe.MoeLayer(T, d, F, E, k, algo=3)
    ref = split(logits, hidden, w, None)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    a = moe.plan_views(one.shape, one.ws)
    b = moe.plan_views(split.shape, split.ws)
    U, _ = moe.plan_summary(one.shape, one.ws)
    assert (U, _) == moe.plan_summary(split.shape, split.ws)
    for key in ("counts", "offsets"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["touched"][:U], b["touched"][:U])
    R = T * k
    pos = a["route_pos"].cpu().numpy()[:R]
    tok = a["pos_token"].cpu().numpy()[:R]
    ids = one.ids.cpu().numpy().reshape(-1)
    offsets = a["offsets"].cpu().numpy()
    assert sorted(pos.tolist()) == list(range(R))
    for r in range(R):
        assert tok[pos[r]] == r // k
        assert offsets[ids[r]] <= pos[r] < offsets[ids[r] + 1]
    # a forward on the left plan (hidden staged again) gives the layer's output
    again = one.experts(hidden, w, None)
    torch.cuda.synchronize()
    assert torch.equal(again, out)


def test_one_launch_layers_interleaved_with_other_calls():
    # one-launch layers with new routing each time, between them forwards on the left plan
    # and a layer of the split steps on the same workspace; every output against the oracle
    import routed_moe_decode_gb300 as moe
    T, d, F, E, k = 4, 512, 256, 64, 8
    layer = moe.MoeLayer(T, d, F, E, k)
    assert _one_launch_applies(moe, layer.shape)
    cfg, inp0 = _inputs(T, d, F, E, k, seed=13, tag=440)
    w = device_weights(inp0, "cuda")
    for step in range(5):
        inp = mi.gen_layer(cfg, seed=100 + step, weights=False)
        logits = torch.from_numpy(inp["logits"]).cuda()
        hidden = bf16_tensor(inp["hidden"], "cuda")
        res = bf16_tensor(inp["residual"], "cuda")
        out = layer(logits, hidden, w, res)
        reuse = layer.experts(hidden, w, res)
        layer.route(logits)  # the split steps, on the same workspace
        layer.plan()
        split = layer.experts(hidden, w, res)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(out, reuse) and torch.equal(out, split)
        ids_ref, w_ref = O.route_topk(inp["logits"], k)
        oref = O.moe_experts((T, d, F, E, k), inp["hidden"], ids_ref, w_ref, inp0, inp["residual"], None)
        assert_parity(out.float().cpu().numpy(), oref, f"interleaved step {step}")


def test_one_launch_layer_in_a_cuda_graph():
    # eight layers captured once and replayed with new inputs: the counter-set parity is
    # device state, so replays alternate it like eager calls
    import routed_moe_decode_gb300 as moe
    T, d, F, E, k = 2, 256, 256, 32, 4
    layer = moe.MoeLayer(T, d, F, E, k)
    assert _one_launch_applies(moe, layer.shape)
    cfg, inp0 = _inputs(T, d, F, E, k, seed=14, tag=450)
    w = device_weights(inp0, "cuda")
    L = 8
    logits = torch.zeros((L, T, E), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((L, T, d), dtype=torch.bfloat16, device="cuda")
    outs = torch.zeros((L, T, d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(logits[0], hidden[0], w, None, outs[0])  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(L):
            layer(logits[i], hidden[i], w, None, outs[i])
    for rep in range(3):
        refs = []
        for i in range(L):
            inp = mi.gen_layer(cfg, seed=200 + 10 * rep + i, weights=False)
            logits[i].copy_(torch.from_numpy(inp["logits"]))
            hidden[i].copy_(bf16_tensor(inp["hidden"], "cuda"))
            refs.append(inp)
        g.replay()
        torch.cuda.synchronize()
        assert layer.status() == 0
        for i, inp in enumerate(refs):
            ids_ref, w_ref = O.route_topk(inp["logits"], k)
            oref = O.moe_experts((T, d, F, E, k), inp["hidden"], ids_ref, w_ref, inp0, None, None)
            assert_parity(outs[i].float().cpu().numpy(), oref, f"graph replay {rep} layer {i}")
