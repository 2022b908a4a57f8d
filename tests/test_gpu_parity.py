"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing ids must match bit for bit; routing weights within 2e-6 relative; the layer
output within max|d| <= 2e-2 * RMS(ref) and sum|d| / sum|ref| <= 5e-3.  Small workloads
are compared on every output; the full-size workloads on every routing id and on the
outputs of a sample of tokens the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_helpers import (MAX_ABS_OVER_RMS, MEAN_REL, WEIGHT_RTOL, assert_parity, bf16_tensor, config_inputs,
                         device_weights, parity_metrics, run_layer)
from oracle import oracle as O

pytestmark = pytest.mark.gpu

ALGOS = {"auto": 0, "tcgen05": 1, "simt": 2, "mma": 3, "wide": 4}

# tokens checked against the oracle at full size (all tokens when None)
SAMPLES = {
    "tiny": None,
    "b1": None,
    "b8": [0, 1, 2, 3, 13, 22, 30, 31],
    "b64": [0, 1, 37, 100, 128, 200, 254, 255],
    "b64_literal": [0, 5, 77, 255],
    "prefill": [0, 1, 2, 1000, 4095, 6000, 8190, 8191],
}


@pytest.fixture(scope="module", autouse=True)
def _build():
    import __graft_entry__
    __graft_entry__.build()


def _check_layer(cfg, inp, algo, tokens=None, residual=True):
    ids, wts, out, layer = run_layer(cfg, inp, algo=algo, residual=residual)
    assert layer.status() == 0
    ids_ref, w_ref = O.route_topk(inp["logits"], cfg.k)
    np.testing.assert_array_equal(ids, ids_ref)
    np.testing.assert_allclose(wts, w_ref, rtol=WEIGHT_RTOL, atol=1e-7)
    mask = None
    if tokens is not None:
        mask = np.zeros(cfg.T, np.uint8)
        mask[tokens] = 1
    res = inp["residual"] if residual else None
    ref = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids_ref, w_ref, inp, res, mask)
    rows = slice(None) if tokens is None else tokens
    return assert_parity(out[rows], ref[rows], f"{cfg.name} algo {algo}")


@pytest.mark.parametrize("name", ["b1", "b8", "b64", "b64_literal", "prefill"])
def test_layer_parity_mma(name):
    cfg = mi.CONFIGS[name]
    _check_layer(cfg, config_inputs(name), ALGOS["mma"], SAMPLES[name])


@pytest.mark.parametrize("name", ["tiny", "b1", "b8", "b64", "prefill"])
def test_layer_parity_auto(name):
    # the one-call layer: fused router + plan front (T * k <= 16384), separate kernels above
    cfg = mi.CONFIGS[name]
    _check_layer(cfg, config_inputs(name), ALGOS["auto"], SAMPLES[name])


@pytest.mark.parametrize("T,d,F,E,k", [(4, 2048, 512, 512, 10), (33, 512, 256, 64, 8), (100, 256, 256, 1000, 7),
                                       (256, 2048, 512, 512, 10), (64, 256, 512, 16, 1), (1638, 256, 256, 64, 10),
                                       (1639, 256, 256, 64, 10)])
def test_fused_front_matches_separate_calls(T, d, F, E, k):
    # one moe_layer call (multi-CTA fronts, the last one building the plan; the last shape
    # has T * k just above the fused front's limit) against router + plan + forward
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["tiny"].replace(name=f"front{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=300 + T)
    inp = mi.gen_layer(cfg, seed=6)
    w = device_weights(inp, "cuda")
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    fused = moe.MoeLayer(T, d, F, E, k)
    outs = [fused(logits, hidden, w, res) for _ in range(3)]  # the arrival counter resets itself
    sep = moe.MoeLayer(T, d, F, E, k, algo=moe.auto_algo(fused.shape))
    ref = sep(logits, hidden, w, res)
    torch.cuda.synchronize()
    assert fused.status() == 0 and sep.status() == 0
    assert torch.equal(fused.ids, sep.ids) and torch.equal(fused.weights, sep.weights)
    for o in outs:
        assert torch.equal(o, ref)
    assert moe.plan_summary(fused.shape, fused.ws) == moe.plan_summary(sep.shape, sep.ws)


@pytest.mark.parametrize("algo", ["mma", "tcgen05", "simt", "wide"])
def test_split_expert_and_unroute_calls(algo):
    # moe_forward_expert_kernels + moe_forward_unroute == moe_forward_experts, bit for bit
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["b8"]
    inp = config_inputs("b8")
    w = device_weights(inp, "cuda")
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k, algo=ALGOS[algo])
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    ref = layer(logits, hidden, w, res)
    moe.forward_prepare(layer.shape, hidden, layer.ws)
    moe.forward_expert_kernels(layer.shape, w, layer.ws, ALGOS[algo])
    out = torch.empty_like(ref)
    moe.forward_unroute(layer.shape, res, out, layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("name", ["tiny", "b1", "b8", "b64", "prefill"])
def test_layer_parity_tcgen05(name):
    cfg = mi.CONFIGS[name]
    _check_layer(cfg, config_inputs(name), ALGOS["tcgen05"], SAMPLES[name])


@pytest.mark.parametrize("name", ["tiny", "b1", "b8", "b64", "prefill"])
def test_layer_parity_wide(name):
    cfg = mi.CONFIGS[name]
    _check_layer(cfg, config_inputs(name), ALGOS["wide"], SAMPLES[name])


@pytest.mark.parametrize("T,d,F,E,k", [(400, 256, 128, 4, 2), (1000, 512, 256, 8, 2), (300, 384, 384, 3, 1),
                                       (385, 256, 256, 2, 1), (17, 128, 128, 1, 1), (190, 1024, 512, 32, 32)])
def test_wide_path_many_rows(T, d, F, E, k):
    # (400, .., E=4, k=2): ~200 rows per expert, (1000, .., 8, 2): ~250, (385, .., 2, 1): two
    # passes of 192 and a ragged third; (190, .., 32, 32): every expert holds all 190 rows
    cfg = mi.CONFIGS["tiny"].replace(name=f"wide{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=300 + T)
    inp = mi.gen_layer(cfg, seed=6)
    _check_layer(cfg, inp, ALGOS["wide"])


@pytest.mark.parametrize("name", ["tiny", "b1", "b8"])
def test_layer_parity_simt(name):
    cfg = mi.CONFIGS[name]
    _check_layer(cfg, config_inputs(name), ALGOS["simt"], SAMPLES[name])


def test_last_layer_weight_set_parity():
    cfg = mi.CONFIGS["b1"]
    _check_layer(cfg, mi.gen_layer(cfg, seed=0, layer=11), ALGOS["auto"])


@pytest.mark.parametrize("T,d,F,E,k", [(1, 256, 128, 16, 1), (5, 256, 128, 16, 2), (33, 512, 256, 64, 8),
                                       (100, 256, 128, 32, 4), (3, 384, 384, 1000, 7), (7, 128, 128, 40, 32),
                                       (64, 1024, 256, 16, 16)])
def test_ragged_and_edge_shapes(T, d, F, E, k):
    cfg = mi.CONFIGS["tiny"].replace(name=f"edge{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=100 + T)
    inp = mi.gen_layer(cfg, seed=3)
    _check_layer(cfg, inp, ALGOS["auto"])
    _check_layer(cfg, inp, ALGOS["tcgen05"])
    _check_layer(cfg, inp, ALGOS["wide"])


@pytest.mark.parametrize("T,d,F,E,k", [(1, 256, 256, 16, 1), (5, 512, 256, 16, 2), (33, 512, 512, 64, 8),
                                       (100, 256, 256, 32, 4), (7, 1024, 256, 40, 32), (64, 1024, 256, 16, 16),
                                       (130, 256, 256, 4, 4), (9, 512, 1024, 16, 4), (9, 256, 2048, 8, 2)])
def test_mma_path_shapes(T, d, F, E, k):
    # (130, ..., E=4, k=4): every expert holds all 130 rows -> three 64-row passes
    cfg = mi.CONFIGS["tiny"].replace(name=f"mma{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=200 + T)
    inp = mi.gen_layer(cfg, seed=4)
    _check_layer(cfg, inp, ALGOS["mma"])


def test_mma_path_rejects_unsupported_shape():
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["tiny"]  # ffn = 128 is below the 256-element chunk
    with pytest.raises(moe.MoeError):
        run_layer(cfg, dict(config_inputs("tiny")), algo=ALGOS["mma"])
    cfg = cfg.replace(name="mma_d768", d=768, ffn=256)  # not a power of two
    with pytest.raises(moe.MoeError):
        run_layer(cfg, mi.gen_layer(cfg, seed=5), algo=ALGOS["mma"])


def _route_only(logits, k):
    import routed_moe_decode_gb300 as moe
    T, E = logits.shape
    shape = moe.shape_of(T, 128, 128, E, k)
    dl = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.route_topk(shape, dl, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("E,k", [(512, 10), (64, 8), (16, 2), (1000, 32), (33, 32)])
def test_route_ties_and_signed_zero(E, k):
    rng = np.random.default_rng(E + k)
    T = 300
    logits = (rng.integers(-3, 4, size=(T, E)) * 0.25).astype(np.float32)  # heavy ties
    logits[:10] = 0.0
    logits[5:10, ::3] = -0.0  # -0 and +0 compare equal: lower index wins
    ids, w = _route_only(logits, k)
    ids_ref, w_ref = O.route_topk(logits, k)
    np.testing.assert_array_equal(ids, ids_ref)
    np.testing.assert_allclose(w, w_ref, rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.parametrize("E,k", [(512, 10), (1024, 32), (96, 12), (1000, 32), (510, 10)])
@pytest.mark.parametrize("layout", ["mod32", "block"])
def test_route_winners_concentrated_in_few_experts(E, k, layout):
    # every winner sits in one or two groups of experts: ids of one residue mod 32, or one
    # contiguous block of E/32 ids -- the ids one warp lane of the router holds -- so one lane
    # holds more winners than it keeps sorted at a time and must rebuild its list
    rng = np.random.default_rng(7 * E + k)
    T = 64
    npl = 1 << max(0, int(np.ceil(np.log2(max(1, (E + 31) // 32)))))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    for t in range(T):
        lanes = [t % 32] if t % 2 == 0 else [t % 32, (t * 7 + 3) % 32]
        for ln in lanes:
            sel = np.arange(ln, E, 32) if layout == "mod32" else np.arange(ln * npl, min(E, ln * npl + npl))
            if sel.size == 0:
                continue
            logits[t, sel] = 10.0 + rng.standard_normal(sel.size).astype(np.float32)
            if t % 4 == 0:
                logits[t, sel[::2]] = 11.0  # exact ties inside the group
    ids, w = _route_only(logits, k)
    ids_ref, w_ref = O.route_topk(logits, k)
    np.testing.assert_array_equal(ids, ids_ref)
    np.testing.assert_allclose(w, w_ref, rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.parametrize("name", ["b1", "b8", "b64", "prefill"])
def test_route_full_size_bit_exact(name):
    cfg = mi.CONFIGS[name]
    for layer in (0, 5):
        logits = mi.gen_logits(cfg, 0, layer)
        ids, w = _route_only(logits, cfg.k)
        ids_ref, w_ref = O.route_topk(logits, cfg.k)
        np.testing.assert_array_equal(ids, ids_ref)
        np.testing.assert_allclose(w, w_ref, rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", "b8", "b64", "prefill"])
def test_plan_matches_oracle_bucketing(name):
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS[name]
    logits = mi.gen_logits(cfg, 0, 0)
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    layer.route(torch.from_numpy(logits).cuda())
    layer.plan()
    torch.cuda.synchronize()
    ids = layer.ids.cpu().numpy()
    counts, offsets, touched = O.plan(ids, cfg.E)
    v = {key: t.cpu().numpy() for key, t in moe.plan_views(layer.shape, layer.ws).items()}
    U, maxrows = moe.plan_summary(layer.shape, layer.ws)
    np.testing.assert_array_equal(v["counts"], counts)
    np.testing.assert_array_equal(v["offsets"], offsets)
    assert U == len(touched) and maxrows == counts.max()
    np.testing.assert_array_equal(v["touched"][:U], touched)
    # route positions: a bijection onto [0, T*k) that keeps each route inside its expert's segment
    pos = v["route_pos"]
    assert sorted(pos.tolist()) == list(range(cfg.T * cfg.k))
    e_of_route = ids.ravel()
    assert np.all(pos >= offsets[e_of_route]) and np.all(pos < offsets[e_of_route + 1])
    np.testing.assert_array_equal(v["pos_token"][pos], np.arange(cfg.T * cfg.k) // cfg.k)
    assert layer.status() == 0


def test_bad_expert_id_sets_status():
    import routed_moe_decode_gb300 as moe
    shape = moe.shape_of(4, 256, 128, 16, 2)
    ws = moe.Workspace(shape)
    ids = torch.tensor([[0, 1], [2, 16], [3, 4], [5, -1]], dtype=torch.int32, device="cuda")
    w = torch.full((4, 2), 0.5, device="cuda")
    moe.plan(shape, ids, w, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) & moe.MOE_DEV_BAD_EXPERT_ID
    assert moe.read_status(ws) == 0  # cleared by the first read


def test_zero_hidden_gives_residual_exactly():
    cfg = mi.CONFIGS["b1"]
    inp = dict(config_inputs("b1"))
    inp["hidden"] = np.zeros_like(inp["hidden"])
    _, _, out, _ = run_layer(cfg, inp, algo=0)
    res = (inp["residual"].astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(out, res)


def test_no_residual_and_out_aliasing_residual():
    cfg = mi.CONFIGS["b8"]
    inp = config_inputs("b8")
    _check_layer(cfg, inp, 0, SAMPLES["b8"], residual=False)
    import routed_moe_decode_gb300 as moe
    w = device_weights(inp, "cuda")
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    hidden = bf16_tensor(inp["hidden"], "cuda")
    buf = bf16_tensor(inp["residual"], "cuda").clone()
    ref_out = layer(torch.from_numpy(inp["logits"]).cuda(), hidden, w, buf.clone())
    out = layer(torch.from_numpy(inp["logits"]).cuda(), hidden, w, buf, out=buf)  # in place
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)


def _shared_or_disjoint_logits(T, E, k, shared):
    logits = np.random.default_rng(9).standard_normal((T, E)).astype(np.float32)
    if shared:  # every token on the same k experts
        logits[:, 7:7 + k] += 50.0
    else:  # no two tokens share an expert
        for t in range(T):
            logits[t, t * k:(t + 1) * k] += 50.0
    return logits


@pytest.mark.parametrize("shared,T", [(True, 4), (True, 64), (True, 100), (False, 32)])
def test_all_equal_and_all_disjoint_routing(shared, T):
    cfg = mi.CONFIGS["b1"].replace(name=f"route_shared{shared}{T}", T=T, tag=50 + T)
    inp = dict(config_inputs("b1"))  # b1's weights; this workload's own activations
    inp.update(mi.gen_layer(cfg, seed=1, weights=False))
    inp["logits"] = _shared_or_disjoint_logits(T, cfg.E, cfg.k, shared)
    tokens = None if T <= 32 else [0, 1, T // 2, T - 1]
    _check_layer(cfg, inp, 0, tokens)


def test_all_experts_identical_output_independent_of_routing():
    cfg = mi.CONFIGS["tiny"].replace(name="same_experts", T=16, tag=77)
    inp = dict(mi.gen_layer(cfg, seed=2))
    for key in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        inp[key] = np.ascontiguousarray(np.broadcast_to(inp[key][:1], inp[key].shape))
    _, _, a, _ = run_layer(cfg, inp, algo=0)
    inp2 = dict(inp, logits=np.ascontiguousarray(inp["logits"][:, ::-1]))
    _, _, b, _ = run_layer(cfg, inp2, algo=0)
    mx, mean_rel = parity_metrics(a, b)
    assert mx < 2e-2 and mean_rel < 2e-3
    _check_layer(cfg, inp, 0)


def test_repeat_is_bitwise_deterministic_and_forward_reuses_plan():
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["b8"]
    inp = config_inputs("b8")
    w = device_weights(inp, "cuda")
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    first = layer(logits, hidden, w, res)
    outs = [layer.experts(hidden, w, res) for _ in range(3)]  # forward again on the same plan
    outs.append(layer(logits, hidden, w, res))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, first)
    assert layer.status() == 0


def test_cuda_graph_replays_with_changed_inputs():
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["b8"]
    a = config_inputs("b8", 0, 0)
    b = mi.gen_layer(cfg, seed=0, layer=1, weights=False)
    w = device_weights(a, "cuda")
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits = torch.from_numpy(a["logits"]).cuda()
    hidden = bf16_tensor(a["hidden"], "cuda")
    res = bf16_tensor(a["residual"], "cuda")
    out = torch.empty_like(res)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(logits, hidden, w, res, out=out)  # warm-up (and per-device setup) outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(logits, hidden, w, res, out=out)
    for src in (b, a, b):
        logits.copy_(torch.from_numpy(src["logits"]))
        hidden.copy_(bf16_tensor(src["hidden"], "cuda"))
        res.copy_(bf16_tensor(src["residual"], "cuda"))
        g.replay()
        torch.cuda.synchronize()
        ids_ref, w_ref = O.route_topk(src["logits"], cfg.k)
        np.testing.assert_array_equal(layer.ids.cpu().numpy(), ids_ref)
        toks = SAMPLES["b8"][:4]
        mask = np.zeros(cfg.T, np.uint8)
        mask[toks] = 1
        ref = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), src["hidden"], ids_ref, w_ref, a,
                            src["residual"], mask)
        assert_parity(out.float().cpu().numpy()[toks], ref[toks], "graph replay")
    assert layer.status() == 0


def test_hidden_out_of_fp16_range_sets_status():
    cfg = mi.CONFIGS["tiny"]
    inp = dict(config_inputs("tiny"))
    hid = inp["hidden"].copy()
    hid[1, 3] = 0x4780  # bf16 65536.0, above the FP16 maximum
    inp["hidden"] = hid
    _, _, _, layer = run_layer(cfg, inp, algo=0)
    import routed_moe_decode_gb300 as moe
    assert layer.status() & moe.MOE_DEV_HIDDEN_RANGE


def _shard_partial_oracle(cfg, inp, ids, wts, e_begin, e_end, residual):
    """Oracle of one expert shard: the slots of other shards' experts get weight 0, so they
    add exactly nothing; the residual is added by one shard only."""
    w = np.where((ids >= e_begin) & (ids < e_end), wts, 0.0).astype(np.float32)
    return O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids, w, inp,
                         inp["residual"] if residual else None)


@pytest.mark.parametrize("name,bounds", [
    ("tiny", (0, 8, 16)), ("b1", (0, 128, 256, 384, 512)), ("b8", (0, 200, 512)),
    ("ep2048x256x128x64x16", (0, 32, 64)),   # 32768 routes: multi-CTA plan and the wide kernel
])
def test_expert_parallel_shards_sum_to_layer(name, bounds):
    """moe_layer_expert_range on each shard of a partition of the experts (local weights
    only, residual on the first shard): every shard matches its partial oracle, the ids
    agree across shards, and the shards' outputs summed in FP32 match the whole layer."""
    import routed_moe_decode_gb300 as moe
    if name in mi.CONFIGS:
        cfg = mi.CONFIGS[name]
        inp = config_inputs(name)
    else:
        cfg = mi.CONFIGS["tiny"].replace(name=name, T=2048, d=256, ffn=128, E=64, k=16, tag=400)
        inp = mi.gen_layer(cfg, seed=7)
    dev = torch.device("cuda")
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    res = bf16_tensor(inp["residual"], dev)
    ids_ref, wts_ref = O.route_topk(inp["logits"], cfg.k)
    full = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids_ref, wts_ref, inp, inp["residual"])
    full64 = full.astype(np.float64)
    rms, l1 = float(np.sqrt(np.mean(full64 ** 2))), float(np.abs(full64).sum())
    total = np.zeros((cfg.T, cfg.d), np.float64)
    for si, (e0, e1) in enumerate(zip(bounds[:-1], bounds[1:])):
        local = {n: np.ascontiguousarray(inp[n][e0:e1]) for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")}
        local["w13_ts"], local["w2_ts"] = inp["w13_ts"], inp["w2_ts"]
        w = device_weights(local, dev)
        ws = moe.Workspace(shape)
        ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
        wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
        out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
        moe.layer_expert_range(shape, e0, e1, logits, hidden, w, res if si == 0 else None, out, ids, wts, ws)
        torch.cuda.synchronize()
        assert moe.read_status(ws) == 0
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        got = out.float().cpu().numpy()
        ref = _shard_partial_oracle(cfg, inp, ids_ref, wts_ref, e0, e1, si == 0)
        # a shard's output is part of the layer's: its error is measured on the layer's scale
        err = np.abs(got.astype(np.float64) - ref)
        assert np.all(np.isfinite(got))
        assert err.max() <= MAX_ABS_OVER_RMS * rms and err.sum() <= MEAN_REL * l1, \
            f"{name} shard [{e0},{e1}): max|d| {err.max():.3g} (rms {rms:.3g}), sum|d| / sum|layer| {err.sum() / l1:.3e}"
        total += got
    assert_parity(total.astype(np.float32), full, f"{name} sum of {len(bounds) - 1} shards")


@pytest.mark.parametrize("name,e0,e1", [("b1", 128, 384), ("b8", 0, 200), ("tiny", 9, 16)])
def test_expert_range_plan_forward_pair_matches_one_call(name, e0, e1):
    """moe_route_topk + moe_plan_expert_range + moe_forward_prepare +
    moe_forward_experts_expert_range (the range passed to each call) gives the bits of one
    moe_layer_expert_range call."""
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS[name]
    inp = config_inputs(name)
    dev = torch.device("cuda")
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    res = bf16_tensor(inp["residual"], dev)
    local = {n: np.ascontiguousarray(inp[n][e0:e1]) for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")}
    local["w13_ts"], local["w2_ts"] = inp["w13_ts"], inp["w2_ts"]
    w = device_weights(local, dev)
    outs = []
    for split in (False, True):
        ws = moe.Workspace(shape)
        ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
        wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
        out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
        if split:
            moe.route_topk(shape, logits, ids, wts)
            moe.plan_expert_range(shape, e0, e1, ids, wts, ws)
            moe.forward_prepare(shape, hidden, ws)
            moe.forward_experts_expert_range(shape, e0, e1, w, res, out, ws)
        else:
            moe.layer_expert_range(shape, e0, e1, logits, hidden, w, res, out, ids, wts, ws)
        torch.cuda.synchronize()
        assert moe.read_status(ws) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_expert_range_rejects_bad_bounds():
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["tiny"]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    for e0, e1 in ((-1, 4), (4, 4), (8, 17), (9, 3)):
        with pytest.raises(moe.MoeError):
            moe.layer_expert_range(shape, e0, e1, None, None, {"w13_codes": None, "w13_scales": None, "w13_ts": 1.0,
                                                              "w2_codes": None, "w2_scales": None, "w2_ts": 1.0},
                                   None, None, None, None, moe.Workspace(shape))


@pytest.mark.parametrize("T,d,F,E,k,algo", [(512, 256, 256, 16, 2, "wide"), (256, 512, 256, 32, 4, "wide"),
                                            (32, 256, 256, 64, 8, "mma"), (4, 256, 128, 16, 2, "tcgen05")])
def test_expert_kernel_parts_equal_the_whole(T, d, F, E, k, algo):
    # moe_selftest_expert_part: the preparing kernels (part 0) then the expert kernel alone
    # (part 1) leave exactly what moe_forward_expert_kernels leaves
    import routed_moe_decode_gb300 as moe
    cfg = mi.CONFIGS["tiny"].replace(name=f"parts{T}x{d}x{F}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=700 + T)
    inp = mi.gen_layer(cfg, seed=21)
    layer = moe.MoeLayer(T, d, F, E, k, algo=ALGOS[algo])
    w = device_weights(inp, "cuda")
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    outs = []
    for split in (False, True):
        layer.route(logits)
        layer.plan()
        moe.forward_prepare(layer.shape, hidden, layer.ws)
        if split:
            moe.selftest_expert_part(layer.shape, w, layer.ws, ALGOS[algo], 0)
            moe.selftest_expert_part(layer.shape, w, layer.ws, ALGOS[algo], 1)
        else:
            moe.forward_expert_kernels(layer.shape, w, layer.ws, ALGOS[algo])
        out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        moe.forward_unroute(layer.shape, res, out, layer.ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(outs[0], outs[1])
    ids_ref, w_ref = O.route_topk(inp["logits"], k)
    ref = O.moe_experts((T, d, F, E, k), inp["hidden"], ids_ref, w_ref, inp, inp["residual"], None)
    assert_parity(outs[1].float().cpu().numpy(), ref, f"parts {algo}")


@pytest.mark.parametrize("T,E,k", [(32, 64, 8), (512, 16, 2)])
def test_layer_without_plan_table_then_other_algorithm_finds_no_tasks(T, E, k):
    # a layer whose expert kernel derives its own tasks (gathered decode kernel at 8 < T <=
    # 256, the wide kernel for many rows per expert) leaves the plan's task table unwritten and
    # its task counts at 0; a later forward on that plan with MOE_ALGO_TCGEN05 (which reads the
    # table) finds no tasks and returns with a clean status (its un-route sums whatever
    # per-route outputs the workspace holds); AUTO on the same plan reproduces the layer
    import routed_moe_decode_gb300 as moe
    d, F = 256, 256
    cfg = mi.CONFIGS["tiny"].replace(name=f"notable{T}x{E}x{k}", T=T, d=d, ffn=F, E=E, k=k, tag=800 + T)
    inp = mi.gen_layer(cfg, seed=23)
    layer = moe.MoeLayer(T, d, F, E, k)
    assert moe.auto_algo(layer.shape) in (ALGOS["mma"], ALGOS["wide"])
    w = device_weights(inp, "cuda")
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    out = layer(logits, hidden, w, res)
    again = layer.experts(hidden, w, res)  # AUTO on the left plan
    other = torch.empty_like(out)
    moe.forward_experts(layer.shape, w, res, other, layer.ws, ALGOS["tcgen05"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(again, out)
    assert torch.isfinite(other.float()).all()
