"""The steps on either side of the layer, on the GPU against the oracle.

Router projection (moe_router_logits, moe_layer_from_hidden): logits = hidden x Wr^T with BF16
inputs and FP32 sums ("Router: selection and expert-task production" of "Persistent execution
for Flash-Next GGUF on SM70").  The kernel's sums run in another order than the oracle's, so
its logits are compared within the FP32 accumulation bound; the routing, an integer decision
taken on floats, is then checked in the kernel's precision: the GPU's ids must equal the
oracle's router applied to the GPU's logits, bit for bit.

Gated residual update + GemmaRMSNorm (moe_forward_unroute_gated, moe_layer_gated), TokenSpeed's
"Residual update and normalization fusion": both outputs are BF16 on both sides, so an element
may differ by one BF16 step where the two FP32 values straddle a rounding boundary; the
comparison allows that step (2^-7 |ref|) on top of max|d| <= 2e-2 RMS and keeps mean rel <= 5e-3.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_helpers import (MAX_ABS_OVER_RMS, MEAN_REL, assert_parity, bf16_tensor, config_inputs, device_weights,
                         parity_metrics)
from oracle import oracle as O

pytestmark = pytest.mark.gpu

BF16_STEP_REL = 2.0 ** -7


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_moe_decode_gb300 as m
    return m


def _f(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def _gpu_logits(moe, cfg, hidden_bits, wr_bits):
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits = torch.full((cfg.T, cfg.E), float("nan"), dtype=torch.float32, device="cuda")
    moe.router_logits(shape, bf16_tensor(hidden_bits, "cuda"), bf16_tensor(wr_bits, "cuda"), logits)
    torch.cuda.synchronize()
    return logits.cpu().numpy()


def _assert_logits_close(got, hidden_bits, wr_bits):
    ref = O.router_logits(hidden_bits, wr_bits)
    # both are FP32 sums of d exact products: each is within d * 2^-24 * sum|x||w| of the exact
    # value, so they are within twice that of each other
    d = hidden_bits.shape[1]
    bound = 2 * d * 2.0 ** -24 * (np.abs(_f(hidden_bits)).astype(np.float64) @ np.abs(_f(wr_bits)).astype(np.float64).T)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got.astype(np.float64) - ref) <= bound + 1e-30)


@pytest.mark.parametrize("T,d,E", [(1, 256, 16), (4, 2048, 512), (7, 512, 64), (33, 1024, 128), (300, 256, 48)])
def test_router_logits_within_fp32_accumulation_bound(moe, T, d, E):
    cfg = mi.CONFIGS["tiny"].replace(name=f"router{T}x{d}x{E}", T=T, d=d, E=E, tag=800 + T)
    hidden = mi.gen_hidden(cfg, seed=2)
    wr = mi.gen_router_weight(cfg, seed=2)
    _assert_logits_close(_gpu_logits(moe, cfg, hidden, wr), hidden, wr)


@pytest.mark.parametrize("name", ["b8", "b64", "prefill"])
def test_router_logits_full_size_sampled(moe, name):
    cfg = mi.CONFIGS[name]
    hidden = mi.gen_hidden(cfg, seed=0)
    wr = mi.gen_router_weight(cfg, seed=0)
    got = _gpu_logits(moe, cfg, hidden, wr)
    rows = np.unique(np.linspace(0, cfg.T - 1, 9).astype(int))
    _assert_logits_close(got[rows], hidden[rows], wr)
    again = _gpu_logits(moe, cfg, hidden, wr)
    np.testing.assert_array_equal(again, got)  # fixed-order partial sums: the same bits every run


@pytest.mark.parametrize("name", ["tiny", "b1", "b8"])
def test_layer_from_hidden_routes_on_its_own_logits(moe, name):
    cfg = mi.CONFIGS[name]
    inp = config_inputs(name)
    wr = mi.gen_router_weight(cfg, seed=0)
    dev = "cuda"
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    w = device_weights(inp, dev)
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    moe.layer_from_hidden(shape, bf16_tensor(inp["hidden"], dev), bf16_tensor(wr, dev), logits, w,
                          bf16_tensor(inp["residual"], dev), out, ids, wts, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    lg = logits.cpu().numpy()
    _assert_logits_close(lg, inp["hidden"], wr)
    ids_ref, w_ref = O.route_topk(lg, cfg.k)  # the decision in the kernel's precision
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(wts.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    ref = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids_ref, w_ref, inp, inp["residual"])
    assert_parity(out.float().cpu().numpy(), ref, f"{name} layer from hidden")


def test_router_rejects_unsupported_shapes(moe):
    for T, d, E in ((4, 2048, 500), (4, 2080, 512)):
        shape = moe.shape_of(T, d, 256, E, 2)
        x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
        wr = torch.zeros((E, d), dtype=torch.bfloat16, device="cuda")
        lg = torch.zeros((T, E), dtype=torch.float32, device="cuda")
        with pytest.raises(moe.MoeError):
            moe.router_logits(shape, x, wr, lg)


# ---------------------------------------------------------------- gated residual + GemmaRMSNorm
def _assert_bf16_outputs(got, ref, what):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    assert np.all(np.isfinite(got)), what
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(got - ref) - BF16_STEP_REL * np.abs(ref)
    mean_rel = float(np.abs(got - ref).sum() / np.abs(ref).sum())
    assert excess.max() <= MAX_ABS_OVER_RMS * rms and mean_rel <= MEAN_REL, \
        f"{what}: max excess {excess.max() / rms:.3e} rms, mean rel {mean_rel:.3e}"


def _gated_case(moe, cfg, inp, G, eps, algo=0):
    dev = "cuda"
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    w = device_weights(inp, dev)
    gi = mi.gen_gated_inputs(cfg, G, seed=5)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    branches = bf16_tensor(gi["branches"], dev)
    inject = torch.from_numpy(gi["inject"]).to(dev)
    norm_w = bf16_tensor(gi["norm_w"], dev)
    r_out = torch.empty_like(branches)
    n_out = torch.empty_like(branches)
    if algo == 0:
        moe.layer_gated(shape, G, logits, hidden, w, branches, inject, norm_w, eps, r_out, n_out, ids, wts, ws)
    else:
        moe.front(shape, logits, hidden, ids, wts, ws)
        moe.forward_expert_kernels(shape, w, ws, algo)
        moe.forward_unroute_gated(shape, G, branches, inject, norm_w, eps, r_out, n_out, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    ids_ref, w_ref = O.route_topk(inp["logits"], cfg.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    o_ref = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids_ref, w_ref, inp, None)
    r_ref, n_ref = O.gated_residual_norm(o_ref, gi["branches"], gi["inject"], gi["norm_w"], eps)
    return r_out, n_out, r_ref, n_ref


@pytest.mark.parametrize("name,G", [("tiny", 1), ("tiny", 4), ("b1", 4), ("b8", 4), ("b8", 1)])
def test_layer_gated_matches_oracle(moe, name, G):
    cfg = mi.CONFIGS[name]
    r_out, n_out, r_ref, n_ref = _gated_case(moe, cfg, config_inputs(name), G, 1e-6)
    _assert_bf16_outputs(_f(r_out.view(torch.int16).cpu().numpy().view(np.uint16)), _f(r_ref), f"{name} G={G} R'")
    _assert_bf16_outputs(n_out.float().cpu().numpy(), n_ref, f"{name} G={G} N")


@pytest.mark.parametrize("algo", [1, 3, 4])
def test_gated_unroute_after_each_expert_kernel(moe, algo):
    # tcgen05 (FP32 y), warp-MMA (FP32 y), wide (FP16 y / 16) per-route outputs
    cfg = mi.CONFIGS["tiny"].replace(name="gated_algo", T=96, d=256, ffn=256, E=8, k=2, tag=820)
    inp = mi.gen_layer(cfg, seed=9)
    r_out, n_out, r_ref, n_ref = _gated_case(moe, cfg, inp, 3, 1e-5, algo)
    _assert_bf16_outputs(_f(r_out.view(torch.int16).cpu().numpy().view(np.uint16)), _f(r_ref), f"algo {algo} R'")
    _assert_bf16_outputs(n_out.float().cpu().numpy(), n_ref, f"algo {algo} N")


@pytest.mark.parametrize("name", ["b1", "b8"])
def test_gated_with_unit_gate_is_the_plain_layer(moe, name):
    # one branch, injection logit 0 (2 sigmoid(0) = 1 exactly): R' = BF16(R + O) is the plain
    # layer's out = BF16(residual + O), bit for bit (same slot order, same FP32 operations)
    cfg = mi.CONFIGS[name]
    inp = config_inputs(name)
    dev = "cuda"
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    w = device_weights(inp, dev)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    res = bf16_tensor(inp["residual"], dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    plain = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    moe.layer(shape, logits, hidden, w, res, plain, ids, wts, ws)
    r_out = torch.empty((1, cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    n_out = torch.empty_like(r_out)
    moe.layer_gated(shape, 1, logits, hidden, w, res.view(1, cfg.T, cfg.d), torch.zeros((cfg.T, 1), device=dev),
                    torch.zeros((1, cfg.d), dtype=torch.bfloat16, device=dev), 1e-6, r_out, n_out, ids, wts, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    assert torch.equal(r_out[0], plain)


def test_gated_in_place_residual(moe):
    cfg = mi.CONFIGS["b1"]
    inp = config_inputs("b1")
    dev = "cuda"
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    w = device_weights(inp, dev)
    gi = mi.gen_gated_inputs(cfg, 2, seed=5)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    inject = torch.from_numpy(gi["inject"]).to(dev)
    norm_w = bf16_tensor(gi["norm_w"], dev)
    outs = []
    for in_place in (False, True):
        br = bf16_tensor(gi["branches"], dev).clone()
        r_out = br if in_place else torch.empty_like(br)
        n_out = torch.empty_like(br)
        moe.layer_gated(shape, 2, logits, hidden, w, br, inject, norm_w, 1e-6, r_out, n_out, ids, wts, ws)
        torch.cuda.synchronize()
        outs.append((r_out.clone(), n_out.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_gated_rejects_bad_arguments(moe):
    cfg = mi.CONFIGS["tiny"]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    t = torch.zeros((9, cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((cfg.T, 9), device="cuda")
    for G, eps in ((0, 1e-6), (9, 1e-6), (2, -1.0)):
        with pytest.raises(moe.MoeError):
            moe.forward_unroute_gated(shape, G, t, a, t[0], eps, t, t, ws)
