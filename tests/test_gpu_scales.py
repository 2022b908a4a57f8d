"""Tensor scales and block scales of the NVFP4 weights, pinned on the GPU against the oracle.

The workloads run every weight tensor at tensor scale 1.0 and block scales in the narrow
E4M3 range 0x18..0x28, which would let a kernel that dropped or doubled a tensor-scale
multiply, or decoded a block scale outside that range wrongly, pass its parity tests.
Here every expert kernel (and both un-route forms: fused into the decode kernel for a
few tokens, a kernel of its own otherwise) runs against the CPU oracle with:
  - non-unit tensor scales, powers of two and not (the FP32 tensor scale of each weight
    tensor, "one FP32 tensor scale" of the NVFP4 format on the page "How I forked vLLM and
    made Qwen3.8-Flash-Next decode 1.6x faster on one GPU", section "The model and the
    constraint");
  - block scales taken from one band of 16 E4M3 codes at a time, with random signs, so that
    the zero code, every subnormal, every normal exponent up to 448 and the negative codes
    each decide some outputs (the tensor scales bring every band to the same magnitude, so
    the bands' exact results are identical up to the powers of two);
  - block scales spread over every finite E4M3 code at once.
Intermediates that leave the FP16 store range must set the documented status bits.

The output is compared with max |d_i| <= 2e-2 RMS(ref) + 2^-8 |ref_i| (the output's own
BF16 rounding allowed on top of the layer's tolerance: these cases reach |out| ~ 6 RMS,
where BF16 rounding alone can exceed 2e-2 RMS) and sum |d| / sum |ref| <= 5e-3.
"""
import numpy as np
import pytest

import moe_inputs as mi
from gpu_helpers import assert_parity, run_layer
from oracle import oracle as O

pytestmark = pytest.mark.gpu

AUTO, TCGEN05, SIMT, MMA, WIDE = 0, 1, 2, 3, 4

# (T, d, ffn, E, k): a decode-kernel shape with the un-route fused (T <= 8), one with the
# separate un-route kernel and experts of one and two 8-row tiles, and a many-row shape
# that MOE_ALGO_AUTO runs on the wide tcgen05 kernel (64 routed rows per expert)
SHAPES = {
    "dec4": ((4, 256, 256, 16, 2), (AUTO, TCGEN05, SIMT, WIDE)),
    "dec40": ((40, 512, 256, 32, 4), (AUTO, TCGEN05)),
    "many512": ((512, 256, 256, 16, 2), (AUTO, MMA)),
}


def _band_ts(band):
    # the E4M3 exponent field of band b is 2b or 2b + 1: 2^(3 - 2b) brings it back to the
    # workloads' magnitude; 0.75 and 1.3 keep the tensor scales off powers of two
    return 0.75 * 2.0 ** (3 - 2 * band), 1.3 * 2.0 ** (3 - 2 * band)


SCALE_CASES = ([(f"band{b}",) + _band_ts(b) for b in range(8)]
               + [("default", 0.375, 2.5), ("default", 0.7071, 1.3),
                  ("all_finite", 0.75 * 2.0 ** -11, 1.3 * 2.0 ** -11)])


def _inputs(shape_name, scales, ts13, ts2, seed=11):
    T, d, F, E, k = SHAPES[shape_name][0]
    cfg = mi.CONFIGS["tiny"].replace(name=f"scales_{shape_name}", T=T, d=d, ffn=F, E=E, k=k, tag=600 + T)
    inp = mi.gen_layer(cfg, seed=seed, weights=False)
    inp.update(mi.gen_weights(cfg, seed=seed, scales=scales, w13_ts=ts13, w2_ts=ts2))
    return cfg, inp


def _parity(cfg, inp, algo, what):
    ids, wts, out, layer = run_layer(cfg, inp, algo=algo)
    status = layer.status()
    assert status == 0, f"{what}: device status {status:#x}"
    ids_ref, w_ref = O.route_topk(inp["logits"], cfg.k)
    np.testing.assert_array_equal(ids, ids_ref)
    ref = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids_ref, w_ref, inp, inp["residual"])
    # block scales from one band give heavier-tailed outputs than the workloads' (up to
    # ~6 RMS), so the output's own BF16 rounding is allowed on top of the tolerance
    return assert_parity(out, ref, what, bf16_rounding=True)


@pytest.mark.parametrize("scales,ts13,ts2", SCALE_CASES, ids=[f"{c[0]}-{c[1]:.4g}-{c[2]:.4g}" for c in SCALE_CASES])
@pytest.mark.parametrize("shape_name", sorted(SHAPES))
def test_scales_every_kernel(shape_name, scales, ts13, ts2):
    cfg, inp = _inputs(shape_name, scales, ts13, ts2)
    for algo in SHAPES[shape_name][1]:
        _parity(cfg, inp, algo, f"{shape_name} {scales} ts=({ts13:.4g}, {ts2:.4g}) algo {algo}")


def test_dropped_tensor_scale_would_fail():
    # the bar these cases set: the oracle with the down tensor scale dropped (or the gate/up
    # one doubled) is far outside the tolerance of the correct result
    cfg, inp = _inputs("dec4", "default", 0.375, 2.5)
    ids, w = O.route_topk(inp["logits"], cfg.k)
    dims = (cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ref = O.moe_experts(dims, inp["hidden"], ids, w, inp, inp["residual"]).astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    for bad in (dict(inp, w2_ts=1.0), dict(inp, w13_ts=0.75)):
        got = O.moe_experts(dims, inp["hidden"], ids, w, bad, inp["residual"])
        assert np.abs(got - ref).max() > 10 * 2e-2 * rms


@pytest.mark.parametrize("band", [0, 7])
def test_scale_bands_full_decode_size(band):
    # B=1 verify shape (T=4, d=2048, ffn=512, E=512, top-10) through the one-call layer
    ts13, ts2 = _band_ts(band)
    base = mi.CONFIGS["b1"]
    cfg = base.replace(name=f"b1_band{band}", tag=620 + band)
    inp = mi.gen_layer(cfg, seed=0, weights=False)
    inp.update(mi.gen_weights(cfg, seed=0, scales=f"band{band}", w13_ts=ts13, w2_ts=ts2))
    _parity(cfg, inp, AUTO, f"b1 band{band}")


def _status_of(cfg, inp, algo):
    _, _, out, layer = run_layer(cfg, inp, algo=algo)
    assert np.all(np.isfinite(out))
    return layer.status()


@pytest.mark.parametrize("shape_name,algo", [("dec4", AUTO), ("dec4", TCGEN05), ("dec4", SIMT), ("dec4", WIDE),
                                             ("dec40", AUTO), ("many512", AUTO)])
def test_h_past_fp16_store_range_sets_status(shape_name, algo):
    # band-7 gate/up scales (up to 448) at tensor scale 1: |silu(g) u| far above 2^4 * 65504
    import routed_moe_decode_gb300 as moe
    cfg, inp = _inputs(shape_name, "band7", 1.0, 2.0 ** -20)
    st = _status_of(cfg, inp, algo)
    assert st & moe.MOE_DEV_H_SATURATED, f"status {st:#x}"


@pytest.mark.parametrize("shape_name,algo", [("many512", AUTO), ("dec4", WIDE)])
def test_wide_kernel_y_past_fp16_store_range_sets_status(shape_name, algo):
    # per-route down outputs of the wide kernel are stored as FP16(y / 16): a down tensor
    # scale of 2^14 puts |y| near 10^7; h stays in range
    import routed_moe_decode_gb300 as moe
    ts13, ts2 = _band_ts(3)
    cfg, inp = _inputs(shape_name, "band3", ts13, ts2 * 2.0 ** 14)
    st = _status_of(cfg, inp, algo)
    assert st & moe.MOE_DEV_Y_SATURATED and not st & moe.MOE_DEV_H_SATURATED, f"status {st:#x}"


@pytest.mark.parametrize("algo", [AUTO, TCGEN05])
def test_decode_kernels_keep_large_y_exact(algo):
    # the decode kernels keep per-route outputs in FP32: the same large-y case is in range
    ts13, ts2 = _band_ts(3)
    cfg, inp = _inputs("dec4", "band3", ts13, ts2 * 2.0 ** 14)
    _parity(cfg, inp, algo, "dec4 large y")


@pytest.mark.parametrize("T,d,F,E,k", [(4, 256, 256, 16, 2), (40, 512, 256, 32, 4), (8, 384, 256, 16, 2),
                                       (512, 256, 256, 16, 2), (4, 2048, 512, 512, 10)])
def test_per_expert_tensor_scales(T, d, F, E, k):
    # moe_layer_expert_scales through MOE_ALGO_AUTO, which picks the decode kernel for <= 8 tokens,
    # the warp-MMA kernel, the 16-row tcgen05 kernel (d = 384) and the wide kernel (64 rows/expert)
    import routed_moe_decode_gb300 as moe
    import torch
    from gpu_helpers import bf16_tensor, device_weights
    cfg = mi.CONFIGS["tiny"].replace(name=f"ts_e{T}x{d}", T=T, d=d, ffn=F, E=E, k=k, tag=640 + T)
    inp = mi.gen_layer(cfg, seed=12)
    t13, t2 = mi.gen_expert_tensor_scales(cfg, seed=12)
    dev = "cuda"
    shape = moe.shape_of(T, d, F, E, k)
    ws = moe.Workspace(shape)
    w = device_weights(inp, dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    moe.layer_expert_scales(shape, torch.from_numpy(inp["logits"]).to(dev), bf16_tensor(inp["hidden"], dev), w,
                            torch.from_numpy(t13).to(dev), torch.from_numpy(t2).to(dev),
                            bf16_tensor(inp["residual"], dev), out, ids, wts, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    ids_ref, w_ref = O.route_topk(inp["logits"], k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    ref = O.moe_experts_ts((T, d, F, E, k), inp["hidden"], ids_ref, w_ref, inp, t13, t2, inp["residual"])
    assert_parity(out.float().cpu().numpy(), ref, f"per-expert scales T={T} d={d}", bf16_rounding=True)
