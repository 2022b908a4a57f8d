"""Helpers of the GPU parity tests: upload seeded inputs, run the C-ABI path, compare."""
from __future__ import annotations

import functools
import json
import os

import numpy as np
import torch

import moe_inputs as mi

# Tolerance of the layer output against the FP32 oracle (max and mean relative error).
MAX_ABS_OVER_RMS = 2e-2
MEAN_REL = 5e-3
WEIGHT_RTOL = 2e-6


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def device_weights(inp: dict, dev) -> dict:
    w = {n: torch.from_numpy(np.ascontiguousarray(inp[n])).to(dev)
         for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")}
    w["w13_ts"], w["w2_ts"] = float(inp["w13_ts"]), float(inp["w2_ts"])
    return w


@functools.lru_cache(maxsize=8)
def config_inputs(name: str, seed: int = 0, layer: int = 0) -> dict:
    return mi.gen_layer(mi.CONFIGS[name], seed=seed, layer=layer)


def run_layer(cfg, inp: dict, algo=0, dev="cuda", residual=True, w=None):
    """Router + plan + experts through the C ABI.  Returns (ids, weights, out_f32, layer)."""
    import routed_moe_decode_gb300 as moe
    dev = torch.device(dev)
    if w is None:
        w = device_weights(inp, dev)
    layer = moe.MoeLayer(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k, device=dev, algo=algo)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(dev)
    hidden = bf16_tensor(inp["hidden"], dev)
    res = bf16_tensor(inp["residual"], dev) if residual else None
    out = layer(logits, hidden, w, res)
    torch.cuda.synchronize()
    return layer.ids.cpu().numpy(), layer.weights.cpu().numpy(), out.float().cpu().numpy(), layer


def parity_metrics(got: np.ndarray, ref: np.ndarray):
    ref = ref.astype(np.float64)
    err = np.abs(got.astype(np.float64) - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(err.max()) / rms, float(err.sum() / np.abs(ref).sum())


# The layer's output is BF16, whose own round-to-nearest error reaches 2^-8 of the value
# (half a unit in the last place at the bottom of a binade).  Where a case's outputs have a
# heavier tail than the workloads' (max |out| above ~5 RMS), that rounding alone can exceed
# 2e-2 RMS; such cases compare with the rounding allowed on top of the tolerance.
BF16_HALF_ULP_REL = 2.0 ** -8


def parity_metrics_bf16(got: np.ndarray, ref: np.ndarray):
    """max over elements of (|d| - 2^-8 |ref|) / RMS(ref): the error left after the output's
    own BF16 rounding is allowed for."""
    ref = ref.astype(np.float64)
    err = np.abs(got.astype(np.float64) - ref) - BF16_HALF_ULP_REL * np.abs(ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(err.max()) / rms


def assert_parity(got: np.ndarray, ref: np.ndarray, what="", bf16_rounding=False):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean_rel = parity_metrics(got, ref)
    if bf16_rounding:
        mx = parity_metrics_bf16(got, ref)
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "rows": int(got.shape[0]), "max_abs_over_rms": mx,
                                "mean_rel": mean_rel}) + "\n")
    assert mx <= MAX_ABS_OVER_RMS and mean_rel <= MEAN_REL, \
        f"{what}: max|d|/rms {mx:.3e} (<= {MAX_ABS_OVER_RMS}), mean rel {mean_rel:.3e} (<= {MEAN_REL})"
    return mx, mean_rel
