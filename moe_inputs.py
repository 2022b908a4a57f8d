"""Seeded synthetic inputs for the routed MoE layer (tests, smoke run and bench).

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no softmax, no top-k, no dequantisation, no FFN).  The CUDA
path and the CPU oracle both consume what it produces and share nothing else.

Workloads (one per named configuration; sizes from the routed-MoE decode/prefill
setting of Qwen3.8-Flash-Next: 512 experts, top-10, NVFP4 experts, verify steps of
k+1 = 4 rows per request, 8192-token prefill chunks):

  tiny     T=4    d=256  ffn=128 E=16  k=2   logits ~N(0,1)
  b1       T=4    d=2048 ffn=512 E=512 k=10  logits ~N(0,1)               (1 request x 4 rows)
  b8       T=32   d=2048 ffn=512 E=512 k=10  logits ~N(0,1) + per-request bias ~N(0, std 2)
                                             on 40 experts drawn without replacement
  b64      T=256  d=2048 ffn=512 E=512 k=10  logits ~N(0,1) + c*ln(Zipf pmf, s=1.1) over a
                                             random rank permutation of the experts
  prefill  T=8192 d=2048 ffn=512 E=512 k=10  logits ~N(0,1)

Hidden and residual are BF16 rounded (round-to-nearest-even) from N(0,1).  NVFP4
weights: every E2M1 nibble uniform over its 16 codes (so every code byte uniform over
256 values), every E4M3 block scale the round-to-nearest-even E4M3 value of
U[0.5, 2] * 2^-3, FP32 tensor scales 1.0.  Each tensor has its own counter-based
stream keyed by (seed, config, layer, tensor), so any layer can be regenerated alone.

Layouts (row-major, C order):
  logits     float32 [T, E]
  hidden     uint16  [T, d]      BF16 bit patterns
  residual   uint16  [T, d]      BF16 bit patterns
  w13_codes  uint8   [E, 2*ffn, d/2]   element 2i in the low nibble of byte i
  w13_scales uint8   [E, 2*ffn, d/16]  E4M3 codes, one per 16 consecutive K elements
  w2_codes   uint8   [E, d, ffn/2]
  w2_scales  uint8   [E, d, ffn/16]
Rows 0..ffn-1 of w13 are the gate projection, rows ffn..2*ffn-1 the up projection.
"""
from __future__ import annotations

import dataclasses
import numpy as np

try:  # torch is used only for its BF16 / E4M3 rounding of drawn values
    import torch
except ImportError:  # pragma: no cover - torch is present in every supported image
    torch = None

__all__ = ["Config", "CONFIGS", "ZIPF_COEF_CALIBRATED", "ZIPF_COEF_LITERAL", "E4M3_FINITE_CODES",
           "gen_logits", "gen_hidden", "gen_residual", "gen_weights", "gen_layer", "gen_router_weight",
           "gen_gated_inputs", "gen_expert_tensor_scales",
           "weight_bytes_per_expert"]

# Zipf popularity bias for the T=256 decode batch.  The literal coefficient (1.5 on the
# natural log of the pmf) concentrates ~all rows on a few dozen experts; the stated
# outcome ("hot experts up to ~60 rows, tail 0-2") is reached with 0.25 (i.e. a
# -0.275*ln(rank) bias).  The calibrated value is the default; the literal one is kept
# as an extra parity workload.
ZIPF_COEF_CALIBRATED = 0.25
ZIPF_COEF_LITERAL = 1.5

_TENSOR_TAGS = {"logits": 1, "hidden": 2, "residual": 3, "w13_codes": 4, "w13_scales": 5,
                "w2_codes": 6, "w2_scales": 7, "bias_pick": 8, "bias_val": 9, "zipf_perm": 10,
                "router_w": 11, "branches": 12, "inject": 13, "norm_w": 14, "ts_e": 15}


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    d: int
    ffn: int
    E: int
    k: int
    logits: str = "normal"          # normal | request_bias | zipf
    rows_per_request: int = 4
    bias_experts: int = 40
    bias_std: float = 2.0
    zipf_s: float = 1.1
    zipf_coef: float = ZIPF_COEF_CALIBRATED
    layers: int = 12
    tag: int = 0

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": Config("tiny", T=4, d=256, ffn=128, E=16, k=2, layers=1, tag=0),
    "b1": Config("b1", T=4, d=2048, ffn=512, E=512, k=10, tag=1),
    "b8": Config("b8", T=32, d=2048, ffn=512, E=512, k=10, logits="request_bias", tag=2),
    "b64": Config("b64", T=256, d=2048, ffn=512, E=512, k=10, logits="zipf", tag=3),
    "prefill": Config("prefill", T=8192, d=2048, ffn=512, E=512, k=10, tag=4),
    "b64_literal": Config("b64_literal", T=256, d=2048, ffn=512, E=512, k=10, logits="zipf",
                          zipf_coef=ZIPF_COEF_LITERAL, layers=1, tag=5),
}


def weight_bytes_per_expert(cfg: Config) -> int:
    """NVFP4 bytes of one expert: codes (half a byte per weight) plus one scale byte per 16."""
    n13 = 2 * cfg.ffn * cfg.d
    n2 = cfg.d * cfg.ffn
    return (n13 + n2) // 2 + (n13 + n2) // 16


def _rng(seed: int, cfg: Config, layer: int, tensor: str) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), int(cfg.tag), int(layer), _TENSOR_TAGS[tensor]])
    return np.random.Generator(np.random.PCG64(ss))


def _raw_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    words = rng.bit_generator.random_raw((n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def gen_logits(cfg: Config, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Router logits float32 [T, E] with the configuration's routing structure."""
    rng = _rng(seed, cfg, layer, "logits")
    logits = rng.standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if cfg.logits == "request_bias":
        pick = _rng(seed, cfg, layer, "bias_pick")
        val = _rng(seed, cfg, layer, "bias_val")
        nreq = (cfg.T + cfg.rows_per_request - 1) // cfg.rows_per_request
        for r in range(nreq):
            experts = pick.choice(cfg.E, size=min(cfg.bias_experts, cfg.E), replace=False)
            bias = (val.standard_normal(experts.size) * cfg.bias_std).astype(np.float32)
            rows = slice(r * cfg.rows_per_request, min(cfg.T, (r + 1) * cfg.rows_per_request))
            logits[rows, experts] += bias[None, :]
    elif cfg.logits == "zipf":
        perm = _rng(seed, cfg, layer, "zipf_perm")
        rank = perm.permutation(cfg.E).astype(np.float64) + 1.0
        harmonic = np.sum(np.arange(1, cfg.E + 1, dtype=np.float64) ** (-cfg.zipf_s))
        ln_pmf = -cfg.zipf_s * np.log(rank) - np.log(harmonic)
        logits += (cfg.zipf_coef * ln_pmf).astype(np.float32)[None, :]
    elif cfg.logits != "normal":
        raise ValueError(f"unknown logits kind {cfg.logits!r}")
    return np.ascontiguousarray(logits, dtype=np.float32)


def gen_hidden(cfg: Config, seed: int = 0, layer: int = 0) -> np.ndarray:
    """BF16 hidden states as uint16 bit patterns [T, d], values N(0,1) rounded RNE."""
    rng = _rng(seed, cfg, layer, "hidden")
    return _to_bf16_bits(rng.standard_normal((cfg.T, cfg.d), dtype=np.float32))


def gen_residual(cfg: Config, seed: int = 0, layer: int = 0) -> np.ndarray:
    """BF16 residual as uint16 bit patterns [T, d], values N(0,1) rounded RNE."""
    rng = _rng(seed, cfg, layer, "residual")
    return _to_bf16_bits(rng.standard_normal((cfg.T, cfg.d), dtype=np.float32))


def _gen_scales(rng: np.random.Generator, n: int) -> np.ndarray:
    u = rng.random(n, dtype=np.float32)
    return _to_e4m3_codes((u * np.float32(1.5) + np.float32(0.5)) * np.float32(0.125))


# E4M3 codes that are not NaN (S.1111.111 is the format's only NaN; there is no infinity).
E4M3_FINITE_CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _gen_band_codes(rng: np.random.Generator, n: int, band: int) -> np.ndarray:
    """E4M3 codes drawn uniformly from the 16 magnitudes 16*band .. 16*band + 15 (the
    exponent fields 2*band and 2*band + 1; band 0 holds zero and the subnormals, band 7
    the largest values up to 448; the NaN code is left out) with a uniform sign bit."""
    if not 0 <= band <= 7:
        raise ValueError("band must be in 0..7")
    mags = np.arange(16 * band, 16 * band + 16, dtype=np.uint8)
    mags = mags[mags != 0x7F]
    codes = mags[rng.integers(0, mags.size, size=n)]
    return codes | (rng.integers(0, 2, size=n, dtype=np.uint8) << 7)


def _gen_scale_codes(rng: np.random.Generator, n: int, scales: str) -> np.ndarray:
    if scales == "default":
        return _gen_scales(rng, n)
    if scales == "all_finite":  # every finite code, both signs, uniformly
        return E4M3_FINITE_CODES[rng.integers(0, E4M3_FINITE_CODES.size, size=n)]
    if scales.startswith("band"):
        return _gen_band_codes(rng, n, int(scales[4:]))
    raise ValueError(f"unknown block-scale distribution {scales!r}")


def gen_weights(cfg: Config, seed: int = 0, layer: int = 0, scales: str = "default",
                w13_ts: float = 1.0, w2_ts: float = 1.0) -> dict:
    """NVFP4 expert weights of one layer (see the module docstring for layouts).

    `scales` picks the E4M3 block-scale distribution: "default" (the workloads'
    E4M3(U[0.5, 2] * 2^-3)), "band0" .. "band7" (one band of 16 codes, see
    _gen_band_codes, random signs) or "all_finite" (every non-NaN code).  The FP32
    tensor scales are passed through as given (the workloads use 1.0)."""
    E, F, d = cfg.E, cfg.ffn, cfg.d
    if d % 16 or F % 16:
        raise ValueError("d and ffn must be multiples of 16 for NVFP4 blocks")
    w13_codes = _raw_bytes(_rng(seed, cfg, layer, "w13_codes"), E * 2 * F * d // 2)
    w13_scales = _gen_scale_codes(_rng(seed, cfg, layer, "w13_scales"), E * 2 * F * d // 16, scales)
    w2_codes = _raw_bytes(_rng(seed, cfg, layer, "w2_codes"), E * d * F // 2)
    w2_scales = _gen_scale_codes(_rng(seed, cfg, layer, "w2_scales"), E * d * F // 16, scales)
    return {
        "w13_codes": w13_codes.reshape(E, 2 * F, d // 2),
        "w13_scales": w13_scales.reshape(E, 2 * F, d // 16),
        "w13_ts": float(w13_ts),
        "w2_codes": w2_codes.reshape(E, d, F // 2),
        "w2_scales": w2_scales.reshape(E, d, F // 16),
        "w2_ts": float(w2_ts),
    }


def gen_router_weight(cfg: Config, seed: int = 0, layer: int = 0) -> np.ndarray:
    """BF16 router weight [E, d] (uint16 bits), values N(0, 1/d) rounded RNE, so that the
    projected logits of N(0,1) hidden rows are about N(0,1) like the workloads' logits."""
    rng = _rng(seed, cfg, layer, "router_w")
    return _to_bf16_bits(rng.standard_normal((cfg.E, cfg.d), dtype=np.float32) / np.float32(np.sqrt(cfg.d)))


def gen_gated_inputs(cfg: Config, G: int, seed: int = 0, layer: int = 0) -> dict:
    """Inputs of the gated residual update for G residual branches: the branches [G, T, d]
    (BF16 bits, N(0,1)), the injection logits [T, G] (float32, N(0,1)) and the consuming
    normalisation's weight [G, d] (BF16 bits, N(0, 0.1^2): GemmaRMSNorm scales by 1 + w)."""
    return {
        "branches": _to_bf16_bits(_rng(seed, cfg, layer, "branches").standard_normal((G, cfg.T, cfg.d),
                                                                                  dtype=np.float32)),
        "inject": _rng(seed, cfg, layer, "inject").standard_normal((cfg.T, G), dtype=np.float32),
        "norm_w": _to_bf16_bits(_rng(seed, cfg, layer, "norm_w").standard_normal((G, cfg.d), dtype=np.float32)
                                * np.float32(0.1)),
    }


def gen_expert_tensor_scales(cfg: Config, seed: int = 0, layer: int = 0) -> tuple:
    """Per-expert FP32 tensor scales (w13 [E], w2 [E]): powers of two from 2^-2 to 2^2 times
    one of (0.75, 1, 1.3), drawn independently per expert and tensor."""
    rng = _rng(seed, cfg, layer, "ts_e")
    t13 = (np.float32(2.0) ** rng.integers(-2, 3, cfg.E).astype(np.float32)) * \
        rng.choice(np.array([0.75, 1.0, 1.3], np.float32), cfg.E)
    t2 = (np.float32(2.0) ** rng.integers(-2, 3, cfg.E).astype(np.float32)) * \
        rng.choice(np.array([0.75, 1.0, 1.3], np.float32), cfg.E)
    return t13.astype(np.float32), t2.astype(np.float32)


def gen_layer(cfg: Config, seed: int = 0, layer: int = 0, weights: bool = True) -> dict:
    """All inputs of one layer call: logits, hidden, residual (and weights if asked)."""
    out = {"logits": gen_logits(cfg, seed, layer),
           "hidden": gen_hidden(cfg, seed, layer),
           "residual": gen_residual(cfg, seed, layer)}
    if weights:
        out.update(gen_weights(cfg, seed, layer))
    return out
