"""Pins of the oracle's functions for the rows next to the layer: BF16 rounding, the router
projection, the gated residual update with its normalisation, and per-expert tensor scales.

Each function is checked against something other than itself: hand-worked bit patterns,
a library routine in float64, closed forms and invariants that a dropped term, a wrong sign
or factor or a misplaced index would break."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from conftest import read_golden
from oracle import oracle as O


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _f(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- BF16 rounding
def test_bf16_rounding_golden():
    for fbits, bbits, *_ in read_golden("bf16_rounding.txt"):
        x = np.array([int(fbits, 16)], dtype=np.uint32).view(np.float32)
        assert O.bf16_round(x)[0] == int(bbits, 16), fbits


def test_bf16_rounding_matches_torch_on_random_patterns():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    np.testing.assert_array_equal(O.bf16_round(x), _bf16(x))


# ---------------------------------------------------------------- router projection
def _router_case(T, d, E, seed):
    rng = np.random.default_rng(seed)
    hidden = _bf16(rng.standard_normal((T, d)))
    wr = _bf16(rng.standard_normal((E, d)) * 0.05)
    return hidden, wr


def test_router_logits_against_float64_matmul():
    hidden, wr = _router_case(5, 384, 40, 2)
    ref = _f(hidden).astype(np.float64) @ _f(wr).astype(np.float64).T
    got = O.router_logits(hidden, wr)
    bound = 384 * 2.0 ** -24 * (np.abs(_f(hidden)).astype(np.float64) @ np.abs(_f(wr)).astype(np.float64).T)
    assert np.all(np.abs(got - ref) <= bound)
    np.testing.assert_allclose(O.router_logits(hidden, wr, "f64"), ref, rtol=1e-12, atol=1e-12)


def test_router_logits_one_hot_hidden_selects_a_weight_column():
    _, wr = _router_case(1, 256, 17, 3)
    hidden = np.zeros((3, 256), np.uint16)
    for t, c in enumerate((0, 100, 255)):
        hidden[t, c] = 0x3F80  # 1.0
    got = O.router_logits(hidden, wr)
    for t, c in enumerate((0, 100, 255)):
        np.testing.assert_array_equal(got[t], _f(wr[:, c]))


# ---------------------------------------------------------------- gated residual + GemmaRMSNorm
def _norm_case(T, d, G, seed, w_scale=0.2):
    rng = np.random.default_rng(seed)
    moe_out = (rng.standard_normal((T, d)) * 3).astype(np.float32)
    resid = _bf16(rng.standard_normal((G, T, d)))
    a = rng.standard_normal((T, G)).astype(np.float32)
    w = _bf16(rng.standard_normal((G, d)) * w_scale)
    return moe_out, resid, a, w


def test_gated_norm_golden_worked_example():
    # d = 4, R = 1, O = 0, w = (0, 0.5, -0.5, 1): mean(R'^2) = 1, N = (1 + w) / sqrt(1 + 1e-6)
    resid = np.full((1, 1, 4), 0x3F80, np.uint16)
    w = _bf16(np.array([[0.0, 0.5, -0.5, 1.0]]))
    r, n = O.gated_residual_norm(np.zeros((1, 4), np.float32), resid, np.zeros((1, 1), np.float32), w, 1e-6)
    np.testing.assert_array_equal(r, resid)
    np.testing.assert_allclose(n[0, 0], np.array([1.0, 1.5, 0.5, 2.0]) / np.sqrt(1.000001), rtol=1e-7)


def test_gated_norm_zero_update_keeps_residual_and_reads_the_rounded_value():
    moe_out, resid, a, w = _norm_case(3, 256, 4, 4)
    r0, n0 = O.gated_residual_norm(np.zeros_like(moe_out), resid, a, w)
    np.testing.assert_array_equal(r0, resid)
    # the normalisation reads R' after its BF16 rounding: re-normalising the stored R' (with a
    # zero update) reproduces the first call's N bit for bit
    r1, n1 = O.gated_residual_norm(moe_out, resid, a, w)
    r2, n2 = O.gated_residual_norm(np.zeros_like(moe_out), r1, a, w)
    np.testing.assert_array_equal(r2, r1)
    np.testing.assert_array_equal(n2, n1)


def test_gated_norm_gate_is_twice_the_sigmoid():
    moe_out, resid, _, w = _norm_case(2, 128, 2, 5)
    T, G = 2, 2
    full = np.full((T, G), 40.0, np.float32)   # sigmoid = 1 in FP32: R' = BF16(R + 2 O)
    half = np.zeros((T, G), np.float32)        # sigmoid = 1/2:      R' = BF16(R + O)
    off = np.full((T, G), -40.0, np.float32)   # sigmoid ~ 4e-18:    R' = R
    rf, _ = O.gated_residual_norm(moe_out, resid, full, w)
    rh, _ = O.gated_residual_norm(moe_out, resid, half, w)
    ro, _ = O.gated_residual_norm(moe_out, resid, off, w)
    base = _f(resid)
    np.testing.assert_array_equal(rf, _bf16(base + 2 * moe_out[None]))
    np.testing.assert_array_equal(rh, _bf16(base + moe_out[None]))
    np.testing.assert_array_equal(ro, resid)


def test_gated_norm_weight_enters_as_one_plus_w():
    moe_out, resid, a, w = _norm_case(3, 256, 2, 6)
    _, n_w = O.gated_residual_norm(moe_out, resid, a, w)
    _, n_0 = O.gated_residual_norm(moe_out, resid, a, np.zeros_like(w))
    np.testing.assert_array_equal(n_w, n_0 * (np.float32(1) + _f(w))[:, None, :])


def test_gated_norm_unit_rms_and_scale_invariance():
    moe_out, resid, a, w = _norm_case(4, 512, 3, 7)
    zero_w = np.zeros_like(w)
    r, n = O.gated_residual_norm(moe_out, resid, a, zero_w, eps=1e-6)
    rms = np.sqrt(np.mean(n.astype(np.float64) ** 2, axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=2e-6)
    # scaling R and O by 4 scales R' exactly (BF16 rounding commutes with powers of two) and
    # leaves N unchanged up to the eps term
    r4, n4 = O.gated_residual_norm(moe_out * 4, _bf16(_f(resid) * 4), a, zero_w, eps=1e-6)
    np.testing.assert_array_equal(_f(r4), _f(r) * 4)
    np.testing.assert_allclose(n4, n, rtol=1e-5, atol=1e-6)


def test_gated_norm_branches_are_independent():
    moe_out, resid, a, w = _norm_case(2, 128, 4, 8)
    r, n = O.gated_residual_norm(moe_out, resid, a, w)
    perm = [2, 0, 3, 1]
    rp, np_ = O.gated_residual_norm(moe_out, resid[perm], a[:, perm], w[perm])
    np.testing.assert_array_equal(rp, r[perm])
    np.testing.assert_array_equal(np_, n[perm])


def test_gated_norm_fp32_against_fp64_shadow():
    moe_out, resid, a, w = _norm_case(3, 1024, 4, 9)
    r32, n32 = O.gated_residual_norm(moe_out, resid, a, w, precision="f32")
    r64, n64 = O.gated_residual_norm(moe_out.astype(np.float64), resid, a, w, precision="f64")
    # the stored residual may differ by one BF16 step where the FP32 and FP64 sums straddle
    # a rounding boundary; the normalised values agree to FP32 rounding
    assert np.mean(r32 != r64) < 1e-3
    np.testing.assert_allclose(n32, n64, rtol=1e-4, atol=1e-4)


# ---------------------------------------------------------------- per-expert tensor scales
def test_per_expert_tensor_scales_follow_the_expert():
    # top-1 routing: each token's output is one expert's FFN, so with per-expert scales it must
    # equal the one-scale oracle run at that expert's scales, token by token
    cfg = mi.CONFIGS["tiny"].replace(name="ts_e", T=12, k=1, tag=700)
    inp = mi.gen_layer(cfg, seed=3)
    ids, wts = O.route_topk(inp["logits"], 1)
    rng = np.random.default_rng(3)
    t13 = (2.0 ** rng.integers(-3, 3, cfg.E) * rng.choice([0.75, 1.0, 1.3], cfg.E)).astype(np.float32)
    t2 = (2.0 ** rng.integers(-3, 3, cfg.E) * rng.choice([0.5, 1.0, 2.5], cfg.E)).astype(np.float32)
    dims = (cfg.T, cfg.d, cfg.ffn, cfg.E, 1)
    got = O.moe_experts_ts(dims, inp["hidden"], ids, wts, inp, t13, t2, inp["residual"])
    for t in range(cfg.T):
        e = ids[t, 0]
        one = dict(inp, w13_ts=float(t13[e]), w2_ts=float(t2[e]))
        ref = O.moe_experts(dims, inp["hidden"], ids, wts, one, inp["residual"])
        np.testing.assert_array_equal(got[t], ref[t])
    # all scales equal: the per-expert form is the one-scale form
    same = O.moe_experts_ts(dims, inp["hidden"], ids, wts, inp, np.full(cfg.E, 0.75, np.float32),
                            np.full(cfg.E, 2.5, np.float32), inp["residual"])
    np.testing.assert_array_equal(same, O.moe_experts(dims, inp["hidden"], ids, wts,
                                                      dict(inp, w13_ts=0.75, w2_ts=2.5), inp["residual"]))
