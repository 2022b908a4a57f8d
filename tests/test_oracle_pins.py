"""Pins for the CPU oracle: checks against facts fixed outside the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a wrong exponent bias, a
swapped nibble, gate/up swapped, a transposed weight, a dropped residual, a wrong tie
rule) fails at least one of them:
  * hand-worked E2M1 / E4M3 decode tables (tests/golden), and the E4M3 table against
    torch's independent float8_e4m3fn conversion;
  * brute-force routing by a full stable sort on small and tie-heavy inputs;
  * the FFN against a float64 numpy matmul over weights dequantised through the golden
    tables (a different code path end to end);
  * closed forms (all weights one), special cases (zero hidden, k=1, constant logits),
    invariants (linearity in the down tensor scale, expert relabelling, batch
    independence, all-equal experts make routing irrelevant);
  * the FP32 oracle against its FP64 shadow.
"""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import oracle as O
from conftest import read_golden


def _golden_e2m1():
    return {int(c, 16): float(v) for c, v in read_golden("e2m1_values.txt")}


def _golden_e4m3():
    return {int(c, 16): float(v) for c, v in read_golden("e4m3_values.txt")}


def test_e2m1_table_matches_hand_worked_values():
    table = _golden_e2m1()
    assert len(table) == 16
    for code, val in table.items():
        got = O.e2m1_value(code)
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), (code, got, val)


def test_e4m3_hand_worked_values():
    for code, val in _golden_e4m3().items():
        got = O.e4m3_value(code)
        if math.isnan(val):
            assert math.isnan(got), code
        else:
            assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), (code, got, val)


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for b in range(256):
        got = O.e4m3_value(b)
        if np.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b], (b, got, ref[b])


def test_dequant_row_nibble_order_and_block_scales():
    # byte i holds element 2i in its low nibble: 0x21 -> [0.5, 1.0]; 0xF7 -> [6.0, -6.0]
    codes = np.array([0x21, 0xF7] + [0x00] * 6 + [0x22] * 8, dtype=np.uint8)  # K = 32
    scales = np.array([0x38, 0x40], dtype=np.uint8)  # block 0 scale 1.0, block 1 scale 2.0
    out = O.dequant_row(codes, scales, 0.5, 32)
    expect = np.zeros(32, dtype=np.float32)
    expect[:4] = [0.5, 1.0, 6.0, -6.0]
    expect[:16] *= 1.0 * 0.5
    expect[16:] = 1.0 * 2.0 * 0.5
    np.testing.assert_array_equal(out, expect)


def _brute_route(logits, k):
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    for t in range(T):
        row = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-row[e], e))  # larger first, ties -> lower id
        ids[t] = order[:k]
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        p /= p.sum()
        sel = p[ids[t]]
        w[t] = sel / sel.sum()
    return ids, w


@pytest.mark.parametrize("T,E,k,kind", [(4, 16, 2, "normal"), (7, 64, 8, "ties"), (3, 512, 10, "normal"),
                                        (5, 512, 10, "ties"), (6, 33, 33, "normal"), (9, 40, 1, "ties")])
def test_route_matches_brute_force(T, E, k, kind):
    rng = np.random.default_rng(1234 + T * E + k)
    if kind == "ties":
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32) * np.float32(0.5)
    else:
        logits = rng.standard_normal((T, E), dtype=np.float32)
    ids_ref, w_ref = _brute_route(logits, k)
    ids32, w32 = O.route_topk(logits, k, "f32")
    ids64, w64 = O.route_topk(logits, k, "f64")
    np.testing.assert_array_equal(ids32, ids_ref)
    np.testing.assert_array_equal(ids64, ids_ref)
    np.testing.assert_allclose(w64, w_ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(w32, w_ref, rtol=2e-6, atol=1e-7)


def test_route_special_cases():
    # constant logits: ids 0..k-1, equal weights
    ids, w = O.route_topk(np.zeros((2, 16), np.float32), 4)
    np.testing.assert_array_equal(ids, np.tile(np.arange(4, dtype=np.int32), (2, 1)))
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=1e-7)
    # k = 1 gives weight exactly one
    rng = np.random.default_rng(5)
    ids, w = O.route_topk(rng.standard_normal((8, 64), dtype=np.float32), 1)
    assert np.all(w == 1.0)
    # -0 and +0 are equal: the lower index wins
    l = np.full((1, 8), -1.0, np.float32)
    l[0, 5] = 0.0
    l[0, 2] = -0.0
    ids, _ = O.route_topk(l, 2)
    np.testing.assert_array_equal(ids[0], [2, 5])
    # weights sum to one, descending with the logits
    logits = rng.standard_normal((16, 512), dtype=np.float32)
    ids, w = O.route_topk(logits, 10)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert all(len(set(r)) == 10 for r in ids)


def test_plan_matches_counting():
    rng = np.random.default_rng(7)
    ids = rng.integers(0, 64, size=(37, 5)).astype(np.int32)
    counts, offsets, touched = O.plan(ids, 64)
    np.testing.assert_array_equal(counts, np.bincount(ids.ravel(), minlength=64))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(touched, np.nonzero(counts)[0])
    with pytest.raises(ValueError):
        O.plan(np.array([[64]], np.int32), 64)


def _np_dequant(codes, scales, ts):
    """Float64 dequantisation through the golden E2M1 table and torch's E4M3 decode."""
    e2m1 = np.array([_golden_e2m1()[i] for i in range(16)], np.float64)
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return e2m1[nib] * np.repeat(s, 16, axis=-1) * ts


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _np_layer(cfg, inp, ids, w):
    W13 = _np_dequant(inp["w13_codes"], inp["w13_scales"], inp["w13_ts"])
    W2 = _np_dequant(inp["w2_codes"], inp["w2_scales"], inp["w2_ts"])
    x = _bf16_to_f64(inp["hidden"])
    res = _bf16_to_f64(inp["residual"])
    out = res.copy()
    F = cfg.ffn
    for t in range(cfg.T):
        acc = np.zeros(cfg.d)
        for j in range(cfg.k):
            e = ids[t, j]
            g = W13[e, :F] @ x[t]
            u = W13[e, F:] @ x[t]
            h = g / (1.0 + np.exp(-g)) * u
            acc += w[t, j] * (W2[e] @ h)
        out[t] += acc
    return out


def _rms(a):
    return float(np.sqrt(np.mean(np.square(a, dtype=np.float64))))


def test_experts_match_numpy_matmul_tiny():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=0)
    ids, w64 = O.route_topk(inp["logits"], cfg.k, "f64")
    ref = _np_layer(cfg, inp, ids, w64)
    out64 = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids, w64, inp,
                          inp["residual"], precision="f64")
    assert np.max(np.abs(out64 - ref)) <= 1e-10 * _rms(ref)
    ids32, w32, out32 = O.moe_layer(cfg, inp)
    np.testing.assert_array_equal(ids32, ids)
    assert np.max(np.abs(out32 - ref)) <= 1e-5 * _rms(ref)


def test_experts_closed_form_all_ones():
    # all codes 0x22 (both nibbles = 1.0), all scales 0x38 (1.0): g = u = sum(x),
    # h = silu(S) * S, y_r = F * h, and out = residual + F * h because sum_j w_j = 1
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=3)
    for n in ("w13_codes", "w2_codes"):
        inp[n] = np.full_like(inp[n], 0x22)
    for n in ("w13_scales", "w2_scales"):
        inp[n] = np.full_like(inp[n], 0x38)
    ids, w, out = O.moe_layer(cfg, inp, precision="f64")
    x = _bf16_to_f64(inp["hidden"])
    S = x.sum(1)
    h = S / (1.0 + np.exp(-S)) * S
    expect = _bf16_to_f64(inp["residual"]) + (cfg.ffn * h)[:, None]
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-9)
    _, _, out32 = O.moe_layer(cfg, inp)
    np.testing.assert_allclose(out32, expect, rtol=1e-5, atol=1e-3)


def test_experts_zero_hidden_gives_residual_exactly():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=4)
    inp["hidden"] = np.zeros_like(inp["hidden"])
    _, _, out = O.moe_layer(cfg, inp)
    np.testing.assert_array_equal(out, _bf16_to_f64(inp["residual"]).astype(np.float32))


def test_experts_linear_in_down_tensor_scale():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=5)
    inp["residual"] = np.zeros_like(inp["residual"])
    _, _, a = O.moe_layer(cfg, inp)
    inp2 = dict(inp, w2_ts=2.0)
    _, _, b = O.moe_layer(cfg, inp2)
    np.testing.assert_array_equal(b, 2.0 * a)


def test_experts_invariant_under_expert_relabelling():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=6)
    perm = np.random.default_rng(0).permutation(cfg.E)  # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    inp2 = dict(inp)
    inp2["logits"] = np.ascontiguousarray(inp["logits"][:, inv])
    for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        inp2[n] = np.ascontiguousarray(inp[n][inv])
    ids, w, a = O.moe_layer(cfg, inp, precision="f64")
    ids2, w2, b = O.moe_layer(cfg, inp2, precision="f64")
    np.testing.assert_array_equal(ids2, perm[ids])
    # only the softmax denominator's summation order changes
    np.testing.assert_allclose(w2, w, rtol=1e-13)
    assert np.max(np.abs(a - b)) <= 1e-12 * _rms(a)


def test_experts_all_equal_experts_make_routing_irrelevant():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=8)
    for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        inp[n] = np.ascontiguousarray(np.broadcast_to(inp[n][:1], inp[n].shape))
    _, _, a = O.moe_layer(cfg, inp, precision="f64")
    inp2 = dict(inp, logits=np.ascontiguousarray(inp["logits"][::-1]))
    _, _, b = O.moe_layer(cfg, inp2, precision="f64")
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-9)


def test_experts_rows_are_independent_and_mask_selects_rows():
    cfg = mi.CONFIGS["tiny"]
    inp = mi.gen_layer(cfg, seed=9)
    _, _, full = O.moe_layer(cfg, inp)
    mask = np.array([0, 1, 0, 1], np.uint8)
    _, _, part = O.moe_layer(cfg, inp, token_mask=mask)
    np.testing.assert_array_equal(part[1], full[1])
    np.testing.assert_array_equal(part[3], full[3])
    assert np.all(np.isnan(part[0])) and np.all(np.isnan(part[2]))
    # changing token 0's hidden leaves token 1's output unchanged
    inp2 = dict(inp)
    inp2["hidden"] = inp["hidden"].copy()
    inp2["hidden"][0] ^= 0x0100
    _, _, b = O.moe_layer(cfg, inp2)
    np.testing.assert_array_equal(b[1:], full[1:])


@pytest.mark.parametrize("name,tokens", [("tiny", None), ("b1", [0, 3])])
def test_f32_oracle_within_shadow_bound(name, tokens):
    cfg = mi.CONFIGS[name]
    inp = mi.gen_layer(cfg, seed=0)
    mask = None
    if tokens is not None:
        mask = np.zeros(cfg.T, np.uint8)
        mask[tokens] = 1
    ids, w32, out32 = O.moe_layer(cfg, inp, token_mask=mask)
    ids64, w64, out64 = O.moe_layer(cfg, inp, token_mask=mask, precision="f64")
    np.testing.assert_array_equal(ids, ids64)
    rows = slice(None) if tokens is None else tokens
    ref = out64[rows]
    err = np.abs(out32[rows] - ref)
    # the FP32 oracle's own error is far below the parity tolerance (2e-2 RMS max, 5e-3 mean rel)
    assert err.max() <= 1e-5 * _rms(ref)
    assert err.sum() / np.abs(ref).sum() <= 1e-6
