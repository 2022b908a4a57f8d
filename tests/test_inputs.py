"""The seeded workload generators: determinism and the stated workload structure."""
import numpy as np

import moe_inputs as mi


def test_generators_are_deterministic_and_layer_keyed():
    cfg = mi.CONFIGS["tiny"]
    a = mi.gen_layer(cfg, seed=0, layer=0)
    b = mi.gen_layer(cfg, seed=0, layer=0)
    c = mi.gen_layer(cfg, seed=0, layer=1)
    for key in ("logits", "hidden", "residual", "w13_codes", "w13_scales", "w2_codes", "w2_scales"):
        np.testing.assert_array_equal(a[key], b[key])
        assert not np.array_equal(a[key], c[key])


def test_weight_layouts_and_value_sets():
    cfg = mi.CONFIGS["tiny"]
    w = mi.gen_weights(cfg)
    assert w["w13_codes"].shape == (cfg.E, 2 * cfg.ffn, cfg.d // 2)
    assert w["w13_scales"].shape == (cfg.E, 2 * cfg.ffn, cfg.d // 16)
    assert w["w2_codes"].shape == (cfg.E, cfg.d, cfg.ffn // 2)
    assert w["w2_scales"].shape == (cfg.E, cfg.d, cfg.ffn // 16)
    # block scales: E4M3 codes of U[0.5, 2] * 2^-3 span 0x18 (0.0625) .. 0x28 (0.25)
    for s in (w["w13_scales"], w["w2_scales"]):
        assert s.min() >= 0x18 and s.max() <= 0x28
    # every nibble value occurs with roughly equal frequency
    nib = np.concatenate([w["w13_codes"].ravel() & 15, w["w13_codes"].ravel() >> 4])
    freq = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(freq - 1 / 16) < 0.01)
    assert mi.weight_bytes_per_expert(mi.CONFIGS["b1"]) == 1769472


def _route_counts(cfg, layer=0):
    l = mi.gen_logits(cfg, 0, layer)
    ids = np.argsort(-l, axis=1, kind="stable")[:, :cfg.k]
    return np.bincount(ids.ravel(), minlength=cfg.E)


def test_routing_structure_of_decode_workloads():
    b1 = _route_counts(mi.CONFIGS["b1"])
    assert 30 <= (b1 > 0).sum() <= 40
    b8 = _route_counts(mi.CONFIGS["b8"])
    assert 140 <= (b8 > 0).sum() <= 220 and b8.max() >= 4  # draft rows of a request share experts
    b64 = _route_counts(mi.CONFIGS["b64"])
    assert (b64 > 0).sum() >= 450 and 40 <= b64.max() <= 90  # hot experts ~60 rows, long tail
    lit = _route_counts(mi.CONFIGS["b64_literal"])
    assert (lit > 0).sum() <= 80 and lit.max() >= 200


def test_hidden_is_bf16_normal():
    cfg = mi.CONFIGS["b8"]
    h = mi.gen_hidden(cfg)
    x = (h.astype(np.uint32) << 16).view(np.float32)
    assert h.dtype == np.uint16 and h.shape == (cfg.T, cfg.d)
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
