"""moe_layer_static_workspace: the whole layer for callers that cannot allocate device
memory (e.g. code running under CUDA-graph capture or inside a framework that owns all
device memory).  Its scratch is the library's fixed device array instead of a caller
workspace; its results must match the ordinary entry point, moe_layer, call after call.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes when run alone in a fresh process."""
import ctypes

import pytest
import torch

import moe_inputs as mi
from gpu_helpers import assert_parity, bf16_tensor, device_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_moe_decode_gb300 as m
    return m


def _static_call(m, shape, logits, hidden, w, residual, out, ids, wts):
    lib = m.lib()
    return lib.moe_layer_static_workspace(
        ctypes.byref(shape), ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(hidden.data_ptr()),
        ctypes.c_void_p(w["w13_codes"].data_ptr()), ctypes.c_void_p(w["w13_scales"].data_ptr()),
        float(w["w13_ts"]), ctypes.c_void_p(w["w2_codes"].data_ptr()), ctypes.c_void_p(w["w2_scales"].data_ptr()),
        float(w["w2_ts"]), ctypes.c_void_p(residual.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(wts.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["b1", "b8"])
def test_static_workspace_matches_moe_layer_twice_in_a_row(moe, name):
    cfg = mi.CONFIGS[name]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    w = device_weights(mi.gen_weights(cfg, seed=0, layer=0), "cuda")
    ws = moe.Workspace(shape)
    for layer in (0, 1):  # two calls in a row with different activations
        inp = mi.gen_layer(cfg, seed=0, layer=layer, weights=False)
        logits = torch.from_numpy(inp["logits"]).cuda()
        hidden = bf16_tensor(inp["hidden"], "cuda")
        res = bf16_tensor(inp["residual"], "cuda")
        ids_a = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
        wts_a = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
        out_a = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.layer(shape, logits, hidden, w, res, out_a, ids_a, wts_a, ws)
        ids_b = torch.empty_like(ids_a)
        wts_b = torch.empty_like(wts_a)
        out_b = torch.full_like(out_a, float("nan"))
        assert _static_call(moe, shape, logits, hidden, w, res, out_b, ids_b, wts_b) == 0
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the results must be bit-identical (the
        # parity tolerance is reported as well, for the log)
        assert torch.equal(ids_b, ids_a)
        assert torch.equal(wts_b, wts_a)
        assert torch.equal(out_b, out_a)
        assert_parity(out_b.float().cpu().numpy(), out_a.float().cpu().numpy(), f"static workspace {name}")
        assert _static_status(moe) == 0
    assert moe.read_status(ws) == 0


def _static_status(m):
    bits = ctypes.c_uint32(0xffffffff)
    rc = m.lib().moe_static_workspace_read_status(1, ctypes.byref(bits),
                                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert (rc == 0) == (bits.value == 0)  # MOE_OK, or MOE_ERR_DEVICE with bits set
    return int(bits.value)


def test_static_workspace_reports_device_status(moe):
    # an out-of-FP16-range hidden value sets MOE_DEV_HIDDEN_RANGE in the static array's
    # status word, which the accessor reads (and clears)
    cfg = mi.CONFIGS["b1"]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    w = device_weights(mi.gen_weights(cfg, seed=0, layer=0), "cuda")
    inp = mi.gen_layer(cfg, seed=0, layer=0, weights=False)
    logits = torch.from_numpy(inp["logits"]).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    hidden[1, 5] = 1.0e6
    res = bf16_tensor(inp["residual"], "cuda")
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    assert _static_call(moe, shape, logits, hidden, w, res, out, ids, wts) == 0
    torch.cuda.synchronize()
    assert _static_status(moe) & moe.MOE_DEV_HIDDEN_RANGE
    assert _static_status(moe) == 0  # cleared by the read


def test_static_workspace_under_cuda_graph_capture(moe):
    # the reason for the entry point: captured into a graph (no allocation while capturing),
    # replayed with new inputs, equal to moe_layer on the same inputs
    cfg = mi.CONFIGS["b1"]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    w = device_weights(mi.gen_weights(cfg, seed=0, layer=0), "cuda")
    logits = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    res = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture (looks up the array's address)
        assert _static_call(moe, shape, logits, hidden, w, res, out, ids, wts) == 0
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert _static_call(moe, shape, logits, hidden, w, res, out, ids, wts) == 0
    ws = moe.Workspace(shape)
    for layer in (2, 3):
        inp = mi.gen_layer(cfg, seed=0, layer=layer, weights=False)
        logits.copy_(torch.from_numpy(inp["logits"]))
        hidden.copy_(bf16_tensor(inp["hidden"], "cuda"))
        res.copy_(bf16_tensor(inp["residual"], "cuda"))
        g.replay()
        ref = torch.empty_like(out)
        ids_r = torch.empty_like(ids)
        wts_r = torch.empty_like(wts)
        moe.layer(shape, logits, hidden, w, res, ref, ids_r, wts_r, ws)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_r) and torch.equal(wts, wts_r)
        assert torch.equal(out, ref)
        assert _static_status(moe) == 0


def test_static_workspace_rejects_shapes_beyond_its_size(moe):
    cfg = mi.CONFIGS["prefill"]
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    assert moe.workspace_bytes(shape) > (16 << 20)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    w = {"w13_codes": dummy, "w13_scales": dummy, "w2_codes": dummy, "w2_scales": dummy, "w13_ts": 1.0,
         "w2_ts": 1.0}
    rc = _static_call(moe, shape, dummy, dummy, w, dummy, dummy, dummy, dummy)
    assert rc == moe._lib.MOE_ERR_WORKSPACE
    assert b"static array" in moe.lib().moe_last_cuda_error()
