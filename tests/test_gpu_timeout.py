"""Failure detection of the expert kernels' bounded waits.

Forward progress in the persistent expert kernels rests on readiness counters, not grid
barriers ("Persistent execution for Flash-Next GGUF on SM70", section "First implementation
boundary"): a down task waits until every gate/up task of its expert has been published.  A
dependency that can never be met must end the launch with an error status that the host can
read, not a hang.  Each case builds a real plan, rewrites one down task to wait for a counter
that nothing increments, runs the kernel with every wait limited to ~0.5 ms, and checks that
(1) the launch completes, (2) the workspace status word carries MOE_DEV_TIMEOUT, and (3) the
same workspace, re-planned, then gives the bits of a clean call.  No GPU faults, traps or
hangs: the stuck wait is an unmet counter, and the kernel's own limit ends it.
"""
import time

import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_helpers import bf16_tensor, config_inputs, device_weights

pytestmark = pytest.mark.gpu

AUTO, TCGEN05, MMA, WIDE = 0, 1, 3, 4
WAIT_LIMIT_CYCLES = 1 << 20  # ~0.5 ms at 2 GHz

# (workload, algo): the decode kernel with the rows resident (B=1 through AUTO) and with
# gathered rows (B=8), the warp-MMA kernel of larger batches (B=64), the 16-row tcgen05
# kernel and the wide tcgen05 kernel
CASES = [("b1", AUTO), ("b8", MMA), ("b64", MMA), ("b8", TCGEN05), ("b8", WIDE)]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_moe_decode_gb300 as m
    return m


@pytest.mark.parametrize("name,algo", CASES)
def test_unmet_readiness_wait_times_out_and_workspace_recovers(moe, name, algo):
    cfg = mi.CONFIGS[name]
    inp = config_inputs(name)
    w = device_weights(inp, "cuda")
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).cuda()
    hidden = bf16_tensor(inp["hidden"], "cuda")
    res = bf16_tensor(inp["residual"], "cuda")
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")

    def clean_call():
        out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
        moe.front(shape, logits, hidden, ids, wts, ws)
        moe.forward_experts(shape, w, res, out, ws, algo)
        torch.cuda.synchronize()
        return out

    ref = clean_call()
    assert moe.read_status(ws) == 0

    # the failure: a fresh plan, down task 0 made to wait for a counter nobody publishes
    moe.front(shape, logits, hidden, ids, wts, ws)
    junk = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    moe.selftest_expert_timeout(shape, w, res, junk, ws, algo, 0, WAIT_LIMIT_CYCLES)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = moe.read_status(ws)  # read and clear
    assert status & moe.MOE_DEV_TIMEOUT, f"status {status:#x}"
    assert elapsed < 20.0, f"the launch took {elapsed:.1f} s to give up"

    # recovery: the same workspace, re-planned, gives the clean call's bits
    again = clean_call()
    assert moe.read_status(ws) == 0
    assert torch.equal(again, ref)


def test_timeout_selftest_rejects_bad_arguments(moe):
    cfg = mi.CONFIGS["b1"]
    inp = config_inputs("b1")
    w = device_weights(inp, "cuda")
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    ws = moe.Workspace(shape)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    for algo, dn_task, limit in ((2, 0, 1 << 20), (AUTO, -1, 1 << 20), (AUTO, 0, 0)):
        with pytest.raises(moe.MoeError):
            moe.selftest_expert_timeout(shape, w, None, out, ws, algo, dn_task, limit)
