"""The bench's multi-process plumbing on CPU: two gloo ranks, barrier and max over ranks
(the timing rule for N > 1), and replica accounting of whole-job throughput."""
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT

CHILD = r"""
import os, sys, json, time
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch
import bench
d = bench.Dist(torch)
rank = d.rank
time.sleep(0.05 * rank)
d.barrier()
t = 10.0 + rank                      # per-rank "elapsed ms"
mx = d.max(t)
print(json.dumps({"rank": rank, "world": d.world, "max": mx}), flush=True)
d.close()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_barrier_and_max(tmp_path):
    port = _free_port()
    procs = []
    env0 = dict(os.environ, REPO_ROOT=ROOT, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                CUDA_VISIBLE_DEVICES="")
    for r in range(2):
        env = dict(env0, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, e
        outs.append(o.strip().splitlines()[-1])
    import json
    res = sorted((json.loads(o) for o in outs), key=lambda r: r["rank"])
    assert [r["world"] for r in res] == [2, 2]
    assert all(r["max"] == 11.0 for r in res)  # every rank sees the slowest rank's time


EP_CHILD = r"""
import os, sys, json
sys.path.insert(0, os.environ["REPO_ROOT"])
import numpy as np
import torch
import torch.distributed as dist
import moe_inputs as mi
from oracle import oracle as O
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
cfg = mi.CONFIGS["tiny"].replace(name="ep-host", T=24, E=16, k=4, tag=500)
inp = mi.gen_layer(cfg, seed=11)
ids, wts = O.route_topk(inp["logits"], cfg.k)           # every rank routes all tokens
e0, e1 = rank * cfg.E // world, (rank + 1) * cfg.E // world  # contiguous expert blocks
local = (ids >= e0) & (ids < e1)
w = np.where(local, wts, 0.0).astype(np.float32)        # other ranks' slots add nothing
part = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids, w, inp,
                     inp["residual"] if rank == 0 else None)
owners = torch.from_numpy(local.astype(np.int32))
dist.all_reduce(owners)                                 # each route owned by exactly one rank
t = torch.from_numpy(part.astype(np.float64))
dist.all_reduce(t)                                      # the exchange step of expert parallelism
full = O.moe_experts((cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k), inp["hidden"], ids, wts, inp, inp["residual"])
err = float(np.abs(t.numpy() - full).max() / np.sqrt(np.mean(full.astype(np.float64) ** 2)))
print(json.dumps({"rank": rank, "owners_ok": bool((owners.numpy() == 1).all()), "err": err,
                  "local_routes": int(local.sum())}), flush=True)
dist.destroy_process_group()
"""


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_expert_parallel_partial_sums(world):
    """Expert-parallel partition checked on host ranks: each rank computes the oracle's
    partial layer over its block of experts (residual on rank 0 only), an all-reduce sums
    the partials, and the sum matches the whole layer's oracle to FP32 rounding."""
    port = _free_port()
    env0 = dict(os.environ, REPO_ROOT=ROOT, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                CUDA_VISIBLE_DEVICES="")
    procs = [subprocess.Popen([sys.executable, "-c", EP_CHILD], env=dict(env0, RANK=str(r), LOCAL_RANK=str(r)),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(world)]
    import json
    res = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, e
        res.append(json.loads(o.strip().splitlines()[-1]))
    assert all(r["owners_ok"] for r in res)
    assert sum(r["local_routes"] for r in res) == 24 * 4
    assert all(r["err"] <= 1e-5 for r in res)
