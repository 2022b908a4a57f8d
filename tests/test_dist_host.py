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
