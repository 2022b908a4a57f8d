#!/usr/bin/env python
"""Benchmark of the routed MoE layer (router + plan + NVFP4 experts + un-route) on GB300.

One step = one layer call (moe_route_topk, moe_plan, moe_forward) on one batch of the
workload.  Steps cycle over 12 independent layer weight sets (10.9 GB for the d=2048
shapes), so the streamed weights never fit the 129 MB L2.  The timed region replays
CUDA graphs of those calls; the expert kernel is additionally timed alone with CUDA
events for its roofline figure; `e2e` times the public C-ABI call with host buffers
(H2D of logits/hidden/residual, D2H of the output) per step.

A default run (B=1 verify, MOE_ALGO_AUTO) also measures the metric's other
configurations -- T=32, T=256 and the T=8192 prefill chunk -- on the same weight sets,
each with its own steps, warm-up, expert-kernel samples, roofline and clock record,
under "configs" in the same line; the headline `value` stays the B=1 figure.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_inputs as mi  # noqa: E402

METRIC = "MoE layer µs and tokens/s at T=4/32/256/8192; % of HBM roofline (unique-expert bytes)"
DEFAULT_STEPS = {"tiny": 20000, "b1": 48000, "b8": 12000, "b64": 6000, "prefill": 1200, "b64_literal": 6000}
WORKLOAD = {
    "tiny": "tiny parity case: T=4 d=256 ffn=128 E=16 top-2",
    "b1": "decode verify B=1 (1 request x 4 rows): T=4 d=2048 ffn=512 E=512 top-10, NVFP4 experts",
    "b8": "decode verify B=8 (8 requests x 4 rows, per-request expert bias): T=32 d=2048 ffn=512 E=512 top-10",
    "b64": "decode batch B=64 (Zipf expert popularity): T=256 d=2048 ffn=512 E=512 top-10",
    "prefill": "prefill chunk: T=8192 d=2048 ffn=512 E=512 top-10",
    "b64_literal": "decode batch B=64, literal Zipf coefficient: T=256 d=2048 ffn=512 E=512 top-10",
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--config", default="b1", choices=sorted(mi.CONFIGS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--algo", default="auto", choices=["auto", "mma", "tcgen05", "simt", "wide"])
    p.add_argument("--layers", type=int, default=None, help="weight sets cycled (default 12)")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-sub-configs", action="store_true",
                   help="measure the headline configuration only (default: also T=32, 256 and 8192)")
    p.add_argument("--kernel-samples", type=int, default=None,
                   help="expert-kernel launches timed alone for the roofline (default max(400, min(steps, 2000)))")
    return p.parse_args()


# ----------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data-path collective)
# ----------------------------------------------------------------------------------
class Dist:
    def __init__(self, torch):
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if self.torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local])
            else:
                self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        dev = f"cuda:{self.local}" if self.torch.cuda.is_available() else "cpu"
        t = self.torch.tensor([v], dtype=self.torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tensor_peak():
    """Dense FP16/BF16 tensor peak in TFLOP/s for a kernel timed alone (the burst figure):
    kind::f16 MMAs run FP16 and BF16 operands at the same rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured cuBLAS bf16 GEMM (burst)"
    return 1900.0, "fallback bf16 (burst)"


def kernel_source_digest(kernel: str) -> str:
    """First 16 hex digits of the SHA-256 of the kernel's .cu file followed by every shared
    header of the CUDA sources (sorted by name): the source a DRAM capture was taken of."""
    csrc = os.path.join(ROOT, "routed_moe_decode_gb300", "csrc")
    h = hashlib.sha256(open(os.path.join(csrc, f"{kernel}.cu"), "rb").read())
    for name in sorted(f for f in os.listdir(csrc) if f.endswith(".cuh")):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str, kernel: str):
    """DRAM bytes per expert-kernel launch from the committed ncu summary of this workload,
    or None if there is none or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}_dram.txt")
    if not os.path.exists(path):
        return None
    digest = kernel_source_digest(kernel)
    vals = {}
    for line in open(path):
        if line.startswith("#") or ":" not in line:
            continue
        # the source hash line's key holds a colon itself ("<kernel>.cu sha256[:16]: <hex>")
        k, v = line.rsplit(":", 1) if "sha256[:16]" in line else line.split(":", 1)
        vals[k.strip()] = v.strip()
    if vals.get(f"{kernel}.cu sha256[:16]", vals.get("source_sha256_16")) != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ----------------------------------------------------------------------------------
def time_oracle(cfg, inp, budget_s: float, max_steps: int | None = None, warmup: int = 1):
    """Oracle on one token per step (routing of the batch + that token's k expert routes),
    cycling over the batch's tokens until the budget (or max_steps) is used."""
    from oracle import oracle as O
    ids, wts = O.route_topk(inp["logits"], cfg.k)
    dims = (cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    out = np.zeros((cfg.T, cfg.d), np.float32)

    def one(t):
        mask = np.zeros(cfg.T, np.uint8)
        mask[t] = 1
        O.route_topk(inp["logits"][t:t + 1], cfg.k)
        O.moe_experts(dims, inp["hidden"], ids, wts, inp, inp["residual"], mask, out=out)

    for i in range(warmup):
        one(i % cfg.T)
    n, t0 = 0, time.perf_counter()
    while True:
        one(n % cfg.T)
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or el >= budget_s:
            break
    return n, el


def reference_arm(args, cfg, dist):
    if dist.rank != 0:
        return None
    steps = args.steps if args.steps is not None else 10
    warm = min(args.warmup if args.warmup is not None else 1, 2)
    inp = mi.gen_layer(cfg, seed=0, layer=0)
    n, el = time_oracle(cfg, inp, budget_s=120.0, max_steps=steps, warmup=warm)
    value = n / el
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": n,
        "warmup": warm, "ms_per_step": 1e3 * el / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded moe_inputs workload)",
        "config": {"workload": WORKLOAD[cfg.name], "T": cfg.T, "d": cfg.d, "ffn": cfg.ffn, "E": cfg.E, "k": cfg.k,
                   "step": "one token of the batch (its k expert routes) through the CPU oracle"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} single-token steps of layer 0 ({cfg.name}), FP32 C++ oracle, 1 thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# ----------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------
def load_weight_sets(cfg, L, dev, torch):
    """L independent layer weight sets of `cfg`, resident in HBM."""
    Wd = []
    for layer in range(L):
        w = mi.gen_weights(cfg, seed=0, layer=layer)
        d = {n: torch.from_numpy(w[n]).to(dev) for n in ("w13_codes", "w13_scales", "w2_codes", "w2_scales")}
        d["w13_ts"], d["w2_ts"] = w["w13_ts"], w["w2_ts"]
        Wd.append(d)
    torch.cuda.synchronize()
    return Wd


def measure(cfg, moe, torch, dist, dev, Wd, algo, K, W, kernel_samples, e2e_steps=0, clock_gpu=None):
    """Time K layer calls of `cfg` (CUDA-graph replays over the weight sets Wd, inputs of
    each layer resident in HBM), then the expert kernel alone over `kernel_samples`
    launches, then (if e2e_steps) the public call with host buffers.  Returns a dict."""
    L = len(Wd)
    shape = moe.shape_of(cfg.T, cfg.d, cfg.ffn, cfg.E, cfg.k)
    logits, hidden, resid, host = [], [], [], []
    for layer in range(L):
        inp = mi.gen_layer(cfg, seed=0, layer=layer, weights=False)
        logits.append(torch.from_numpy(inp["logits"]).to(dev))
        hidden.append(torch.from_numpy(inp["hidden"].view(np.int16)).to(dev).view(torch.bfloat16))
        resid.append(torch.from_numpy(inp["residual"].view(np.int16)).to(dev).view(torch.bfloat16))
        host.append(inp)
    ws = moe.Workspace(shape, device=dev)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)

    def step(l):
        if algo == moe.ALGO_AUTO:
            # the public one-call layer (fused router + plan front for moderate T * k)
            moe.layer(shape, logits[l], hidden[l], Wd[l], resid[l], out, ids, wts, ws)
            return
        moe.route_topk(shape, logits[l], ids, wts)
        moe.plan(shape, ids, wts, ws)
        moe.forward_prepare(shape, hidden[l], ws)
        moe.forward_experts(shape, Wd[l], resid[l], out, ws, algo)

    # front kernel(s), expert kernel(s), un-route kernel (none when the expert kernel runs it);
    # the library reports the launches of its own layer call
    fused_unroute = moe.unroute_fused(shape, algo)
    run_algo = moe.auto_algo(shape) if algo == moe.ALGO_AUTO else algo
    one_launch = algo == moe.ALGO_AUTO and moe.layer_launches(shape) == 1
    # the decode kernel (expert_dec.cu) serves the warp-MMA path up to 256 tokens
    dec_kernel = run_algo == moe.ALGO_MMA and cfg.T <= 256
    if algo == moe.ALGO_AUTO:
        kernels_per_step = moe.layer_launches(shape)
    else:
        front_kernels = 3
        # the SIMT path runs two expert kernels; the wide kernel runs after its route-order
        # gather and its task-table kernel
        expert_kernels = {moe.ALGO_SIMT: 2, moe.ALGO_WIDE: 3}.get(run_algo, 1)
        kernels_per_step = front_kernels + expert_kernels + (0 if fused_unroute else 1)

    # ---- unique experts per layer (outside any timed region) ----
    U = []
    for l in range(L):
        step(l)
        u, _ = moe.plan_summary(shape, ws)
        U.append(u)
    if moe.read_status(ws):
        raise RuntimeError("device status bits set during set-up")
    bpe = mi.weight_bytes_per_expert(cfg)
    R = cfg.T * cfg.k
    # expert kernel besides the weights: FP16 hidden read, FP16 h written and read back,
    # FP32 per-route down outputs written
    act_bytes = cfg.T * cfg.d * 2 + 2 * R * cfg.ffn * 2 + R * cfg.d * 4
    if fused_unroute:
        # and the un-route: per-route outputs read back, positions and weights, residual, out
        act_bytes += R * cfg.d * 4 + R * 8 + 2 * cfg.T * cfg.d * 2
    if one_launch:
        # and the router's logits
        act_bytes += cfg.T * cfg.E * 4
    unique_bytes = [u * bpe for u in U]

    # ---- CUDA graphs: one of all L layers, one per single layer (for K % L) ----
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l in range(L):
            step(l)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all):
        for l in range(L):
            step(l)
    g_one = []
    for l in range(L):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(l)
        g_one.append(g)

    def run_steps(n, offset=0):
        done = 0
        while done < n and (offset + done) % L != 0:
            g_one[(offset + done) % L].replay()
            done += 1
        while n - done >= L:
            g_all.replay()
            done += L
        while done < n:
            g_one[(offset + done) % L].replay()
            done += 1

    # Up to kOneGraphSteps timed steps run as ONE graph of exactly those K layer calls (layers
    # (W + i) mod L), so that a short timed region has no graph boundaries inside it; longer
    # runs replay the graph of all L layers (plus single-layer graphs for the ends).
    g_timed = None
    if K <= ONE_GRAPH_STEPS:
        g_timed = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_timed):
            for i in range(K):
                step((W + i) % L)

    def run_timed():
        if g_timed is not None:
            g_timed.replay()
        else:
            run_steps(K, offset=W % L)

    # ---- warm-up and timed region ----
    run_steps(W)
    torch.cuda.synchronize()
    sampler = ClockSampler(clock_gpu)
    sampler.start()
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    run_timed()
    ev1.record()
    ev1.synchronize()
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    t_ms = ev0.elapsed_time(ev1)
    t_ms = dist.max(t_ms)
    status = moe.read_status(ws)
    del g_all, g_one, g_timed

    steps_layers = [(W + i) % L for i in range(K)]
    us_per_layer = 1e3 * t_ms / K
    mean_unique = sum(unique_bytes[l] for l in steps_layers) / K

    # ---- the expert kernel's duration ----
    # The one-launch layer is its own expert kernel: the timed region's events bracket its K
    # launches and nothing else.  Otherwise, CUDA events around each expert-kernel launch
    # outside the timed region, after a GPU-side sleep that keeps the device busy while the
    # host enqueues the front kernels, the events and the expert kernel.
    Kk = K if one_launch else kernel_samples
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(0 if one_launch else Kk)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(0 if one_launch else Kk)]
    kbytes = sum(unique_bytes[l] for l in steps_layers) + K * act_bytes if one_launch else 0.0
    for i in range(0 if one_launch else Kk):
        l = i % L
        torch.cuda._sleep(200_000)
        moe.route_topk(shape, logits[l], ids, wts)
        moe.plan(shape, ids, wts, ws)
        moe.forward_prepare(shape, hidden[l], ws)
        if fused_unroute:
            starts[i].record()
            moe.forward_experts(shape, Wd[l], resid[l], out, ws, algo)  # one kernel
            ends[i].record()
        else:
            # the kernels that prepare the expert kernel's input (the wide path's route-order
            # gather and task table) run before the events, the expert kernel between them
            moe.selftest_expert_part(shape, Wd[l], ws, algo, 0)
            starts[i].record()
            moe.selftest_expert_part(shape, Wd[l], ws, algo, 1)
            ends[i].record()
            moe.forward_unroute(shape, resid[l], out, ws)
        kbytes += unique_bytes[l] + act_bytes
    torch.cuda.synchronize()
    kdur_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)] if not one_launch else [t_ms / K]
    k_avg_ms = sum(kdur_ms) / len(kdur_ms)
    achieved = kbytes / Kk / (k_avg_ms * 1e-3) / 1e9
    peak, peak_kind = load_peaks()
    kname = {moe.ALGO_MMA: "expert_dec" if dec_kernel else "expert_mma", moe.ALGO_TCGEN05: "expert_tc",
             moe.ALGO_WIDE: "expert_wide"}.get(run_algo)
    traffic = profiled_traffic(cfg.name, kname) if kname else None

    # ---- end to end through the public C-ABI call with host buffers ----
    e2e = None
    if e2e_steps:
        Ke = e2e_steps
        pin = [{k_: torch.from_numpy(h[k_] if k_ == "logits" else h[k_].view(np.int16)).pin_memory()
                for k_ in ("logits", "hidden", "residual")} for h in host]
        d_log = torch.empty_like(logits[0])
        d_hid = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device=dev)
        d_res = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device=dev)
        h_out = torch.empty((cfg.T, cfg.d), dtype=torch.int16).pin_memory()

        def e2e_step(l):
            d_log.copy_(pin[l]["logits"], non_blocking=True)
            d_hid.copy_(pin[l]["hidden"], non_blocking=True)
            d_res.copy_(pin[l]["residual"], non_blocking=True)
            moe.layer(shape, d_log, d_hid.view(torch.bfloat16), Wd[l], d_res.view(torch.bfloat16), out, ids, wts, ws)
            h_out.copy_(out.view(torch.int16), non_blocking=True)

        for i in range(3):
            e2e_step(i % L)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(Ke):
            e2e_step(i % L)
        e1.record()
        e1.synchronize()
        et = dist.max(e0.elapsed_time(e1))
        e2e = {"value": cfg.T * Ke * dist.world / (et * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": cfg.T * cfg.E * 4 + 2 * cfg.T * cfg.d * 2,
               "d2h_bytes_per_step": cfg.T * cfg.d * 2, "steps": Ke,
               "us_per_layer": 1e3 * et / Ke}

    roofline_hbm = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "peak_kind": f"{peak_kind} copy bandwidth",
                    "algorithmic_bytes": "unique experts x NVFP4 bytes per expert + FP16 hidden + FP16 h (write+read) + "
                                         "FP32 per-route down outputs"
                                         + (" (written and read back) + route positions and weights + BF16 residual and out"
                                            if fused_unroute else ""),
                    "algorithmic_bytes_per_launch": kbytes / Kk}
    # the wide kernel is a dense contraction: 2 flops per weight per routed row, gate/up
    # (2F x d) and down (d x F) for each of the T * k routes
    tpeak, tpeak_kind = load_tensor_peak()
    tflops = 6.0 * R * cfg.d * cfg.ffn / (k_avg_ms * 1e-3) / 1e12
    roofline_tensor = {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                       "peak_kind": tpeak_kind, "mma": "tcgen05 kind::f16 (FP16 x FP16 -> FP32)",
                       "algorithmic_flops": "6 x T x k x d x ffn per launch",
                       "hbm_achieved_gbs": achieved, "hbm_frac": achieved / peak}
    roofline = roofline_hbm if run_algo != moe.ALGO_WIDE else roofline_tensor
    roofline.update({"traffic": traffic,
                     "traffic_source": (f"profiles/{kname}_{cfg.name}_dram.txt (ncu dram__bytes_read.sum + "
                                        "dram__bytes_write.sum of one launch; null once the kernel source changed)")
                     if kname else None,
                     "kernel": (f"{kname}_kernel"
                                + ("<own front, fused un-route> (the whole layer)" if one_launch
                                   else "<fused un-route>" if fused_unroute
                                   else "<gathered rows>" if dec_kernel else "")
                                + (" (timed alone: its route-order gather and task table run before the events)" if run_algo == moe.ALGO_WIDE else "")) if kname
                               else "simt kernels",
                     "kernel_us": 1e3 * k_avg_ms, "kernel_samples": Kk,
                     "kernel_timing": "the timed region's events (K launches of this one kernel)" if one_launch
                                      else "CUDA events around each launch, outside the timed region"})
    return {
        "t_ms": t_ms, "K": K, "W": W, "us_per_layer": us_per_layer,
        "tokens_per_s": cfg.T * K * dist.world / (t_ms * 1e-3),
        "unique_experts_mean": sum(U[l] for l in steps_layers) / K,
        "unique_bytes_mean": mean_unique,
        "hbm_frac_layer": (mean_unique / (us_per_layer * 1e-6) / 1e9) / peak,
        "roofline": roofline, "clocks": clocks, "status": status, "e2e": e2e,
        "gpu_launches": kernels_per_step * K, "kernels_per_step": kernels_per_step,
    }


ONE_GRAPH_STEPS = 2400

# Configurations measured besides the headline one in a default run (the metric is quoted
# at T = 4 / 32 / 256 / 8192): steps, warm-up and expert-kernel samples of each.
SUB_CONFIGS = {"b8": (240, 24, 200), "b64": (120, 24, 120), "prefill": (36, 12, 24)}


def cpu_info():
    """Host CPU model name and logical core count."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
            for line in r.stdout.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"model": model or platform.processor() or platform.machine(), "arch": platform.machine(),
            "nproc": os.cpu_count()}


def our_arm(args, cfg, dist, torch):
    import __graft_entry__
    __graft_entry__.build()  # no-op when the in-tree library is current
    import routed_moe_decode_gb300 as moe
    dev = torch.device(f"cuda:{dist.local}")
    torch.cuda.set_device(dev)
    algo = {"auto": moe.ALGO_AUTO, "mma": moe.ALGO_MMA, "tcgen05": moe.ALGO_TCGEN05, "simt": moe.ALGO_SIMT,
            "wide": moe.ALGO_WIDE}[args.algo]
    L = args.layers if args.layers is not None else min(12, max(1, cfg.layers))
    K = args.steps if args.steps is not None else DEFAULT_STEPS[cfg.name]
    W = args.warmup if args.warmup is not None else max(3, 2 * L)
    W = max(W, 3)
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clock_gpu = gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}"

    t_gen = time.perf_counter()
    Wd = load_weight_sets(cfg, L, dev, torch)
    t_gen = time.perf_counter() - t_gen
    ksamples = args.kernel_samples if args.kernel_samples is not None else max(400, min(K, 2000))
    m = measure(cfg, moe, torch, dist, dev, Wd, algo, K, W, ksamples,
                e2e_steps=0 if args.no_e2e else min(max(K, 200), 3000), clock_gpu=clock_gpu)

    # ---- the metric's other configurations, on the same weight sets (same shapes) ----
    subs = {}
    same_shape = lambda c: (c.d, c.ffn, c.E, c.k) == (cfg.d, cfg.ffn, cfg.E, cfg.k)
    if cfg.name == "b1" and not args.no_sub_configs and algo == moe.ALGO_AUTO:
        for name, (ks, ws_, kk) in SUB_CONFIGS.items():
            sc = mi.CONFIGS[name]
            if not same_shape(sc):
                continue
            sm = measure(sc, moe, torch, dist, dev, Wd, algo, ks, ws_, kk, clock_gpu=clock_gpu)
            subs[name] = {
                "workload": WORKLOAD[name], "T": sc.T, "steps": ks, "warmup": ws_,
                "us_per_layer": sm["us_per_layer"], "tokens_per_s": sm["tokens_per_s"],
                "unique_experts_mean": sm["unique_experts_mean"], "unique_bytes_mean": sm["unique_bytes_mean"],
                "hbm_frac_layer": sm["hbm_frac_layer"], "roofline": sm["roofline"], "clocks": sm["clocks"],
                "device_status": sm["status"],
                "weights": "the headline workload's weight sets (same shapes and distribution)",
            }

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, one GPU only) ----
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        keep_host = mi.gen_layer(cfg, seed=0, layer=0)
        n, el = time_oracle(cfg, keep_host, budget_s=args.cpu_seconds)
        info = cpu_info()
        cpu = {"value": n / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "host_cpu": info["model"], "host_arch": info["arch"], "host_nproc": info["nproc"],
               "sample": f"{n} single-token steps of layer 0 ({cfg.name}) through the FP32 C++ oracle, "
                         f"{el:.1f} s on 1 host thread of {info['nproc']} ({info['model']})"}

    line = {
        "metric": METRIC,
        "value": m["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": W,
        "ms_per_step": m["t_ms"] / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded moe_inputs workload; random NVFP4 weights)",
        "config": {
            "workload": WORKLOAD[cfg.name], "T": cfg.T, "d": cfg.d, "ffn": cfg.ffn, "E": cfg.E, "k": cfg.k,
            "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
            "algo": args.algo, "weights": "NVFP4 (E2M1 + E4M3/16 + FP32)", "mma": "FP16 x FP16 -> FP32",
            "layers_cycled": L, "l2": f"inputs larger than L2: {L} layer weight sets "
                                      f"({L * cfg.E * mi.weight_bytes_per_expert(cfg) / 1e9:.1f} GB) cycled",
            "timing": (f"one CUDA graph of the {K} timed layer calls" if K <= ONE_GRAPH_STEPS
                       else f"CUDA graphs of {L} layer calls replayed") + "; events on the launch stream",
            "us_per_layer": m["us_per_layer"],
            "unique_experts_mean": m["unique_experts_mean"],
            "unique_bytes_mean": m["unique_bytes_mean"],
            "hbm_frac_layer": m["hbm_frac_layer"],
            "input_gen_s": round(t_gen, 1),
        },
        "roofline": m["roofline"],
        "clocks": m["clocks"],
        "gpu_launches": m["gpu_launches"],
        "device_status": m["status"],
    }
    if subs:
        line["configs"] = subs
    if m["e2e"] is not None:
        line["e2e"] = m["e2e"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def main():
    args = parse_args()
    cfg = mi.CONFIGS[args.config]
    import torch
    dist = Dist(torch)
    try:
        if args.impl == "reference":
            line = reference_arm(args, cfg, dist)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
            line = our_arm(args, cfg, dist, torch)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
