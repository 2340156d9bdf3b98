#!/usr/bin/env python3
"""Benchmark: weight-stream GB/s and us/call of the int8 decode GEMM (M <= 32), cold-L2 graph replay.

Workload (default): W8A8 GEMM M=16, K=4096, N=24576, the MLP gate_up decode shape (the largest
single-GPU decode shape of the workloads), int8 x_q and W from a clipped Gaussian (sigma 40, clip
+-127), fp32 scales log-uniform in [1e-4, 1e-1], seeded synthetic data.  R rotating packed-W
buffers, R = max(16, ceil(3 * L2 / W_bytes)), so every call streams its weight cold from HBM
(inputs larger than L2; no flush needed).  One step = one CUDA-graph replay of C calls cycling
through the R buffers.  W warm-up steps, then K timed steps bracketed by a barrier and a device
synchronise, timed with CUDA events on the launching stream; max over ranks.

Beside the headline the line reports the same call launched with PDL, the MLP down shape and the
fused-QKV-like shape (plain and PDL), an end-to-end leg with host buffers, the Q8_0 reads (plain
and RMS-norm), the quantisation rows, the 32 < M <= 128 arm at M = 128 (tensor_memory_arm), the
read ceiling and the oracle's CPU baseline (one thread and all host cores).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]
Under torchrun each rank runs an independent replica (the operator has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-stream GB/s and us/call, int8 decode GEMM M<=32, cold-L2 graph replay"
DATA = {"mlp": "synthetic (seeded SplitMix64 streams; int8 clipped Gaussian sigma=40 clip +-127, fp32 scales "
               "log-uniform [1e-4,1e-1])",
        "uniform": "synthetic (seeded SplitMix64 streams; int8 U[-127,127], fp32 scales U[1e-3,2e-2])"}
# The decode shapes the line reports: the headline (timed as `value`) and the shapes beside it.
WORKLOADS = {
    "gate_up": dict(M=16, K=4096, N=24576, dist="mlp", seed=4, label="MLP gate_up decode shape"),
    "down": dict(M=16, K=12288, N=4096, dist="mlp", seed=4, label="MLP down decode shape"),
    "qkv": dict(M=16, K=4096, N=1536, dist="uniform", seed=1, label="fused-QKV-like decode shape"),
}
HEADLINE = "gate_up"
DEFAULT = WORKLOADS[HEADLINE]
# Sources of the timed kernel and its plan: the committed DRAM-traffic figure is valid only while
# these are unchanged.
KERNEL_SOURCES = ["int8_weight_gemm_gb300/csrc/w8a8_gemm.cu", "int8_weight_gemm_gb300/csrc/common.cuh",
                  "int8_weight_gemm_gb300/csrc/internal.h", "int8_weight_gemm_gb300/csrc/api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "w8a8_gemm_m16_k4096_n24576_traffic.txt")


def workload_config(name: str, world: int) -> dict:
    """The `config` object of a bench line for one workload (shared by both arms)."""
    w = WORKLOADS[name]
    return {"workload": f"W8A8 GEMM M={w['M']}, K={w['K']}, N={w['N']} ({w['label']})",
            "M": w["M"], "K": w["K"], "N": w["N"], "dist": w["dist"], "seed": w["seed"],
            "l2": "inputs larger than L2: each call streams a different packed W buffer, rotating over "
                  "max(16, ceil(3 x L2 / W bytes)) buffers",
            "parallelism": f"replicas x{world}"}


def rank_barrier():
    """Barrier across the ranks of a torchrun launch (no-op for a single process)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    """The largest of the ranks' values (each rank's timed region; the job is as slow as its
    slowest rank).  NCCL reduces a device tensor, gloo a host one."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_call: int, calls_per_rank: int, total_ms_max: float) -> float:
    """Whole-job weight-stream GB/s: every rank streams its own replica's weights (weak scaling),
    timed by the slowest rank."""
    return world * bytes_per_call * calls_per_rank / (total_ms_max / 1e3) / 1e9


def p90(sorted_values):
    """Nearest-rank 90th percentile of an ascending list: the smallest value with at least 90 % of
    the samples at or below it (never below the median)."""
    return sorted_values[max(0, math.ceil(0.9 * len(sorted_values)) - 1)]


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_per_launch():
    """dram read+write bytes per launch from the committed ncu summary, if its kernel is current."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    vals = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != _kernel_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host cores, on a bounded sample of the workload
# ---------------------------------------------------------------------------------------------

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


class OracleOnCores:
    """The oracle's W8A8 GEMM (plain C, one thread per call) over all host cores: the columns of W
    are cut into one contiguous slice per thread and each thread calls the oracle on its slice
    (ctypes releases the interpreter lock for the call).  Columns are independent, so the slices
    together give the whole result; the oracle itself is used as it stands."""

    def __init__(self, x, xs, W, ws, threads=None, cols=None):
        import concurrent.futures as cf

        N = W.shape[1] if cols is None else cols
        self.threads = max(1, min(threads or host_cores(), N // 8))
        cuts = [round(i * N / self.threads) for i in range(self.threads + 1)]
        self.parts = [(np.ascontiguousarray(W[:, a:b]), np.ascontiguousarray(ws[a:b]))
                      for a, b in zip(cuts[:-1], cuts[1:])]
        self.x, self.xs, self.N = x, xs, N
        self.pool = cf.ThreadPoolExecutor(max_workers=self.threads)

    def call(self):
        import oracle

        futs = [self.pool.submit(oracle.w8a8_gemm, self.x, self.xs, Wp, wp) for Wp, wp in self.parts]
        return np.concatenate([f.result() for f in futs], axis=1)

    def close(self):
        self.pool.shutdown()


def cpu_baseline(M, K, N, x, xs, W, ws, budget_s=8.0):
    """The oracle timed on the host: one thread on a column sample, then all host cores on the
    whole workload (threads over column slices), each for about budget_s seconds."""
    import oracle

    cols = min(N, 2048)
    Ws = np.ascontiguousarray(W[:, :cols])
    wss = np.ascontiguousarray(ws[:cols])
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.w8a8_gemm(x, xs, Ws, wss)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or calls >= 200:
            break
    single = {"value": K * cols / (el / calls) / 1e9, "unit": "GB/s", "cores": 1,
              "sample": f"{calls} oracle calls on M={M}, K={K}, N={cols} (of {N}) columns, one thread, "
                        f"{el / calls * 1e3:.1f} ms/call"}
    par = OracleOnCores(x, xs, W, ws)
    par.call()
    calls = 0
    t0 = time.perf_counter()
    while True:
        par.call()
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or calls >= 200:
            break
    par.close()
    per_call = el / calls
    return {"value": K * N / per_call / 1e9, "unit": "GB/s", "cores": par.threads, "kind": "oracle",
            "sample": f"{calls} whole calls of M={M}, K={K}, N={N}, the columns cut over {par.threads} threads "
                      f"(one per host core), {per_call * 1e3:.1f} ms/call",
            "single_thread": single}


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def time_gemm(M, K, N, dist, seed, steps, warmup, blocks=0, device=None, sample_clocks=False, want_e2e=True,
              flags=0):
    import torch

    import int8_weight_gemm_gb300 as lib8
    import synth

    dev = device or torch.device("cuda")
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=seed, dist=dist)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    wbytes = lib8.w8a8_packed_weight_bytes(K, N)
    R = max(16, math.ceil(3 * l2 / wbytes))
    C = R * max(1, math.ceil(256 / R))                     # calls per graph replay
    xd = torch.from_numpy(x).to(dev)
    xsd = torch.from_numpy(xs).to(dev)
    wsd = torch.from_numpy(ws).to(dev)
    Wd = torch.from_numpy(W).to(dev)
    wsp = lib8.alloc_workspace(lib8.w8a8_workspace_bytes(M, K, N, blocks), dev)
    packed0 = lib8.w8a8_pack_weights(Wd, ws=wsp)
    del Wd
    packs = [packed0] + [packed0.clone() for _ in range(R - 1)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(R):                       # eager warm-up (also loads the module)
            lib8.w8a8_gemm(xd, xsd, packs[i], wsd, wsp, N, out=out, blocks=blocks, flags=flags, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in range(C):
            lib8.w8a8_gemm(xd, xsd, packs[c % R], wsd, wsp, N, out=out, blocks=blocks, flags=flags, stream=stream)
    torch.cuda.synchronize(dev)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    rank_barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index or 0) if sample_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.15)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            g.replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    total_ms = max_over_ranks(evs[0].elapsed_time(evs[-1]))
    per_call_us = sorted(s * 1e3 / C for s in step_ms)
    plan = lib8.w8a8_plan(M, K, N, blocks, flags=flags)
    res = {
        "R": R, "C": C, "wbytes": wbytes, "total_ms": total_ms, "steps": steps,
        "kernel": (f"w8a8_gemm_tc_kernel<{plan['n8_tiles'] // 2}>" if plan["tensor_memory"] else
                   f"w8a8_gemm_kernel<{plan['n8_tiles']}, {plan['stages']}, {str(plan['threads'] == 320).lower()}>"),
        "blocks": plan["blocks"],
        "us_median": statistics.median(per_call_us),
        "us_p90": p90(per_call_us),
        "avg_launch_us": total_ms * 1e3 / (steps * C),
        "clocks": clocks,
        "launches": steps * C,
        "inputs": (x, xs, W, ws),
    }
    # correctness spot check of the timed configuration (first rows, against the oracle)
    res["out"] = out
    if want_e2e:
        res["e2e"] = time_e2e(lib8, M, K, N, xd, xsd, packs, wsd, wsp, blocks, dev, steps=min(steps, 200), flags=flags)
    del packs
    return res


def time_e2e(lib8, M, K, N, xd, xsd, packs, wsd, wsp, blocks, dev, steps, flags=0):
    """The same call through the public API with host buffers: every step copies that step's
    activations and their scales from pinned host memory (one contiguous staging buffer, so one
    copy), runs the GEMM on a cold weight, and reads the result back to pinned host memory.  The
    steps are captured in a CUDA graph (copy in, GEMM, copy out, per step), as a serving engine
    captures its decode step; the same steps issued eagerly from Python, bound by the host's launch
    rate, are reported beside it."""
    import torch

    R = len(packs)
    # x_q [M, K] int8 then x_scale [M] fp32 in one buffer (M * K is a multiple of 32, so the scales
    # start 4-byte aligned); the device side is the same layout.
    nb = M * K + 4 * M
    stage_h = torch.empty(nb, dtype=torch.uint8).pin_memory()
    stage_h[: M * K].copy_(xd.cpu().view(torch.uint8).reshape(-1))
    stage_h[M * K:].copy_(xsd.cpu().view(torch.uint8))
    stage_d = torch.empty(nb, dtype=torch.uint8, device=dev)
    x_dev = stage_d[: M * K].view(torch.int8).view(M, K)
    xs_dev = stage_d[M * K:].view(torch.float32)
    outh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)

    def step(i):
        stage_d.copy_(stage_h, non_blocking=True)
        lib8.w8a8_gemm(x_dev, xs_dev, packs[i % R], wsd, wsp, N, out=out, blocks=blocks, flags=flags, stream=stream)
        outh.copy_(out, non_blocking=True)

    # Eager: one Python-issued step after another.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(steps + 3):
            if i == 3:
                e0.record(stream)
            step(i)
        e1.record(stream)
    stream.synchronize()
    eager_us = e0.elapsed_time(e1) * 1e3 / steps
    # Graph: C steps per replay, cycling over the rotating weights.
    C = R * max(1, math.ceil(32 / R))
    with torch.cuda.stream(stream):
        for i in range(C):
            step(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(C):
            step(i)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    reps = max(3, steps // C)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    per_step_us = e0.elapsed_time(e1) * 1e3 / (reps * C)
    del g
    wbytes = lib8.w8a8_packed_weight_bytes(K, N)
    return {"value": wbytes / per_step_us / 1e3, "unit": "GB/s", "us_per_step": per_step_us,
            "h2d_bytes_per_step": nb, "d2h_bytes_per_step": 2 * M * N,
            "launch": f"CUDA graph of {C} steps (copy in, GEMM, copy out per step), {reps} replays",
            "eager_us_per_step": eager_us}


def time_read_ceiling(dev, nbytes=1 << 30, reps=20):
    """The library's read-only probe over a buffer much larger than L2: the achievable HBM read rate."""
    import torch

    import int8_weight_gemm_gb300 as lib8

    buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    for _ in range(3):
        lib8.w8a8_read_probe(buf, sink)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        lib8.w8a8_read_probe(buf, sink)
    e1.record()
    torch.cuda.synchronize(dev)
    s = e0.elapsed_time(e1) / 1e3
    del buf
    torch.cuda.empty_cache()
    return {"value": round(nbytes * reps / s / 1e9, 1), "unit": "GB/s", "bytes_per_read": nbytes,
            "kernel": "w8a8_read_probe (16-byte loads, 2 x SMs x 512 threads)"}


def time_mma_rates(dev, iters=4096, reps=5):
    """The library's tensor-pipe rate probe: the fp16 m16n8k16 MMA the decode kernel uses against
    the int8 m16n8k32 MMA it does not, each as 2 x SMs CTAs of 8 warps (four per sub-partition),
    timed with CUDA events."""
    import torch

    import int8_weight_gemm_gb300 as lib8

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    out = []
    for kind, form, per_mma in ((0, "mma.sync m16n8k16 f16 x f16 -> f32", 4096), (1, "mma.sync m16n8k32 s8 x s8 -> s32", 8192)):
        for _ in range(2):
            lib8.w8a8_mma_rate_probe(kind, iters, sink)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            lib8.w8a8_mma_rate_probe(kind, iters, sink)
        e1.record()
        torch.cuda.synchronize(dev)
        s = e0.elapsed_time(e1) / 1e3
        ops = 2 * sms * 8 * iters * 8 * per_mma * reps
        out.append({"form": form, "kind": kind, "tera_ops_per_s": round(ops / s / 1e12, 1),
                    "us_per_launch": round(s * 1e6 / reps, 2), "mmas_per_launch": 2 * sms * 8 * iters * 8})
    return out


def time_graph_calls(make_call, R, calls=256, reps=20):
    """Median us per call of a CUDA graph of `calls` launches cycling over R buffer sets;
    make_call(i) issues call i on the current stream."""
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(R):
            make_call(i)
    s.synchronize()
    C = R * max(1, math.ceil(calls / R))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(C):
            make_call(i % R)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            g.replay()
            e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / C)
    del g
    return statistics.median(times), C


def time_quantisation_rows(peak):
    """The rows after the hot path: activation quantisation (inputs L2-hot, as when produced by the
    previous kernel), Q8_0 from BF16 and the block re-layout (weights cold: rotating > 3 x L2)."""
    import torch

    import int8_weight_gemm_gb300 as lib8

    dev = torch.device("cuda")
    rows = []
    for (M, K) in ((16, 4096), (32, 12288)):
        x = torch.randn((M, K), device=dev).to(torch.bfloat16)
        xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        xs = torch.empty(M, dtype=torch.float32, device=dev)
        us, _ = time_graph_calls(lambda i: lib8.w8a8_quantize_activations(x, xq, xs), 1)
        nbytes = 2 * M * K + M * K + 4 * M
        rows.append({"op": "w8a8_quantize_activations", "M": M, "K": K, "us_median": round(us, 3),
                     "bytes": nbytes, "GBps": round(nbytes / us / 1e3, 1), "inputs": "L2-hot"})
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20)
    for (N, K) in ((320, 4096), (4096, 320), (24576, 4096)):
        wbytes = 2 * N * K
        R = max(2, math.ceil(3 * l2 / wbytes))
        ws = [torch.randn((N, K), device=dev).to(torch.bfloat16) for _ in range(R)]
        q = torch.empty((N, K), dtype=torch.int8, device=dev)
        d = torch.empty((N, K // 32), dtype=torch.int16, device=dev)
        us, _ = time_graph_calls(lambda i: lib8.q8_0_quantize(ws[i], q, d), R)
        nbytes = 2 * N * K + N * K + 2 * N * (K // 32)
        rows.append({"op": "q8_0_quantize", "N": N, "K": K, "us_median": round(us, 3), "bytes": nbytes,
                     "GBps": round(nbytes / us / 1e3, 1), "frac_of_measured_hbm": round(nbytes / us / 1e3 / peak, 3),
                     "rotating_inputs": R})
        del ws
        bl = N * (K // 32) * 34
        R = max(2, math.ceil(3 * l2 / bl))
        bs = [torch.randint(0, 256, (bl,), dtype=torch.uint8, device=dev) for _ in range(R)]
        us, _ = time_graph_calls(lambda i: lib8.q8_0_split_from_blocks(bs[i], K, N, q, d), R)
        rows.append({"op": "q8_0_split_from_blocks", "N": N, "K": K, "us_median": round(us, 3), "bytes": 2 * bl,
                     "GBps": round(2 * bl / us / 1e3, 1), "frac_of_measured_hbm": round(2 * bl / us / 1e3 / peak, 3),
                     "rotating_inputs": R})
        del bs
        torch.cuda.empty_cache()
    return rows


def time_tensor_memory_arm(args, dev, hbm_peak):
    """The 32 < M <= 128 arm (tcgen05) at M = 128 on the fused-QKV-like shape and the gate_up MLP
    shape: the same rotating-weight graph replays as the headline, reported beside it.  At M = 128
    a weight byte feeds 256 flops, so the line gives both the HBM fraction (weight bytes) and the
    tensor fraction (2 M N K flops against the measured bf16 peak; the fp16 kind has the same
    nominal rate).  The arm is forced (W8A8_FLAG_TENSOR_MEMORY_ARM)."""
    import torch

    import int8_weight_gemm_gb300 as lib8

    peaks = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peaks = json.load(f)
    tensor_peak = float(peaks.get("bf16_tflops", 1900.0))
    rows = []
    for (M, K, N, dist, seed) in ((128, 4096, 1536, "uniform", 5128), (128, 4096, 24576, "mlp", 5)):
        r = time_gemm(M, K, N, dist, seed, min(args.steps, 100), args.warmup, device=dev, want_e2e=False,
                      flags=lib8.W8A8_FLAG_TENSOR_MEMORY_ARM)
        r.pop("inputs")
        us = r["us_median"]
        gbs = r["wbytes"] / (us * 1e-6) / 1e9
        tflops = 2.0 * M * N * K / (us * 1e-6) / 1e12
        rows.append({"M": M, "K": K, "N": N, "kernel": r["kernel"], "blocks": r["blocks"],
                     "us_per_call": {"median": round(us, 3), "p90": round(r["us_p90"], 3)},
                     "weight_GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
                     "tflops": round(tflops, 1), "frac_of_measured_bf16": round(tflops / tensor_peak, 4),
                     "launches_per_call": 2})
        del r
        torch.cuda.empty_cache()
    return rows


def time_q8(T, K, N, iters=200, seed=7, flags=0, rms=False):
    """Median us per Q8_0 read in a graph of calls over rotating weight sets (not L2-resident);
    rms=True times the RMS-norm variant (q8_0_gemv_rms) on the same weights."""
    import torch

    import int8_weight_gemm_gb300 as lib8
    import synth

    x, q, d = synth.q8_0_inputs(T, K, N, seed=seed)
    gd = torch.ones(K, dtype=torch.bfloat16, device="cuda") * 0.75

    def read(xd, qi, di, ws, y, stream):
        if rms:
            lib8.q8_0_gemv_rms(xd, gd, 1e-6, qi, di, ws, y=y, flags=flags, stream=stream)
        else:
            lib8.q8_0_gemv(xd, qi, di, ws, y=y, flags=flags, stream=stream)

    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    nbytes = N * K + 2 * N * (K // 32)
    R = max(8, math.ceil(3 * l2 / nbytes))
    xd = x.cuda()
    q0 = torch.from_numpy(q).cuda()
    d0 = torch.from_numpy(d.view(np.int16)).cuda()
    qs = [q0] + [q0.clone() for _ in range(R - 1)]
    ds = [d0] + [d0.clone() for _ in range(R - 1)]
    ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(R):
            read(xd, qs[i], ds[i], ws, y, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(R):
            read(xd, qs[i], ds[i], ws, y, s)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    samples = []
    for _ in range(max(10, iters // R)):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            g.replay()
            b.record(s)
        s.synchronize()
        samples.append(a.elapsed_time(b) * 1e3 / R)
    samples.sort()
    return {"T": T, "K": K, "N": N, "flags": flags, "rms_norm": rms, "us_median": statistics.median(samples),
            "us_p90": p90(samples), "weight_bytes": nbytes,
            "GBps": nbytes / statistics.median(samples) / 1e3}


def shape_summary(name, res, peak, world):
    """One beside-the-headline entry: median / p90 us per call, GB/s and roofline fraction."""
    w = WORKLOADS[name]
    alg = alg_bytes(w["M"], w["K"], w["N"])
    return {"workload": workload_config(name, world)["workload"], "kernel": res["kernel"], "blocks": res["blocks"],
            "us_per_call": {"median": round(res["us_median"], 4), "p90": round(res["us_p90"], 4)},
            "weight_GBps": round(res["wbytes"] / (res["us_median"] * 1e-6) / 1e9, 1),
            "roofline_frac": round(alg / (res["avg_launch_us"] * 1e-6) / 1e9 / peak, 4),
            "rotating_weight_buffers": res["R"]}


def alg_bytes(M, K, N):
    """Algorithmic bytes of one W8A8 call: the weight, the activations and both scale vectors read,
    the bf16 output written."""
    return K * N + M * K + 4 * M + 4 * N + 2 * M * N


def run_ours(args):
    import torch

    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    cfg = DEFAULT
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    res = time_gemm(M, K, N, cfg["dist"], cfg["seed"], args.steps, args.warmup, device=dev, sample_clocks=(rank == 0))
    x, xs, W, ws = res.pop("inputs")
    wbytes = res["wbytes"]
    value = whole_job_gbs(world, wbytes, res["launches"], res["total_ms"])
    peak, peak_kind = _peaks()
    alg = alg_bytes(M, K, N)
    achieved = alg / (res["avg_launch_us"] * 1e-6) / 1e9
    traffic = _traffic_per_launch()
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["total_ms"] / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": DATA[cfg["dist"]],
        "config": workload_config(HEADLINE, world),
        "timing": {"rotating_weight_buffers": res["R"], "calls_per_step": res["C"],
                   "weight_bytes_per_call": wbytes, "steps": args.steps},
        "us_per_call": {"median": round(res["us_median"], 4), "p90": round(res["us_p90"], 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (copy, MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic, "alg_bytes_per_launch": alg,
                     "frac_of_8tbs_nominal": round(achieved / 8000.0, 4), "kernel": res["kernel"]},
        "gpu_launches": res["launches"],
        "e2e": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in res["e2e"].items()},
        "clocks": res["clocks"],
    }
    # The same calls launched with programmatic dependent launch (W8A8_FLAG_PDL): each call starts
    # streaming its weight while the previous call finishes, as in a chain of decode-step GEMMs.
    # Reported beside the default line, not as its value.
    import int8_weight_gemm_gb300 as lib8
    rp = time_gemm(M, K, N, cfg["dist"], cfg["seed"], min(args.steps, 300), args.warmup, device=dev,
                   want_e2e=False, flags=lib8.W8A8_FLAG_PDL)
    rp.pop("inputs")
    out["pdl"] = {"value": round(whole_job_gbs(world, wbytes, rp["launches"], rp["total_ms"]), 2), "unit": "GB/s",
                  "us_per_call": {"median": round(rp["us_median"], 4), "p90": round(rp["us_p90"], 4)},
                  "roofline_frac": round(alg / (rp["avg_launch_us"] * 1e-6) / 1e9 / peak, 4),
                  "launch": "W8A8_FLAG_PDL, same graph of rotating-weight calls"}
    del rp
    # The other decode shapes, plain and with PDL.
    out["shapes"] = []
    for name in ("down", "qkv"):
        w = WORKLOADS[name]
        entry = None
        for flags in (0, lib8.W8A8_FLAG_PDL):
            r = time_gemm(w["M"], w["K"], w["N"], w["dist"], w["seed"], min(args.steps, 300), args.warmup, device=dev,
                          want_e2e=False, flags=flags)
            r.pop("inputs")
            if flags == 0:
                entry = shape_summary(name, r, peak, world)
            else:
                entry["pdl_us_per_call"] = {"median": round(r["us_median"], 4), "p90": round(r["us_p90"], 4)}
            del r
            torch.cuda.empty_cache()
        out["shapes"].append(entry)
    # Correctness check of the timed configuration against the oracle: every row, a seeded sample of
    # whole columns (the first and last of every 64-row tile among them).
    if rank == 0:
        import oracle
        rng = np.random.default_rng(12345)
        cols = np.unique(np.concatenate([rng.choice(N, 256, replace=False), np.arange(0, N, 64), np.arange(63, N, 64)]))
        ref = oracle.w8a8_gemm(x, xs, np.ascontiguousarray(W[:, cols]), np.ascontiguousarray(ws[cols]))
        got = res["out"].cpu().view(torch.int16).numpy().view(np.uint16)[:, cols]
        out["parity"] = {"outputs_checked": int(ref.size), "columns_checked": int(len(cols)),
                         "mismatches": int(np.count_nonzero(got != ref))}
        if not args.no_q8:
            out["q8_0"] = [time_q8(T, K8, N8, flags=f) for (K8, N8) in ((4096, 320), (320, 4096)) for T in (1, 4, 6)
                           for f in (0, lib8.W8A8_FLAG_PDL)]
            # the RMS-norm variant (q8_0_gemv_rms) on the same reads
            out["q8_0"] += [time_q8(6, K8, N8, flags=f, rms=True) for (K8, N8) in ((4096, 320), (320, 4096))
                            for f in (0, lib8.W8A8_FLAG_PDL)]
        out["tensor_memory_arm"] = time_tensor_memory_arm(args, dev, peak)
        out["read_ceiling"] = time_read_ceiling(dev)
        out["mma_rates"] = time_mma_rates(dev)
        if not args.no_q8:
            out["quantisation"] = time_quantisation_rows(peak)
        out["roofline"]["frac_of_read_ceiling"] = round(achieved / out["read_ceiling"]["value"], 4)
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(M, K, N, x, xs, W, ws)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args):
    """The oracle timed on the host cores on the same metric, config and unit: every step is one
    whole call of the headline workload, its columns cut over one thread per host core.  Under
    torchrun only rank 0 runs it."""
    rank = _env_int("RANK", 0)
    if rank != 0:
        return
    import synth

    cfg = DEFAULT
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=cfg["seed"], dist=cfg["dist"])
    par = OracleOnCores(x, xs, W, ws)
    for _ in range(args.warmup):
        par.call()
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter()
        par.call()
        times.append(time.perf_counter() - a)
    total = time.perf_counter() - t0
    par.close()
    value = K * N * args.steps / total / 1e9
    times.sort()
    sample = (f"each step: one whole oracle call of M={M}, K={K}, N={N}, its columns cut over {par.threads} "
              "threads (one per host core), plain C")
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": _env_int("WORLD_SIZE", 1),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64",
        "data": DATA[cfg["dist"]],
        "config": workload_config(HEADLINE, _env_int("WORLD_SIZE", 1)),
        "us_per_call": {"median": round(statistics.median(times) * 1e6, 1), "p90": round(p90(times) * 1e6, 1)},
        "cpu_baseline": {"kind": "oracle", "cores": par.threads, "sample": sample, "value": round(value, 4),
                         "unit": "GB/s"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


def run_sweep(args):
    """Every workload family (one line each, to stdout), then exit: not the contract line."""
    import torch

    rows = []
    shapes = [(1, 512, 256, "uniform", 0), (16, 4096, 1536, "uniform", 1)]
    shapes += [(M, K, N, "uniform", 3000 + M) for (N, K) in ((2560, 4096), (4096, 2048)) for M in (1, 4, 8, 16, 32)]
    shapes += [(16, 4096, 24576, "mlp", 4), (16, 12288, 4096, "mlp", 4)]
    # 32 < M <= 128: the tensor-memory arm on the same weight shapes
    shapes += [(M, K, N, "uniform", 5000 + M) for (N, K) in ((1536, 4096), (2560, 4096), (4096, 2048))
               for M in (64, 128)]
    shapes += [(128, 4096, 24576, "mlp", 5), (128, 12288, 4096, "mlp", 5), (48, 4096, 1536, "uniform", 5048)]
    # more tile-aligned decode shapes (CTA-count rule of the automatic plan)
    shapes += [(16, 4096, 8192, "mlp", 4), (16, 4096, 12288, "mlp", 4), (16, 4096, 6144, "mlp", 4),
               (16, 14336, 4096, "mlp", 4), (1, 12288, 4096, "mlp", 4), (32, 12288, 4096, "mlp", 4),
               (32, 4096, 1536, "uniform", 1)]
    shapes += [(1, 4096, 24576, "mlp", 4), (32, 4096, 24576, "mlp", 4)]
    shapes += [(24, 4096, 2560, "uniform", 3024), (24, 2048, 4096, "uniform", 3024)]
    if args.shapes:
        shapes = [shapes[int(i)] for i in args.shapes.split(",")]
    peak, _ = _peaks()
    blocks_list = [int(b) for b in args.blocks.split(",")] if args.blocks else [0]
    flags_list = [int(f) for f in args.flags.split(",")] if args.flags else [0]
    for (M, K, N, dist, seed) in shapes:
        for blocks, flags in [(b, f) for b in blocks_list for f in flags_list]:
            import int8_weight_gemm_gb300 as lib8
            slabs = lib8.w8a8_plan(M, K, N)["slabs"]
            if blocks > slabs:
                continue
            r = time_gemm(M, K, N, dist, seed, args.steps, args.warmup, blocks=blocks, want_e2e=False, flags=flags)
            gbs = r["wbytes"] / (r["us_median"] * 1e-6) / 1e9
            row = {"M": M, "K": K, "N": N, "dist": dist, "blocks": blocks or lib8.w8a8_plan(M, K, N)["blocks"],
                   "flags": flags, "kernel": r["kernel"],
                   "tflops": round(2.0 * M * N * K / (r["us_median"] * 1e-6) / 1e12, 1),
                   "us_median": round(r["us_median"], 3), "us_p90": round(r["us_p90"], 3),
                   "weight_GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 3), "R": r["R"]}
            rows.append(row)
            print(json.dumps(row), flush=True)
            del r
            torch.cuda.empty_cache()
    if args.no_q8:
        return
    for (K8, N8) in ((4096, 320), (320, 4096)):
        for T in (1, 4, 6):
            for flags in flags_list:
                print(json.dumps(time_q8(T, K8, N8, flags=flags)), flush=True)
                print(json.dumps(time_q8(T, K8, N8, flags=flags, rms=True)), flush=True)
    for r in time_mma_rates(torch.device("cuda")):
        print(json.dumps(r), flush=True)


def run_ncu_driver(args):
    """Profiling driver (for ncu captures, not a bench line): the default workload's public-API
    calls, eagerly, on rotating packed weights (each call reads a different weight copy), then exit.
    --ncu-op q8_0 runs the Q8_0 read instead (--ncu-shape T,K,N), --ncu-op mma the tensor-pipe rate
    probe (both kinds)."""
    import torch

    import int8_weight_gemm_gb300 as lib8
    import synth

    if args.ncu_op == "mma":
        sink = torch.zeros(1, dtype=torch.int64, device="cuda")
        for _ in range(args.ncu_driver):
            for kind in (0, 1):
                lib8.w8a8_mma_rate_probe(kind, 256, sink)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_driver_calls": args.ncu_driver, "op": "mma"}))
        return
    if args.ncu_op == "q8_0":
        T, K, N = (int(v) for v in (args.ncu_shape or "6,4096,320").split(","))
        x, q, d = synth.q8_0_inputs(T, K, N, seed=7)
        xd = x.cuda()
        qs = [torch.from_numpy(q).cuda() for _ in range(8)]
        ds = [torch.from_numpy(d.view(np.int16)).cuda() for _ in range(8)]
        qws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
        for i in range(args.ncu_driver):
            lib8.q8_0_gemv(xd, qs[i % 8], ds[i % 8], qws)
        torch.cuda.synchronize()
        status = lib8.w8a8_workspace_status(qws)
        print(json.dumps({"ncu_driver_calls": args.ncu_driver, "op": "q8_0", "device_status": status}))
        if status != 0:
            sys.exit(1)
        return

    cfg = DEFAULT
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    if args.ncu_shape:
        M, K, N = (int(v) for v in args.ncu_shape.split(","))
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=cfg["seed"], dist=cfg["dist"])
    dev = torch.device("cuda")
    xd, xsd, wsd = (torch.from_numpy(a).to(dev) for a in (x, xs, ws))
    wsp = lib8.alloc_workspace(lib8.w8a8_workspace_bytes(M, K, N), dev)
    packed = lib8.w8a8_pack_weights(torch.from_numpy(W).to(dev), ws=wsp)
    packs = [packed] + [packed.clone() for _ in range(7)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for i in range(args.ncu_driver):
        lib8.w8a8_gemm(xd, xsd, packs[i % len(packs)], wsd, wsp, N, out=out)
    torch.cuda.synchronize()
    status = lib8.w8a8_workspace_status(wsp)
    print(json.dumps({"ncu_driver_calls": args.ncu_driver, "device_status": status}))
    if status != 0:
        sys.exit(1)


def build_parser():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true", help="time every workload family (extra lines)")
    ap.add_argument("--blocks", default="", help="comma list of CTA counts for --sweep (0 = auto)")
    ap.add_argument("--flags", default="", help="comma list of launch flags for --sweep (1 = PDL)")
    ap.add_argument("--shapes", default="", help="comma list of sweep shape indices (default: all)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-q8", action="store_true", help="skip the Q8_0 timings")
    ap.add_argument("--ncu-shape", default="", help="M,K,N for --ncu-driver (default: the headline shape)")
    ap.add_argument("--ncu-op", default="w8a8", choices=["w8a8", "q8_0", "mma"], help="what --ncu-driver calls")
    ap.add_argument("--ncu-driver", type=int, default=0,
                    help="profiling driver: this many eager calls of the default workload, then exit")
    return ap


def main():
    ap = build_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.ncu_driver:
        run_ncu_driver(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
