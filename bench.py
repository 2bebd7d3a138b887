#!/usr/bin/env python
"""Benchmark of the fused norm/act -> FP8 hot path on GB300.

One step = one pass of the whole path over one batch: residual add + RMSNorm
-> FP8 (vg_fused_add_rms_norm_fp8) followed by SiLU-and-mul -> FP8
(vg_silu_mul_fp8), the two fused ops that bracket an MLP block's gate-up
GEMM.  The default workload is the Llama-3-8B decode shape: T=256 tokens,
hidden 4096 with per-token dynamic scales, intermediate 14336 (the sweep's
hidden/intermediate pairing) with per-token dynamic scales.

Timing (device, CUDA events on the launching stream):
  * inputs are resident in HBM; R buffer sets (each its own copy of every
    input and output) rotate so that R * bytes >= 3 x L2 and no step reads
    data left in L2 by the previous use of its set;
  * the K timed steps are captured once into a CUDA graph (launch cost
    hidden); the timed region is one replay bracketed by a barrier and a
    torch.cuda.synchronize() on both sides; max over ranks;
  * the roofline's per-kernel duration: each op's K launches, over the same
    rotation of buffer sets, captured in a graph of their own and replayed
    right after the timed region (event nodes inside a graph would add
    microseconds per kernel);
  * clocks are sampled by nvidia-smi over a window of untimed replays of the
    same graph just before the timed one, through the per-kernel replays.
e2e repeats the step through the C ABI from pinned HOST buffers: every step
copies its inputs host->device and reads every output back device->host.
--impl reference times the fp64 CPU oracle on the host cores instead.

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "fused norm/act→FP8 GB/s & tokens/s vs ~8 TB/s HBM roofline (1 GB300)"
FALLBACK_HBM_GBS = 6800.0

# A step is a tuple of workloads run back to back on one batch.
CFG3_ACT = gen.Workload("silu_per_group128_16384x28672", "silu", 16384, 28672, gen.PER_GROUP,
                        group_size=128)
STEPS = {
    "llama3_8b_decode": (gen.CFG1, gen.CFG1_ACT),
    "llama3_70b_prefill": (gen.CFG3, CFG3_ACT),
}
# every named single-op workload is also a (one-op) step
STEPS.update({name: (w,) for name, w in gen.NAMED.items()})
DEFAULT_STEP = "llama3_8b_decode"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("vg", "reference"), default="vg")
    p.add_argument("--workload", choices=sorted(STEPS), default=DEFAULT_STEP)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="bound on the oracle's CPU-baseline sample")
    p.add_argument("--clock-window", type=float, default=1.0,
                   help="seconds of untimed replays under clock sampling before the timed one")
    p.add_argument("--tokens", type=int, default=None,
                   help="override num_tokens of every op of the step (smaller profiling captures)")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the step: time every point of the bandwidth sweep and the named "
                        "single-op configs, one JSON record per point")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


# ------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        raise SystemExit(f"WORLD_SIZE={world} but --gpus {args.gpus}")
    return rank, world, local


class Dist:
    def __init__(self, rank, world, local, backend):
        self.rank, self.world, self.local = rank, world, local
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if self.pg.get_backend() == "nccl":
                import torch
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
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
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


# ------------------------------------------------------------------ helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "norm": ["norm_activation_fp8_gb300/csrc/norm_fp8.cu", "norm_activation_fp8_gb300/csrc/common.cuh",
             "norm_activation_fp8_gb300/csrc/dyn_scale.cuh", "norm_activation_fp8_gb300/csrc/tma.cuh",
             "norm_activation_fp8_gb300/csrc/vg_fused.cu"],
    "silu": ["norm_activation_fp8_gb300/csrc/silu_fp8.cu", "norm_activation_fp8_gb300/csrc/common.cuh",
             "norm_activation_fp8_gb300/csrc/vg_fused.cu"],
}


def kernel_source_hash(op: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[op]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(op: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload (profiles/<workload>.md), or None if there is none or the
    kernel's source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(op):
        return None
    return int(m_bytes.group(1))


def step_bytes(step):
    return sum(w.algorithmic_bytes() for w in step)


def step_tokens(step):
    return step[0].T


# -------------------------------------------------------------- GPU arm

class DeviceSet:
    """One copy of every input and output of a step, resident on the GPU."""

    def __init__(self, torch, step, host, weights, dev):
        self.ops = []
        for w, h in zip(step, host):
            if w.op == "norm":
                x = torch.from_numpy(h["x"].view(np.int16)).to(dev)
                res = torch.from_numpy(h["residual"].view(np.int16)).to(dev)
                q = torch.empty((w.T, w.n), dtype=torch.uint8, device=dev)
                scale = self._scale(torch, w, dev)
                self.ops.append(dict(w=w, q=q, res=res, scale=scale, x=x, weight=weights[w.name]))
            else:
                gu = torch.from_numpy(h["gate_up"].view(np.int16)).to(dev)
                q = torch.empty((w.T, w.n), dtype=torch.uint8, device=dev)
                scale = self._scale(torch, w, dev)
                self.ops.append(dict(w=w, q=q, scale=scale, gate_up=gu))

    @staticmethod
    def _scale(torch, w, dev):
        if w.mode == gen.STATIC:
            return torch.full((1,), w.static_scale, dtype=torch.float32, device=dev)
        if w.mode == gen.PER_TOKEN:
            return torch.empty((w.T,), dtype=torch.float32, device=dev)
        return torch.empty((w.T, w.n // w.group_size), dtype=torch.float32, device=dev)


def launch(vg, op):
    w = op["w"]
    if w.op == "norm":
        vg.vg_fused_add_rms_norm_fp8(op["q"], op["res"], op["scale"], op["x"], op["res"],
                                     op["weight"], w.eps, w.mode, w.group_size)
    else:
        vg.vg_silu_mul_fp8(op["q"], op["scale"], op["gate_up"], w.mode, w.group_size)


def run_gpu(args, dist):
    import torch
    import norm_activation_fp8_gb300 as vg
    from norm_activation_fp8_gb300 import build as vg_build

    dev = torch.device("cuda", dist.local)
    if not os.path.exists(vg_build.LIB_PATH):
        vg_build.build()
    vg.load()
    step = select_step(args)
    nbytes = step_bytes(step)
    host = [w.inputs() for w in step]
    weights = {w.name: torch.from_numpy(h["weight"].view(np.int16)).to(dev)
               for w, h in zip(step, host) if w.op == "norm"}
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    resident = nbytes  # every set holds one copy of every input and output
    n_sets = max(2, math.ceil(3 * l2 / max(1, resident)))
    n_sets = min(n_sets, max(2, int(20e9 // max(1, resident))))
    sets = [DeviceSet(torch, step, host, weights, dev) for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=dev)

    # warm-up: W eager steps
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            for op in sets[k % n_sets].ops:
                launch(vg, op)
    torch.cuda.synchronize()

    # The K timed steps captured once into one graph (hides launch cost).
    nk = len(step)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(args.steps):
            for op in sets[(args.warmup + k) % n_sets].ops:
                launch(vg, op)
    # Per-kernel graphs: the same K launches of one op, for its duration.
    op_graphs = []
    for i in range(nk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(args.steps):
                launch(vg, sets[(args.warmup + k) % n_sets].ops[i])
        op_graphs.append(g)
    torch.cuda.synchronize()

    clocks = ClockSampler(dist.local)
    clocks.start()
    t_end = time.time() + args.clock_window
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            graph.replay()
            stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist.barrier()
    with torch.cuda.stream(stream):
        start.record()
        graph.replay()
        end.record()
    torch.cuda.synchronize()
    dist.barrier()
    ms_local = start.elapsed_time(end)
    ms = dist.max(ms_local)

    per_kernel = {}
    for w, g in zip(step, op_graphs):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s0.record()
            g.replay()
            s1.record()
        torch.cuda.synchronize()
        per_kernel[w.name] = s0.elapsed_time(s1) / args.steps
    clk = clocks.stop()

    total_bytes = nbytes * args.steps * dist.world
    value = total_bytes / (ms * 1e-3) / 1e9
    tokens_s = step_tokens(step) * args.steps * dist.world / (ms * 1e-3)

    dom = max(step, key=lambda w: per_kernel[w.name])
    dom_ms = per_kernel[dom.name]
    peak, peak_kind = measured_peak()
    achieved = dom.algorithmic_bytes() / (dom_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                "kernel": dom.name, "kernel_ms": round(dom_ms, 6),
                "traffic": profiled_traffic(dom.op, dom.name)}

    e2e = None if args.no_e2e else run_e2e(torch, vg, step, host, weights, dev, stream, args,
                                          dist)
    cpu = None
    if not args.no_cpu_baseline and dist.rank == 0 and dist.world == 1:
        cpu = run_cpu_baseline(step, host, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "tokens_per_s": round(tokens_s, 1),
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": args.workload if args.tokens is None else f"{args.workload}@T{args.tokens}",
            "ops": [describe(w) for w in step],
            "bytes_per_step": nbytes,
            "l2": f"inputs > L2: {n_sets} rotating buffer sets x {resident / 2**20:.1f} MiB "
                  f"(>= 3x L2 of {l2 / 2**20:.0f} MiB)",
            "timing": "K steps in one CUDA graph replay, CUDA events on the launching stream",
            "per_kernel_ms": {k: round(v, 6) for k, v in per_kernel.items()},
            "per_kernel_timing": "each op's K launches (same buffer rotation) in its own graph, "
                                 "replayed right after the timed region",
            "parallelism": f"replicas x{dist.world} (rows sharded, no collective)",
            "gpu": props.name, "sms": props.multi_processor_count,
            "torch": torch.__version__,
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": len(step) * args.steps,
        "clocks": clk,
    }
    return line


def select_step(args):
    import dataclasses
    step = STEPS[args.workload]
    if args.tokens is not None:
        step = tuple(dataclasses.replace(w, T=args.tokens, name=f"{w.name}@T{args.tokens}")
                     for w in step)
    return step


def describe(w):
    return {"name": w.name, "op": w.op, "T": w.T, "n": w.n,
            "mode": gen.MODE_NAMES[w.mode], "group_size": w.group_size if w.mode == gen.PER_GROUP else None,
            "bytes": w.algorithmic_bytes()}


def run_e2e(torch, vg, step, host, weights, dev, stream, args, dist):
    """The step through the C ABI from pinned host buffers: H2D of every
    input, the two calls, D2H of every output, each step."""
    dset = DeviceSet(torch, step, host, weights, dev)
    pins_in, pins_out = [], []
    h2d = d2h = 0
    for op, h in zip(dset.ops, host):
        if op["w"].op == "norm":
            srcs = [(torch.from_numpy(h["x"].view(np.int16)).pin_memory(), op["x"]),
                    (torch.from_numpy(h["residual"].view(np.int16)).pin_memory(), op["res"])]
            dsts = [op["q"], op["res"]]
        else:
            srcs = [(torch.from_numpy(h["gate_up"].view(np.int16)).pin_memory(), op["gate_up"])]
            dsts = [op["q"]]
        if op["w"].mode != gen.STATIC:
            dsts.append(op["scale"])
        pins_in.append(srcs)
        outs = [(d, torch.empty(d.shape, dtype=d.dtype, pin_memory=True)) for d in dsts]
        pins_out.append(outs)
        h2d += sum(s.numel() * s.element_size() for s, _ in srcs)
        d2h += sum(d.numel() * d.element_size() for d, _ in outs)

    def one_step():
        for op, srcs, outs in zip(dset.ops, pins_in, pins_out):
            for s, d in srcs:
                d.copy_(s, non_blocking=True)
            launch(vg, op)
            for d, hbuf in outs:
                hbuf.copy_(d, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize()
    dist.barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s0.record()
        for _ in range(args.steps):
            one_step()
        s1.record()
    torch.cuda.synchronize()
    dist.barrier()
    ms = dist.max(s0.elapsed_time(s1))
    value = step_bytes(step) * args.steps * dist.world / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms / args.steps, 6)}


# -------------------------------------------------------------- CPU oracle

def oracle_step_runner(step, host, threads):
    """Runs one step with the oracle, its rows split over `threads` host
    threads (the oracle's C code releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    orc = oracle.default()
    pool = ThreadPoolExecutor(threads)

    def blocks(T):
        per = max(1, (T + threads - 1) // threads)
        return [(r, min(T, r + per)) for r in range(0, T, per)]

    def one():
        futs = []
        for w, h in zip(step, host):
            for r0, r1 in blocks(w.T):
                if w.op == "norm":
                    futs.append(pool.submit(orc.fused_add_rms_norm_fp8, h["x"][r0:r1],
                                            h["residual"][r0:r1], h["weight"], w.eps, w.mode,
                                            w.group_size, w.static_scale, False))
                else:
                    futs.append(pool.submit(orc.silu_mul_fp8, h["gate_up"][r0:r1], w.mode,
                                            w.group_size, w.static_scale, False))
        for f in futs:
            f.result()

    return one, pool


def run_cpu_baseline(step, host, seconds):
    threads = os.cpu_count() or 1
    one, pool = oracle_step_runner(step, host, threads)
    one()  # builds/loads the oracle library, warms caches
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            break
    pool.shutdown()
    value = step_bytes(step) * n / el / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} whole steps of this workload ({el:.1f} s of CPU work), rows split "
                      f"over {threads} threads",
            "tokens_per_s": round(step_tokens(step) * n / el, 2)}


def run_reference(args, dist):
    """The fp64 CPU oracle as the reference arm, on this workload."""
    if dist.rank != 0:
        return None
    step = select_step(args)
    host = [w.inputs() for w in step]
    threads = os.cpu_count() or 1
    one, pool = oracle_step_runner(step, host, threads)
    # each step is one whole step of the workload; bounded by the sample rule
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    pool.shutdown()
    value = step_bytes(step) * args.steps / el / 1e9
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{args.steps} whole steps of this workload, rows split over {threads} threads"}
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "tokens_per_s": round(step_tokens(step) * args.steps / el, 2),
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "ops": [describe(w) for w in step],
                   "bytes_per_step": step_bytes(step)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_sweep(args):
    """Per-point kernel throughput: K launches of one op (rotating buffer sets
    larger than 3x L2) in one CUDA graph, timed with CUDA events."""
    import torch
    import norm_activation_fp8_gb300 as vg
    from norm_activation_fp8_gb300 import build as vg_build
    if not os.path.exists(vg_build.LIB_PATH):
        vg_build.build()
    vg.load()
    dev = torch.device("cuda", 0)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132 * 2 ** 20)
    peak, peak_kind = measured_peak()
    stream = torch.cuda.Stream(device=dev)
    points = list(gen.NAMED.values()) + gen.sweep()
    cache = {}
    for w in points:
        key = (w.op, w.T, w.n, w.x_dist)
        if key not in cache:
            cache.clear()
            cache[key] = w.inputs()
        host = cache[key]
        nbytes = w.algorithmic_bytes()
        n_sets = max(2, min(64, math.ceil(3 * l2 / nbytes)))
        weights = {w.name: torch.from_numpy(host["weight"].view(np.int16)).to(dev)} if w.op == "norm" else {}
        sets = [DeviceSet(torch, (w,), [host], weights, dev) for _ in range(n_sets)]
        k_launch = max(args.steps, n_sets)
        with torch.cuda.stream(stream):
            for k in range(args.warmup):
                launch(vg, sets[k % n_sets].ops[0])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(k_launch):
                launch(vg, sets[k % n_sets].ops[0])
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            s0.record()
            g.replay()
            s1.record()
        torch.cuda.synchronize()
        us = s0.elapsed_time(s1) * 1e3 / k_launch
        gbs = nbytes / (us * 1e-6) / 1e9
        print(json.dumps({"point": w.name, "op": w.op, "T": w.T, "n": w.n,
                          "mode": gen.MODE_NAMES[w.mode], "bytes": nbytes, "us": round(us, 3),
                          "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                          "peak": peak, "peak_source": peak_kind,
                          "tokens_per_s": round(w.T / (us * 1e-6), 1)}), flush=True)
        del sets, g
        torch.cuda.empty_cache()
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_setup(args)
    if args.sweep:
        return run_sweep(args) if rank == 0 else 0
    if args.impl == "reference":
        if rank != 0:
            return 0
        line = run_reference(args, Dist(0, 1, 0, "gloo"))
        print(json.dumps(line), flush=True)
        return 0
    import torch
    torch.cuda.set_device(local)
    dist = Dist(rank, world, local, "nccl")
    try:
        line = run_gpu(args, dist)
    finally:
        dist.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
