#!/usr/bin/env python
"""Benchmark of the fused norm/act -> FP8 hot path on GB300.

One step = one pass of the whole path over one batch: residual add + RMSNorm
-> FP8 (vg_fused_add_rms_norm_fp8) followed by SiLU-and-mul -> FP8
(vg_silu_mul_fp8), the two fused ops that bracket an MLP block's gate-up
GEMM.  The default workload is the 70B-shaped prefill: T = 16384 tokens,
hidden 8192 (Student-t(3) x with 0.1 % outliers) with per-group-128 dynamic
scales, then intermediate 28672 (Llama-3-70B's) with per-group-128 dynamic
scales.  The Llama-3-8B decode step (T = 256, hidden 4096 / intermediate
14336, per-token scales) is timed after it and reported under `decode_step`.

Timing (device, CUDA events on the launching stream):
  * inputs are resident in HBM; R buffer sets (each its own copy of every
    input and output) rotate so that R * bytes >= 3 x L2 and no step reads
    data left in L2 by the previous use of its set;
  * the K timed steps are captured once into a CUDA graph (launch cost
    hidden); the timed region is one replay bracketed by a barrier and a
    torch.cuda.synchronize() on both sides; max over ranks;
  * the roofline's per-kernel duration: each op's K launches, over the same
    rotation of buffer sets, captured in a graph of their own, replayed once
    untimed and then timed over several replays (median, p10, p90);
  * clocks are sampled by nvidia-smi over a window of untimed replays of the
    same graph just before the timed one, through the per-kernel replays.
e2e repeats the step through the C ABI from pinned HOST buffers: every step
copies its inputs host->device and reads every output back device->host,
pipelined over three streams as a serving loop would overlap them.
--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded row sample of the same workload.

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
    CFG3_ACT.name: (CFG3_ACT,),
}
# every named single-op workload and every sweep point is also a (one-op) step
STEPS.update({name: (w,) for name, w in gen.NAMED.items()})
STEPS.update({w.name: (w,) for w in gen.sweep()})
STEPS.update({w.name: (w,) for w in gen.mla_workloads()})
STEPS.update({w.name: (w,) for w in gen.pad_workloads()})
STEPS.update({w.name: (w,) for w in gen.qk_workloads()})
STEPS.update({w.name: (w,) for w in gen.nvfp4_workloads()})
STEPS.update({w.name: (w,) for w in gen.group_option_workloads()})
DEFAULT_STEP = "llama3_70b_prefill"
DECODE_STEP = "llama3_8b_decode"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("vg", "reference"), default="vg")
    p.add_argument("--workload", choices=sorted(STEPS), default=DEFAULT_STEP)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-large-token", action="store_true",
                   help="skip timing the large-token single-op configs after the step")
    p.add_argument("--no-decode", action="store_true",
                   help="skip timing the decode step after the default (prefill) step")
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
    p.add_argument("--sweep-filter", default=None,
                   help="with --sweep: only points whose name contains one of these "
                        "comma-separated substrings")
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


def replay_spread(torch, graph, stream, steps, replays=10):
    """Median, p10 and p90 of ms per step over `replays` further replays of
    a graph of `steps` steps, each bracketed by CUDA events (context for the
    single timed replay)."""
    per = []
    for _ in range(replays):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            graph.replay()
            b.record()
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) / steps)
    q = np.percentile(per, [10, 50, 90])
    return {"p10": round(float(q[0]), 6), "median": round(float(q[1]), 6),
            "p90": round(float(q[2]), 6), "replays": replays}


def whole_job(dist, bytes_per_step, tokens_per_step, steps, ms_local):
    """Weak scaling over replicas: every rank runs the same step on its own
    copy of the data, the job's time is the slowest rank's and its work the
    sum over ranks.  Returns (ms, GB/s, tokens/s) of the whole job."""
    ms = dist.max(ms_local)
    secs = ms * 1e-3
    return (ms, bytes_per_step * steps * dist.world / secs / 1e9,
            tokens_per_step * steps * dist.world / secs)


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


_CSRC = "norm_activation_fp8_gb300/csrc/"
# The translation unit of each op's kernels; the launch plans of every op
# live in vg_fused.cu.
KERNEL_UNITS = {"norm": "norm_fp8.cu", "pad": "norm_fp8.cu", "norm4": "norm_fp8.cu",
                "silu": "silu_fp8.cu", "silu4": "silu_fp8.cu", "mla": "mla_norm.cu",
                "qk": "qk_norm_rope.cu"}


def kernel_sources(op: str):
    """The files an op's kernel and launch plan are built from: its
    translation unit and vg_fused.cu, with every header they include,
    transitively (quoted includes, resolved in csrc/ and include/)."""
    dirs = [os.path.join(ROOT, _CSRC), os.path.join(ROOT, "include")]
    todo = [os.path.join(ROOT, _CSRC, KERNEL_UNITS[op]), os.path.join(ROOT, _CSRC, "vg_fused.cu")]
    seen = []
    while todo:
        path = todo.pop(0)
        if path in seen:
            continue
        seen.append(path)
        with open(path) as f:
            for name in re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), re.M):
                for d in dirs:
                    cand = os.path.join(d, name)
                    if os.path.exists(cand):
                        todo.append(cand)
                        break
    return [os.path.relpath(p, ROOT) for p in seen]


def kernel_source_hash(op: str) -> str:
    h = hashlib.sha256()
    for rel in kernel_sources(op):
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
            elif w.op == "norm4":
                x = torch.from_numpy(h["x"].view(np.int16)).to(dev)
                res = torch.from_numpy(h["residual"].view(np.int16)).to(dev)
                q4 = torch.empty((w.T, w.n // 2), dtype=torch.uint8, device=dev)
                sf = torch.empty((w.T, w.n // 16), dtype=torch.uint8, device=dev)
                gs = torch.full((1,), w.static_scale, dtype=torch.float32, device=dev)
                self.ops.append(dict(w=w, q4=q4, sf=sf, gs=gs, res=res, x=x,
                                     weight=weights[w.name]))
            elif w.op == "silu4":
                gu = torch.from_numpy(h["gate_up"].view(np.int16)).to(dev)
                q4 = torch.empty((w.T, w.n // 2), dtype=torch.uint8, device=dev)
                sf = torch.empty((w.T, w.n // 16), dtype=torch.uint8, device=dev)
                gs = torch.full((1,), w.static_scale, dtype=torch.float32, device=dev)
                self.ops.append(dict(w=w, q4=q4, sf=sf, gs=gs, gate_up=gu))
            elif w.op == "qk":
                qkv = torch.from_numpy(h["qkv"].view(np.int16)).to(dev)
                pos = torch.from_numpy(h["positions"]).to(dev)
                qw, kw, cache = weights[w.name]
                self.ops.append(dict(w=w, qkv=qkv, pos=pos, q_weight=qw, k_weight=kw, cache=cache))
            elif w.op == "pad":
                x = torch.from_numpy(h["x"].view(np.int16)).to(dev)
                res = torch.from_numpy(h["residual"].view(np.int16)).to(dev)
                out = torch.empty((w.T, w.n2), dtype=torch.int16, device=dev)
                self.ops.append(dict(w=w, out=out, res=res, x=x, weight=weights[w.name]))
            elif w.op == "mla":
                # q_c and kv_c as column slices of one projected tensor, as in the model
                proj = np.zeros((w.T, w.n + w.n2 + gen.MLA_ROPE), np.uint16)
                proj[:, :w.n] = h["q_c"]
                proj[:, w.n:w.n + w.n2] = h["kv_c"]
                pt = torch.from_numpy(proj.view(np.int16)).to(dev)
                fp8 = w.mode == gen.PER_TOKEN
                q = torch.empty((w.T, w.n), dtype=torch.uint8 if fp8 else torch.int16, device=dev)
                scale = torch.empty((w.T,), dtype=torch.float32, device=dev) if fp8 else None
                kv = torch.empty((w.T, w.n2), dtype=torch.int16, device=dev)
                qw, kw = weights[w.name]
                self.ops.append(dict(w=w, q=q, scale=scale, kv=kv, q_c=pt[:, :w.n],
                                     kv_c=pt[:, w.n:w.n + w.n2], q_weight=qw, kv_weight=kw))
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
        if w.flags & gen.COL_MAJOR:
            return torch.empty((w.n // w.group_size, (w.T + 3) // 4 * 4), dtype=torch.float32,
                               device=dev)
        return torch.empty((w.T, w.n // w.group_size), dtype=torch.float32, device=dev)


def device_weights(torch, step, host, dev):
    """Each op's weights on the device, shared by all buffer sets."""
    out = {}
    for w, h in zip(step, host):
        if w.op in ("norm", "pad", "norm4"):
            out[w.name] = torch.from_numpy(h["weight"].view(np.int16)).to(dev)
        elif w.op == "mla":
            out[w.name] = tuple(torch.from_numpy(h[k].view(np.int16)).to(dev)
                                for k in ("q_weight", "kv_weight"))
        elif w.op == "qk":  # the weights and the cos/sin cache, model constants
            out[w.name] = (torch.from_numpy(h["q_weight"].view(np.int16)).to(dev),
                           torch.from_numpy(h["k_weight"].view(np.int16)).to(dev),
                           torch.from_numpy(h["cos_sin_cache"]).to(dev))
    return out


def launch(vg, op):
    w = op["w"]
    if w.op == "norm":
        vg.vg_fused_add_rms_norm_fp8(op["q"], op["res"], op["scale"], op["x"], op["res"],
                                     op["weight"], w.eps, w.mode | w.flags, w.group_size)
    elif w.op == "pad":
        vg.vg_fused_add_rms_norm_pad(op["out"], op["res"], op["x"], op["res"], op["weight"], w.eps)
    elif w.op == "norm4":
        vg.vg_fused_add_rms_norm_nvfp4(op["q4"], op["sf"], op["res"], op["x"], op["res"],
                                       op["weight"], op["gs"], w.eps)
    elif w.op == "silu4":
        vg.vg_silu_mul_nvfp4(op["q4"], op["sf"], op["gate_up"], op["gs"])
    elif w.op == "qk":
        vg.vg_fused_qk_norm_rope(op["qkv"], op["q_weight"], op["k_weight"], op["cache"], op["pos"],
                                 w.hq, w.hkv, w.n, w.eps, w.mode == 1)
    elif w.op == "mla":
        if w.mode == gen.PER_TOKEN:
            vg.vg_fused_mla_dual_rms_norm_per_token_quant(op["q"], op["scale"], op["kv"], op["q_c"],
                                                          op["q_weight"], op["kv_c"],
                                                          op["kv_weight"], w.eps, w.eps)
        else:
            vg.vg_fused_mla_dual_rms_norm(op["q"], op["kv"], op["q_c"], op["q_weight"], op["kv_c"],
                                          op["kv_weight"], w.eps, w.eps)
    else:
        vg.vg_silu_mul_fp8(op["q"], op["scale"], op["gate_up"], w.mode | w.flags, w.group_size)


def op_spread(torch, graph, stream, launches, replays=7):
    """Duration per launch of a graph of `launches` launches of one op: one
    untimed replay (the graph's first replay uploads it), then `replays`
    timed replays; the median is the kernel's duration, p10 / p90 its spread."""
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    return replay_spread(torch, graph, stream, launches, replays=replays)


def time_step(torch, vg, step, host, dev, stream, args, dist, l2, clocks=None):
    """Times K steps of `step` as one CUDA graph replay over rotating buffer
    sets (inputs > 3x L2), then each op alone in a graph of its own.  With
    `clocks`, nvidia-smi samples a window of untimed replays before the timed
    one and the per-op replays after it."""
    nbytes = step_bytes(step)
    weights = device_weights(torch, step, host, dev)
    resident = nbytes  # every set holds one copy of every input and output
    n_sets = max(2, math.ceil(3 * l2 / max(1, resident)))
    n_sets = min(n_sets, max(2, int(20e9 // max(1, resident))))
    sets = [DeviceSet(torch, step, host, weights, dev) for _ in range(n_sets)]

    # warm-up: W eager steps
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            for op in sets[k % n_sets].ops:
                launch(vg, op)
    torch.cuda.synchronize()

    # The K timed steps captured once into one graph (hides launch cost).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(args.steps):
            for op in sets[(args.warmup + k) % n_sets].ops:
                launch(vg, op)
    # Per-op graphs: the same K launches of one op, for its duration.
    op_graphs = []
    for i in range(len(step)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(args.steps):
                launch(vg, sets[(args.warmup + k) % n_sets].ops[i])
        op_graphs.append(g)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):  # upload the graph: its first replay is not timed
        graph.replay()
    torch.cuda.synchronize()
    if clocks is not None:
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
    per_kernel = {w.name: op_spread(torch, g, stream, args.steps) for w, g in zip(step, op_graphs)}
    spread = replay_spread(torch, graph, stream, args.steps)
    clk = clocks.stop() if clocks is not None else None
    del graph, op_graphs, sets
    torch.cuda.empty_cache()
    return dict(ms_local=ms_local, per_kernel=per_kernel, spread=spread, n_sets=n_sets,
                resident=resident, clocks=clk)


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
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    stream = torch.cuda.Stream(device=dev)

    t = time_step(torch, vg, step, host, dev, stream, args, dist, l2,
                  clocks=ClockSampler(dist.local))
    ms, value, tokens_s = whole_job(dist, nbytes, step_tokens(step), args.steps, t["ms_local"])
    per_kernel_ms = {k: v["median"] for k, v in t["per_kernel"].items()}

    dom = max(step, key=lambda w: per_kernel_ms[w.name])
    dom_ms = per_kernel_ms[dom.name]
    peak, peak_kind = measured_peak()
    achieved = dom.algorithmic_bytes() / (dom_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                "kernel": dom.name, "kernel_ms": round(dom_ms, 6),
                "kernel_ms_spread": t["per_kernel"][dom.name],
                "algorithmic_bytes_per_launch": dom.algorithmic_bytes(),
                "traffic": profiled_traffic(dom.op, dom.name)}

    weights = device_weights(torch, step, host, dev)
    e2e = None if args.no_e2e else run_e2e(torch, vg, step, host, weights, dev, stream, args,
                                          dist)
    del weights
    torch.cuda.empty_cache()
    cpu = None
    if not args.no_cpu_baseline and dist.rank == 0 and dist.world == 1:
        cpu = run_cpu_baseline(step, host, args.cpu_seconds)
    del host
    decode = None
    if args.workload == DEFAULT_STEP and args.tokens is None and not args.no_decode:
        decode = run_decode_step(torch, vg, dev, stream, args, dist, l2)
    large = None
    if not args.no_large_token and dist.rank == 0 and args.tokens is None:
        large = run_large_token(torch, vg, dev, stream, args, l2)

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
            "l2": f"inputs > L2: {t['n_sets']} rotating buffer sets x "
                  f"{t['resident'] / 2**20:.1f} MiB (>= 3x L2 of {l2 / 2**20:.0f} MiB)",
            "timing": "K steps in one CUDA graph replay, CUDA events on the launching stream",
            "per_kernel_ms": per_kernel_ms,
            "per_kernel_ms_spread": t["per_kernel"],
            "per_kernel_timing": "each op's K launches (same buffer rotation) in its own graph: "
                                 "one untimed replay, then the median of 7 timed replays",
            "per_kernel_sum_ms": round(sum(per_kernel_ms.values()), 6),
            "ms_per_step_spread": t["spread"],
            "parallelism": f"replicas x{dist.world} (rows sharded, no collective)",
            "gpu": props.name, "sms": props.multi_processor_count,
            "torch": torch.__version__,
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": len(step) * args.steps,
        "clocks": t["clocks"],
        "decode_step": decode,
        "large_token": large,
    }
    return line


def run_decode_step(torch, vg, dev, stream, args, dist, l2):
    """The Llama-3-8B decode step (norm per-token 256 x 4096, SiLU per-token
    256 x 14336), timed like the main step, reported beside it."""
    step = STEPS[DECODE_STEP]
    host = [w.inputs() for w in step]
    t = time_step(torch, vg, step, host, dev, stream, args, dist, l2)
    ms = t["ms_local"] / args.steps
    nbytes = step_bytes(step)
    peak, _ = measured_peak()
    per = {k: round(v["median"] * 1e3, 3) for k, v in t["per_kernel"].items()}
    return {"workload": DECODE_STEP, "ops": [describe(w) for w in step], "bytes_per_step": nbytes,
            "us_per_step": round(ms * 1e3, 3), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "tokens_per_s": round(step_tokens(step) / (ms * 1e-3), 1),
            "us_per_step_spread": {k: (round(v * 1e3, 3) if k != "replays" else v)
                                   for k, v in t["spread"].items()},
            "per_kernel_us": per,
            "per_kernel_frac": {w.name: round(w.algorithmic_bytes() / (per[w.name] * 1e-6) / 1e9
                                              / peak, 4) for w in step},
            "l2": f"{t['n_sets']} rotating buffer sets (>= 3x L2)"}


def select_step(args):
    import dataclasses
    step = STEPS[args.workload]
    if args.tokens is not None:
        step = tuple(dataclasses.replace(w, T=args.tokens, name=f"{w.name}@T{args.tokens}")
                     for w in step)
    return step


def mode_name(w):
    if w.op == "qk":
        return "neox" if w.mode == 1 else "gptj"
    if w.op == "pad":
        return f"bf16_padded_to_{w.n2}"
    if w.op == "mla":
        return "q_fp8_per_token" if w.mode == gen.PER_TOKEN else "bf16"
    if w.op in ("norm4", "silu4"):
        return f"nvfp4_gs{w.static_scale:g}"
    opts = "".join(f"_{n}" for f, n in ((gen.UE8M0, "ue8m0"), (gen.COL_MAJOR, "colmajor"))
                   if w.flags & f)
    return gen.MODE_NAMES[w.mode] + opts


def describe(w):
    d = {"name": w.name, "op": w.op, "T": w.T, "n": w.n, "mode": mode_name(w),
         "group_size": w.group_size if w.mode == gen.PER_GROUP and w.op != "mla" else None,
         "bytes": w.algorithmic_bytes()}
    if w.op in ("mla", "pad"):
        d["n2"] = w.n2
    if w.op == "qk":
        d.update(q_heads=w.hq, kv_heads=w.hkv, max_pos=w.max_pos)
    return d


class PackedSet:
    r"""One step's device tensors laid out in a single buffer so that the
    step's inputs are one contiguous span and its outputs another:

        [ x | gate_up | residual | q_norm | scale_norm | q_act | scale_act ]
          \______ inputs (host->device) ____/
                             \______________ outputs (device->host) ______/

    The residual, updated in place, ends the input span and starts the
    output span.  Every tensor starts on a 256-byte boundary."""

    def __init__(self, torch, step, host, weights, dev):
        norm = next(w for w in step if w.op == "norm")
        act = next(w for w in step if w.op == "silu")
        self.norm_w, self.act_w = norm, act
        parts = [("x", norm.T * norm.n * 2), ("gate_up", act.T * 2 * act.n * 2),
                 ("res", norm.T * norm.n * 2), ("q_norm", norm.T * norm.n),
                 ("s_norm", 4 * self._scales(norm)), ("q_act", act.T * act.n),
                 ("s_act", 4 * self._scales(act))]
        off, self.off = 0, {}
        for name, nb in parts:
            self.off[name] = (off, nb)
            off += (nb + 255) // 256 * 256
        self.total = off
        self.dev_buf = torch.empty(off, dtype=torch.uint8, device=dev)
        self.in_span = (self.off["x"][0], self.off["res"][0] + self.off["res"][1])
        self.out_span = (self.off["res"][0], self.off["s_act"][0] + self.off["s_act"][1])
        v = self.view
        self.ops = [
            dict(w=norm, x=v(torch, "x", torch.int16, (norm.T, norm.n)),
                 res=v(torch, "res", torch.int16, (norm.T, norm.n)),
                 q=v(torch, "q_norm", torch.uint8, (norm.T, norm.n)),
                 scale=v(torch, "s_norm", torch.float32, (self._scales(norm),)),
                 weight=weights[norm.name]),
            dict(w=act, gate_up=v(torch, "gate_up", torch.int16, (act.T, 2 * act.n)),
                 q=v(torch, "q_act", torch.uint8, (act.T, act.n)),
                 scale=v(torch, "s_act", torch.float32, (self._scales(act),))),
        ]
        for op in self.ops:
            if op["w"].mode == gen.STATIC:
                op["scale"].fill_(op["w"].static_scale)

    @staticmethod
    def _scales(w):
        return {gen.STATIC: 1, gen.PER_TOKEN: w.T}.get(w.mode, w.T * (w.n // w.group_size))

    def view(self, torch, name, dtype, shape):
        o, nb = self.off[name]
        return self.dev_buf[o:o + nb].view(dtype).view(shape)

    def host_inputs(self, torch, host):
        """Pinned host image of the input span, filled with the step's inputs."""
        lo, hi = self.in_span
        img = torch.zeros(hi - lo, dtype=torch.uint8, pin_memory=True)
        hn = next(h for w, h in zip((self.norm_w, self.act_w), host) if "x" in h)
        ha = next(h for h in host if "gate_up" in h)
        for name, arr in (("x", hn["x"]), ("gate_up", ha["gate_up"]), ("res", hn["residual"])):
            o, nb = self.off[name]
            img[o - lo:o - lo + nb].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
        return img


def run_e2e(torch, vg, step, host, weights, dev, stream, args, dist, ring=4):
    """The step through the C ABI from pinned host buffers, pipelined the
    way a serving loop would run it: every step uploads all its inputs
    (one host->device copy of the input span, stream 1), runs the two calls
    (stream 2) and reads every output back (one device->host copy of the
    output span, stream 3).  A ring of `ring` device buffer sets lets step
    k+1 upload and step k-1 download while step k computes; events order
    each set's reuse.  (Measured on GB300 for the 70B prefill step: either
    ~12.6 ms a step or 16-18 ms, from run to run, whatever the ring depth;
    the same copies alone, both directions at once, take 12.4 ms.)"""
    if sorted(w.op for w in step) != ["norm", "silu"]:
        return None
    sets = [PackedSet(torch, step, host, weights, dev) for _ in range(ring)]
    h_in = sets[0].host_inputs(torch, host)
    lo_o, hi_o = sets[0].out_span
    h_out = [torch.empty(hi_o - lo_o, dtype=torch.uint8, pin_memory=True) for _ in range(ring)]
    h2d, d2h = h_in.numel(), hi_o - lo_o
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def run(nsteps):
        freed = [None] * ring
        for k in range(nsteps):
            b = k % ring
            ps = sets[b]
            up, done, fr = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if freed[b] is not None:
                    s_in.wait_event(freed[b])
                lo, hi = ps.in_span
                ps.dev_buf[lo:hi].copy_(h_in, non_blocking=True)
                up.record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(up)
                for op in ps.ops:
                    launch(vg, op)
                done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                h_out[b].copy_(ps.dev_buf[lo_o:hi_o], non_blocking=True)
                fr.record(s_out)
            freed[b] = fr

    run(args.warmup)
    torch.cuda.synchronize()
    dist.barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(s_in)
    with torch.cuda.stream(s_out):
        s_out.wait_event(s0)
    run(args.steps)
    s1.record(s_out)
    torch.cuda.synchronize()
    dist.barrier()
    ms = dist.max(s0.elapsed_time(s1))
    # self-check of the packing: the last downloaded outputs equal a fresh,
    # unpacked run of the same inputs
    ref = DeviceSet(torch, step, host, weights, dev)
    with torch.cuda.stream(stream):
        for op in ref.ops:
            launch(vg, op)
    torch.cuda.synchronize()
    last = h_out[(args.steps - 1) % ring]
    for name, op in (("q_norm", ref.ops[0] if ref.ops[0]["w"].op == "norm" else ref.ops[1]),
                     ("q_act", ref.ops[0] if ref.ops[0]["w"].op == "silu" else ref.ops[1])):
        o, nb = sets[0].off[name]
        got = last[o - lo_o:o - lo_o + nb]
        if not torch.equal(got, op["q"].reshape(-1).cpu()):
            raise RuntimeError(f"e2e output span check failed for {name}")
    value = step_bytes(step) * args.steps * dist.world / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms / args.steps, 6),
            "pipeline": f"{ring}-deep ring; per step one host->device copy of the input span, "
                        "the two calls, one device->host copy of the output span, on three streams"}


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
                                            h["residual"][r0:r1], h["weight"], w.eps,
                                            w.mode | w.flags,
                                            w.group_size, w.static_scale, False))
                elif w.op == "qk":
                    futs.append(pool.submit(orc.qk_norm_rope, h["qkv"][r0:r1], h["q_weight"],
                                            h["k_weight"], h["cos_sin_cache"],
                                            h["positions"][r0:r1], w.hq, w.hkv, w.n, w.eps,
                                            w.mode == 1, False))
                elif w.op == "norm4":
                    futs.append(pool.submit(orc.fused_add_rms_norm_nvfp4, h["x"][r0:r1],
                                            h["residual"][r0:r1], h["weight"], w.eps,
                                            w.static_scale, False))
                elif w.op == "silu4":
                    futs.append(pool.submit(orc.silu_mul_nvfp4, h["gate_up"][r0:r1],
                                            w.static_scale, False))
                elif w.op == "pad":
                    futs.append(pool.submit(orc.fused_add_rms_norm_pad, h["x"][r0:r1],
                                            h["residual"][r0:r1], h["weight"], w.eps, w.n2, False))
                elif w.op == "mla":
                    futs.append(pool.submit(orc.mla_dual_rms_norm, h["q_c"][r0:r1], h["q_weight"],
                                            h["kv_c"][r0:r1], h["kv_weight"], w.eps, w.eps,
                                            w.mode == gen.PER_TOKEN, False))
                else:
                    futs.append(pool.submit(orc.silu_mul_fp8, h["gate_up"][r0:r1], w.mode | w.flags,
                                            w.group_size, w.static_scale, False))
        for f in futs:
            f.result()

    return one, pool


def sample_step(step, host, rows):
    """The first `rows` rows of every op of a step (the generator's rows are
    independent blocks, so this is a prefix of the same workload)."""
    import dataclasses
    s_step, s_host = [], []
    for w, h in zip(step, host):
        r = min(w.T, rows)
        s_step.append(dataclasses.replace(w, T=r))
        s_host.append({k: (v[:r] if k in ROW_KEYS else v) for k, v in h.items()})
    return tuple(s_step), s_host


# host arrays indexed by token row (the rest are per-op constants)
ROW_KEYS = ("x", "residual", "gate_up", "q_c", "kv_c", "qkv", "positions")


def _time_oracle(step, host, threads, seconds, max_iters=1000):
    one, pool = oracle_step_runner(step, host, threads)
    one()  # builds/loads the oracle library, warms caches
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= max_iters:
            break
    pool.shutdown()
    return n, el


CPU_SAMPLE_ROWS = 4096       # rows per op in one sample step on all host cores
CPU_SAMPLE_ROWS_ONE = 256    # rows per op in one sample step on one thread


def run_cpu_baseline(step, host, seconds):
    """The oracle on all host cores (rows split over threads), then on one
    thread for a third of the time, each over a bounded row sample of the
    step repeated until the time is up."""
    threads = os.cpu_count() or 1
    s_step, s_host = sample_step(step, host, CPU_SAMPLE_ROWS)
    n, el = _time_oracle(s_step, s_host, threads, seconds)
    o_step, o_host = sample_step(step, host, CPU_SAMPLE_ROWS_ONE)
    n1, el1 = _time_oracle(o_step, o_host, 1, seconds / 3)
    rows = "+".join(str(w.T) for w in s_step)
    rows1 = "+".join(str(w.T) for w in o_step)
    return {"value": round(step_bytes(s_step) * n / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n} repetitions of the first {rows} rows of the step's ops "
                      f"({step_bytes(s_step) / 1e6:.1f} MB each, {el:.1f} s of CPU work), rows "
                      f"split over {threads} threads",
            "tokens_per_s": round(step_tokens(s_step) * n / el, 2),
            "single_thread": {"value": round(step_bytes(o_step) * n1 / el1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"{n1} repetitions of the first {rows1} rows on one thread "
                                        f"({el1:.1f} s)"}}


def run_reference(args, dist):
    """The fp64 CPU oracle as the reference arm, on this workload: each step
    is a bounded row sample (the first CPU_SAMPLE_ROWS rows of every op)."""
    if dist.rank != 0:
        return None
    import dataclasses
    full = select_step(args)
    # the generator's rows are independent blocks: inputs drawn for the
    # first R rows are the first R rows of the full workload's inputs
    step = tuple(dataclasses.replace(w, T=min(w.T, CPU_SAMPLE_ROWS)) for w in full)
    host = [w.inputs() for w in step]
    threads = os.cpu_count() or 1
    one, pool = oracle_step_runner(step, host, threads)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    pool.shutdown()
    value = step_bytes(step) * args.steps / el / 1e9
    rows = "+".join(str(w.T) for w in step)
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{args.steps} steps, each the first {rows} rows of the workload's ops "
                     f"({step_bytes(step) / 1e6:.1f} MB), rows split over {threads} threads"}
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "tokens_per_s": round(step_tokens(step) * args.steps / el, 2),
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "ops": [describe(w) for w in full],
                   "bytes_per_step": step_bytes(full),
                   "sample_ops": [describe(w) for w in step],
                   "sample_bytes_per_step": step_bytes(step)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def time_op_point(torch, vg, w, host, dev, stream, steps, warmup, l2, replays=5):
    """Duration (us) of one op's launch: K launches over rotating buffer
    sets (together > 3x L2) in one CUDA graph, one untimed replay, then the
    median of `replays` timed replays (CUDA events)."""
    nbytes = w.algorithmic_bytes()
    n_sets = max(2, min(64, math.ceil(3 * l2 / nbytes)))
    weights = device_weights(torch, (w,), [host], dev)
    sets = [DeviceSet(torch, (w,), [host], weights, dev) for _ in range(n_sets)]
    k_launch = max(steps, n_sets)
    with torch.cuda.stream(stream):
        for k in range(warmup):
            launch(vg, sets[k % n_sets].ops[0])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(k_launch):
            launch(vg, sets[k % n_sets].ops[0])
    torch.cuda.synchronize()
    spread = op_spread(torch, g, stream, k_launch, replays=replays)
    del sets, g, weights
    torch.cuda.empty_cache()
    spread = {k: (v * 1e3 if k != "replays" else v) for k, v in spread.items()}
    return spread["median"], spread


def point_record(w, us, peak, peak_kind, spread=None):
    nbytes = w.algorithmic_bytes()
    gbs = nbytes / (us * 1e-6) / 1e9
    r = {"point": w.name, "op": w.op, "T": w.T, "n": w.n, "mode": mode_name(w),
         "bytes": nbytes, "us": round(us, 3), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
         "peak": peak, "peak_source": peak_kind, "tokens_per_s": round(w.T / (us * 1e-6), 1)}
    if spread:
        r["us_spread"] = {k: (round(v, 3) if k != "replays" else v) for k, v in spread.items()}
    return r


def run_sweep(args):
    """Per-point kernel throughput of the bandwidth sweep and the named
    single-op configs, one JSON record per point."""
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
    cache = {}
    for w in (list(gen.NAMED.values()) + [CFG3_ACT] + gen.sweep() + gen.mla_workloads()
              + gen.pad_workloads() + gen.qk_workloads() + gen.nvfp4_workloads()
              + gen.group_option_workloads()):
        if args.sweep_filter and not any(f in w.name for f in args.sweep_filter.split(",")):
            continue
        key = (w.op, w.T, w.n, w.n2, w.x_dist)
        if key not in cache:
            cache.clear()
            cache[key] = w.inputs()
        us, spread = time_op_point(torch, vg, w, cache[key], dev, stream, args.steps, args.warmup, l2)
        print(json.dumps(point_record(w, us, peak, peak_kind, spread)), flush=True)
    return 0


def large_token_workloads():
    """The configs the >= 80 % roofline gate covers: SiLU 2048 x 14336
    (static and per-group 128), the 70B-shaped prefill norm, and every sweep
    point with T >= 4096 (both ops, all three scale modes, both shapes)."""
    return [gen.CFG2A, gen.CFG2B, gen.CFG3] + [w for w in gen.sweep() if w.T >= 4096]


def run_large_token(torch, vg, dev, stream, args, l2):
    """Every large-token point timed after the step in the same run.  Inputs
    are drawn once per (op, row length, distribution) at the largest T and
    sliced: the generator's rows are independent blocks, so the first T rows
    are exactly the inputs of the T-row point."""
    peak, peak_kind = measured_peak()
    points = large_token_workloads()
    groups = {}
    for w in points:
        groups.setdefault((w.op, w.n, w.x_dist), []).append(w)
    out = []
    for key, ws in groups.items():
        big = max(ws, key=lambda w: w.T)
        full = big.inputs()
        for w in ws:
            host = {k: (v[:w.T] if k in ROW_KEYS else v) for k, v in full.items()}
            us, spread = time_op_point(torch, vg, w, host, dev, stream, max(20, args.steps),
                                       args.warmup, l2)
            r = point_record(w, us, peak, peak_kind, spread)
            out.append({k: r[k] for k in ("point", "us", "GB/s", "frac", "us_spread")})
        del full
    return out


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
