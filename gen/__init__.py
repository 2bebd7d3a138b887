"""Seeded synthetic inputs for the fused norm/act -> FP8 ops.

This module is shared by the tests, the smoke check and the benchmark, and
serves both the oracle and the CUDA path with the same bytes.  It contains
none of the method's arithmetic: it draws random numbers (numpy PCG64 streams
keyed by ``(seed, tensor id, row block)``) and converts them to bf16 with
PyTorch's CPU cast, which rounds to nearest even.

Distributions follow the workloads in the design notes:
  x, residual, gate_up, q_c, kv_c ~ N(0, 1)
  weight               ~ 1 + 0.1 * N(0, 1)
  prefill x            ~ Student-t(3) with 0.1 % of the elements scaled by 100
Each tensor is split into blocks of rows generated independently, so a
tensor's values do not depend on the number of threads used.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

TENSOR_X, TENSOR_RESIDUAL, TENSOR_WEIGHT, TENSOR_GATE_UP = 1, 2, 3, 4
TENSOR_Q_C, TENSOR_KV_C, TENSOR_Q_WEIGHT, TENSOR_KV_WEIGHT = 5, 6, 7, 8
TENSOR_QKV, TENSOR_POSITIONS = 9, 10
_ROW_BLOCK = 64

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
UE8M0, COL_MAJOR = 0x100, 0x200  # per-group scale options, or-ed into the mode
MODE_NAMES = {STATIC: "static", PER_TOKEN: "per_token", PER_GROUP: "per_group"}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _rng(seed: int, tensor_id: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, block])))


def _draw(kind: str, rng: np.random.Generator, shape) -> np.ndarray:
    if kind == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if kind == "weight":
        return (1.0 + 0.1 * rng.standard_normal(shape, dtype=np.float64)).astype(np.float32)
    if kind == "t3_outliers":
        t = rng.standard_t(3, size=shape)
        hit = rng.random(shape) < 0.001
        t[hit] *= 100.0
        return t.astype(np.float32)
    raise ValueError(f"unknown distribution {kind!r}")


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns (PyTorch's RNE cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_tensor(kind: str, seed: int, tensor_id: int, rows: int, cols: int) -> np.ndarray:
    """A [rows, cols] bf16 tensor (uint16 bits) of distribution ``kind``."""
    out = np.empty((rows, cols), np.uint16)
    nblocks = (rows + _ROW_BLOCK - 1) // _ROW_BLOCK

    def work(b):
        r0 = b * _ROW_BLOCK
        r1 = min(rows, r0 + _ROW_BLOCK)
        vals = _draw(kind, _rng(seed, tensor_id, b), (r1 - r0, cols))
        out[r0:r1] = to_bf16_bits(vals)

    if nblocks <= 2:
        for b in range(nblocks):
            work(b)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nblocks)))
    return out


def norm_inputs(T: int, H: int, seed: int = 0, x_dist: str = "normal"):
    """x [T,H], residual [T,H], weight [H] as uint16 bf16 bits."""
    return {
        "x": bf16_tensor(x_dist, seed, TENSOR_X, T, H),
        "residual": bf16_tensor("normal", seed, TENSOR_RESIDUAL, T, H),
        "weight": bf16_tensor("weight", seed, TENSOR_WEIGHT, 1, H).reshape(H),
    }


def silu_inputs(T: int, I: int, seed: int = 0):
    """gate_up [T, 2I] (gate half, then up half) as uint16 bf16 bits."""
    return {"gate_up": bf16_tensor("normal", seed, TENSOR_GATE_UP, T, 2 * I)}


def mla_inputs(T: int, q_dim: int, kv_dim: int, seed: int = 0):
    """q_c [T,q_dim], kv_c [T,kv_dim] and their weights as uint16 bf16 bits."""
    return {
        "q_c": bf16_tensor("normal", seed, TENSOR_Q_C, T, q_dim),
        "kv_c": bf16_tensor("normal", seed, TENSOR_KV_C, T, kv_dim),
        "q_weight": bf16_tensor("weight", seed, TENSOR_Q_WEIGHT, 1, q_dim).reshape(q_dim),
        "kv_weight": bf16_tensor("weight", seed, TENSOR_KV_WEIGHT, 1, kv_dim).reshape(kv_dim),
    }


def rope_cache(max_pos: int, head_dim: int, theta: float = 1.0e6) -> np.ndarray:
    """The rotary embedding's cos/sin table, a model constant the op reads:
    row p = [cos(p f_0), ..., cos(p f_{D/2-1}), sin(p f_0), ...] with
    f_i = theta^(-2i/D), computed in fp64 and stored as fp32."""
    f = theta ** (-np.arange(0, head_dim, 2, dtype=np.float64) / head_dim)
    ang = np.outer(np.arange(max_pos, dtype=np.float64), f)
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def qk_inputs(T: int, hq: int, hkv: int, head_dim: int, max_pos: int, seed: int = 0):
    """qkv [T, (hq + 2 hkv) * D] bf16 bits, q/k weights [D], positions int64
    [T] uniform in [0, max_pos), and the cos/sin cache [max_pos, D]."""
    rng = _rng(seed, TENSOR_POSITIONS, 0)
    return {
        "qkv": bf16_tensor("normal", seed, TENSOR_QKV, T, (hq + 2 * hkv) * head_dim),
        "q_weight": bf16_tensor("weight", seed, TENSOR_Q_WEIGHT, 1, head_dim).reshape(head_dim),
        "k_weight": bf16_tensor("weight", seed, TENSOR_KV_WEIGHT, 1, head_dim).reshape(head_dim),
        "positions": rng.integers(0, max_pos, T).astype(np.int64),
        "cos_sin_cache": rope_cache(max_pos, head_dim),
    }


# ----------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """One op invocation: which op, its shape, scale mode and inputs."""
    name: str
    op: str                  # "norm", "silu", "mla", "pad", "qk"; NVFP4 "norm4", "silu4"
    T: int
    n: int                   # hidden (norm), intermediate (silu) or q_dim (mla)
    mode: int                # mla: PER_TOKEN = q to fp8, STATIC = bf16 q
    n2: int = 0              # mla: kv_dim; pad: padded row length
    hq: int = 0              # qk: query heads (n = head_dim, mode 1 = neox, 0 = gptj)
    hkv: int = 0             # qk: key/value heads
    max_pos: int = 0         # qk: rows of the cos/sin cache
    group_size: int = 128
    flags: int = 0               # per-group options (UE8M0, COL_MAJOR)
    eps: float = 1e-5
    static_scale: float = 0.05   # static fp8 scale; NVFP4: the per-tensor scale gs
    x_dist: str = "normal"
    residual: bool = True
    seed: int = 0
    note: str = field(default="", compare=False)

    def inputs(self):
        if self.op in ("norm", "pad", "norm4"):
            return norm_inputs(self.T, self.n, self.seed, self.x_dist)
        if self.op == "mla":
            return mla_inputs(self.T, self.n, self.n2, self.seed)
        if self.op == "qk":
            return qk_inputs(self.T, self.hq, self.hkv, self.n, self.max_pos, self.seed)
        return silu_inputs(self.T, self.n, self.seed)

    def algorithmic_bytes(self) -> int:
        """Bytes the op must move: every row read once and written once; the
        weight and a static scale read once per launch."""
        if self.op == "norm4":  # x, residual in; residual_out, E2M1 codes, E4M3 block scales out
            per_row = (6 if self.residual else 2) * self.n + self.n // 2 + self.n // 16
            return self.T * per_row + 2 * self.n + 4
        if self.op == "silu4":
            return self.T * (4 * self.n + self.n // 2 + self.n // 16) + 4
        s_row = {STATIC: 0, PER_TOKEN: 4, PER_GROUP: 4 * (self.n // self.group_size)}[self.mode]
        s0 = 4 if self.mode == STATIC else 0
        if self.op == "norm":
            per_row = (7 if self.residual else 3) * self.n + s_row
            return self.T * per_row + 2 * self.n + s0
        if self.op == "qk":  # Q and K heads read and written; each token's cos/sin row and position
            return self.T * ((self.hq + self.hkv) * self.n * 4 + self.n * 4 + 8) + 2 * 2 * self.n
        if self.op == "pad":  # x, residual read; residual_out and the padded row written
            return self.T * (6 * self.n + 2 * self.n2) + 2 * self.n
        if self.op == "mla":  # both rows read; q out as fp8 + scale or bf16; kv out bf16
            q_out = self.n + 4 if self.mode == PER_TOKEN else 2 * self.n
            return self.T * (2 * self.n + 4 * self.n2 + q_out) + 2 * (self.n + self.n2)
        return self.T * (5 * self.n + s_row) + s0


# The named shapes: a small static case, a Llama-3-8B-shaped decode step, the
# SiLU-and-mul 2048 x 14336 case in two modes, a 70B-shaped prefill with
# heavy-tailed activations, and the bandwidth sweep.
CFG0 = Workload("norm_static_16x1024", "norm", 16, 1024, STATIC, eps=1e-6, static_scale=0.05)
CFG1 = Workload("norm_per_token_256x4096", "norm", 256, 4096, PER_TOKEN, eps=1e-5)
CFG2A = Workload("silu_static_2048x14336", "silu", 2048, 14336, STATIC, static_scale=0.1)
CFG2B = Workload("silu_per_group128_2048x14336", "silu", 2048, 14336, PER_GROUP, group_size=128)
CFG3 = Workload("norm_per_group128_16384x8192_t3", "norm", 16384, 8192, PER_GROUP,
                group_size=128, eps=1e-5, x_dist="t3_outliers")
# The SiLU half of the Llama-3-8B decode step: intermediate 14336 pairs with
# hidden 4096 in the sweep's shape list.
CFG1_ACT = Workload("silu_per_token_256x14336", "silu", 256, 14336, PER_TOKEN)

NAMED = {w.name: w for w in (CFG0, CFG1, CFG2A, CFG2B, CFG3, CFG1_ACT)}

# Residual add + RMSNorm into a padded bf16 row at GPT-OSS's hidden size,
# padded to the next multiple of 256.
PAD_HIDDEN, PAD_PADDED = 2880, 3072
PAD_T = (1, 64, 512, 4096, 32768)


def pad_workloads():
    return [Workload(f"norm_pad_{T}x{PAD_HIDDEN}_{PAD_PADDED}", "pad", T, PAD_HIDDEN, PER_TOKEN,
                     n2=PAD_PADDED, eps=1e-6) for T in PAD_T]


# Per-head QK RMSNorm + RoPE at Qwen3-8B's attention shape: 32 query heads,
# 8 key/value heads, head_dim 128, rope theta 1e6, positions in [0, 32768).
QK_HQ, QK_HKV, QK_D, QK_MAX_POS = 32, 8, 128, 32768
QK_T = (1, 64, 512, 4096, 32768)


def qk_workloads():
    return [Workload(f"qk_norm_rope_{'neox' if m else 'gptj'}_{T}x{QK_HQ}q{QK_HKV}kv{QK_D}", "qk", T,
                     QK_D, m, hq=QK_HQ, hkv=QK_HKV, max_pos=QK_MAX_POS, eps=1e-6)
            for m in (1, 0) for T in QK_T]


# The MLA dual norm at DeepSeek-V3's latent sizes (q_lora_rank 1536,
# kv_lora_rank 512), bf16 and per-token-fp8 q, decode and prefill token counts.
MLA_Q_DIM, MLA_KV_DIM, MLA_ROPE = 1536, 512, 64
MLA_T = (1, 64, 512, 4096, 32768)


def mla_workloads():
    return [Workload(f"mla_dual_{'fp8' if m == PER_TOKEN else 'bf16'}_{T}x{MLA_Q_DIM}_{MLA_KV_DIM}",
                     "mla", T, MLA_Q_DIM, m, n2=MLA_KV_DIM, eps=1e-6)
            for m in (STATIC, PER_TOKEN) for T in MLA_T]


# NVFP4 outputs of both fusions at Llama-3-70B's sizes (hidden 8192,
# intermediate 28672).  gs = 448 * 6 / 16, the per-tensor scale of a tensor
# whose amax is 16.
NVFP4_H, NVFP4_I, NVFP4_GS = 8192, 28672, 168.0
NVFP4_T = (1, 64, 512, 4096, 32768)


def nvfp4_workloads():
    return ([Workload(f"norm_nvfp4_{T}x{NVFP4_H}", "norm4", T, NVFP4_H, PER_GROUP, group_size=16,
                      eps=1e-5, static_scale=NVFP4_GS) for T in NVFP4_T]
            + [Workload(f"silu_nvfp4_{T}x{NVFP4_I}", "silu4", T, NVFP4_I, PER_GROUP, group_size=16,
                        static_scale=NVFP4_GS) for T in NVFP4_T])


# Per-group 128 scales in the format a DeepGEMM-style FP8 GEMM on sm100
# consumes: powers of two (UE8M0), stored column-major.
def group_option_workloads():
    f = UE8M0 | COL_MAJOR
    return ([Workload(f"norm_per_group128_ue8m0_colmajor_{T}x8192", "norm", T, 8192, PER_GROUP,
                      flags=f, eps=1e-5) for T in (512, 4096, 32768)]
            + [Workload(f"silu_per_group128_ue8m0_colmajor_{T}x14336", "silu", T, 14336, PER_GROUP,
                        flags=f) for T in (512, 4096, 32768)])


SWEEP_T = (1, 8, 64, 512, 4096, 32768)
SWEEP_SHAPES = ((4096, 14336), (8192, 28672))


def sweep():
    """Both ops x three scale modes x T x (hidden, intermediate)."""
    out = []
    for H, I in SWEEP_SHAPES:
        for mode in (STATIC, PER_TOKEN, PER_GROUP):
            for T in SWEEP_T:
                out.append(Workload(f"norm_{MODE_NAMES[mode]}_{T}x{H}", "norm", T, H, mode,
                                    eps=1e-5, static_scale=0.05))
                out.append(Workload(f"silu_{MODE_NAMES[mode]}_{T}x{I}", "silu", T, I, mode,
                                    static_scale=0.1))
    return out
