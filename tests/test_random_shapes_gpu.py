"""Seeded random shapes for every op, against the oracle.

The launch plans switch kernels at token counts that depend on the SM count
(2, 4, 13 and 40 rows per SM on the 152-SM GB300: T = 304, 608, 1976, 6080)
and at row widths (chunks per thread, TMA staging, column segments).  These
cases draw token counts on both sides of each switch and widths, modes and
options at random (a fixed seed, so the set is the same on every run), and
check each against the oracle under the same tolerances as the fixed cases."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

PG, UE, CM = 2, 0x100, 0x200
_rng = np.random.default_rng(2026)
_EDGES = [303, 304, 305, 607, 608, 609, 1975, 1976, 1977, 6079, 6080, 6081]


def _tokens(n, cap):
    """n token counts: plan edges and random ones, each within the budget."""
    picks = list(_rng.choice(_EDGES, n // 2, replace=False)) + list(_rng.integers(1, 4000, n - n // 2))
    return [int(min(t, cap)) for t in picks]


def _norm_cases(n=14):
    out = []
    for T in _tokens(n, 6100):
        mode = int(_rng.choice([0, 1, 2, 2 | UE, 2 | CM, 2 | UE | CM]))
        G = int(_rng.choice([64, 128]))
        step = G if mode & 0xFF == 2 else 8
        H = int(_rng.integers(1, max(2, min(12288, 6_000_000 // T) // step) + 1)) * step
        out.append((T, H, mode, G, bool(_rng.integers(0, 2))))
    return out


def _silu_cases(n=12):
    out = []
    for T in _tokens(n, 6100):
        mode = int(_rng.choice([0, 1, 2, 2 | UE, 2 | CM, 2 | UE | CM]))
        G = int(_rng.choice([64, 128]))
        step = G if mode & 0xFF == 2 else 8
        I = int(_rng.integers(1, max(2, min(20480, 4_000_000 // T) // step) + 1)) * step
        out.append((T, I, mode, G))
    return out


def _nvfp4_cases(n=10):
    out = []
    for T in _tokens(n, 6100):
        n_cols = int(_rng.integers(1, max(2, min(16384, 4_000_000 // T) // 16) + 1)) * 16
        out.append((T, n_cols, bool(_rng.integers(0, 2)), float(_rng.choice([1.0, 168.0, 37.5]))))
    return out


NORM = _norm_cases()
SILU = _silu_cases()
NVFP4 = _nvfp4_cases()


@pytest.mark.parametrize("T,H,mode,G,res", NORM, ids=[f"{t}x{h}-m{m:#x}-g{g}-r{int(r)}" for t, h, m, g, r in NORM])
def test_random_norm(T, H, mode, G, res):
    d = gen.norm_inputs(T, H, seed=T + H)
    r = d["residual"] if res else None
    g = parity.gpu_norm(d["x"], r, d["weight"], 1e-5, mode, G, scale=0.05)
    o = parity.oracle_norm(d["x"], r, d["weight"], 1e-5, mode, G, scale=0.05)
    parity.check_norm(g, o, mode & 0xFF)


@pytest.mark.parametrize("T,I,mode,G", SILU, ids=[f"{t}x{i}-m{m:#x}-g{g}" for t, i, m, g in SILU])
def test_random_silu(T, I, mode, G):
    gu = gen.silu_inputs(T, I, seed=T + I)["gate_up"]
    g = parity.gpu_silu(gu, mode, G, scale=0.1)
    o = parity.oracle_silu(gu, mode, G, scale=0.1)
    parity.check_silu(g, o, mode & 0xFF)


@pytest.mark.parametrize("T,n,norm,gs", NVFP4, ids=[f"{t}x{n}-{'norm' if k else 'silu'}-gs{gs:g}" for t, n, k, gs in NVFP4])
def test_random_nvfp4(T, n, norm, gs):
    if norm:
        d = gen.norm_inputs(T, n, seed=T + n)
        g = parity.gpu_nvfp4_norm(d["x"], d["residual"], d["weight"], 1e-5, gs)
        o = parity.oracle_nvfp4_norm(d["x"], d["residual"], d["weight"], 1e-5, gs)
    else:
        gu = gen.silu_inputs(T, n, seed=T + n)["gate_up"]
        g = parity.gpu_nvfp4_silu(gu, gs)
        o = parity.oracle_nvfp4_silu(gu, gs)
    parity.check_nvfp4(g, o)


def _pad_cases(n=6):
    out = []
    for T in _tokens(n, 6100):
        H = int(_rng.integers(1, max(2, min(8192, 3_000_000 // T) // 8) + 1)) * 8
        out.append((T, H, H + 8 * int(_rng.integers(0, 64))))
    return out


def _mla_cases(n=8):
    out = []
    for T in _tokens(n, 7000):
        q = int(_rng.choice([512, 1024, 1536, 1536, 2048])) + 8 * int(_rng.integers(-4, 5))
        kv = int(_rng.choice([256, 512, 512])) + 8 * int(_rng.integers(-4, 5))
        out.append((T, q, kv, bool(_rng.integers(0, 2))))
    return out


def _qk_cases(n=6):
    out = []
    for i, T in enumerate(_tokens(n, 4000)):
        D = int(_rng.choice([64, 128, 256]))
        out.append((T, int(_rng.integers(1, 33)), int(_rng.integers(0, 9)), D, i % 2 == 0))
    return out


PAD = _pad_cases()
MLA = _mla_cases()
QK = _qk_cases()


@pytest.mark.parametrize("T,H,P", PAD, ids=[f"{t}x{h}->{p}" for t, h, p in PAD])
def test_random_pad(T, H, P):
    d = gen.norm_inputs(T, H, seed=T + H)
    g = parity.gpu_pad(d["x"], d["residual"], d["weight"], 1e-6, P)
    o = parity.oracle_pad(d["x"], d["residual"], d["weight"], 1e-6, P)
    parity.check_pad(g, o)


@pytest.mark.parametrize("T,q,kv,fp8", MLA, ids=[f"{t}x{q}+{kv}-{'fp8' if f else 'bf16'}" for t, q, kv, f in MLA])
def test_random_mla(T, q, kv, fp8):
    d = gen.mla_inputs(T, q, kv, seed=T + q + kv)
    g = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-6, fp8)
    o = parity.oracle_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-6, fp8)
    parity.check_mla(g, o, fp8)


@pytest.mark.parametrize("T,hq,hkv,D,neox", QK, ids=[f"{t}x{hq}q{hkv}kv{d}-{'neox' if n else 'gptj'}" for t, hq, hkv, d, n in QK])
def test_random_qk(T, hq, hkv, D, neox):
    d = gen.qk_inputs(T, hq, hkv, D, 4096, seed=T + hq + D)
    g = parity.gpu_qk(d, hq, hkv, D, 1e-6, neox)
    parity.check_qk(g, parity.oracle_qk(d, hq, hkv, D, 1e-6, neox), d["qkv"], hq, hkv, D)
