"""NaN and infinity inputs: the CUDA path against the oracle (GPU).

The reading both sides follow: every formula is evaluated in IEEE
arithmetic as written, and the amax of a row or group is the largest |y|
among its non-NaN elements (0 when there is none).  So a NaN in r makes the
whole row NaN (codes 0x7F, dynamic scales at the floor); an infinity in r
gives inv = 0, codes +-0 at the finite elements and 0x7F at the infinite
one; an infinite SiLU activation saturates under a static scale and makes
its row's or group's dynamic scale +inf.  The oracle's side is pinned by
check_nonfinite_norm / check_nonfinite_silu.  Both the register kernels
(few rows) and the pipelined kernels (many rows) are covered.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
UE8M0, COL_MAJOR = parity.UE8M0, parity.COL_MAJOR
NAN16, PINF16, NINF16 = 0x7FC0, 0x7F80, 0xFF80


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from norm_activation_fp8_gb300 import build
    build.build()
    import norm_activation_fp8_gb300 as vg
    vg.load()


def plant_norm(x, res, rng, with_inf=True):
    """NaN / +-inf at random places of a few rows; returns the planted rows."""
    T, H = x.shape
    rows = rng.permutation(T)[:28]
    cols = rng.integers(0, H, rows.size)
    kinds = ["x_nan", "res_nan", "x_inf", "res_ninf", "inf_minus_inf"] if with_inf \
        else ["x_nan", "res_nan"]
    for i, (t, j) in enumerate(zip(rows, cols)):
        k = kinds[i % len(kinds)]
        if k == "x_nan":
            x[t, j] = NAN16
        elif k == "res_nan" and res is not None:
            res[t, j] = NAN16
        elif k == "x_inf":
            x[t, j] = PINF16
        elif k == "res_ninf" and res is not None:
            res[t, j] = NINF16
        elif k == "inf_minus_inf" and res is not None:
            x[t, j], res[t, j] = PINF16, NINF16
        else:
            x[t, j] = NAN16 if i % 2 else PINF16
    return rows


NORM_MODES = [(STATIC, 128), (PER_TOKEN, 128), (PER_GROUP, 128), (PER_GROUP, 64),
              (PER_GROUP | COL_MAJOR, 128), (PER_GROUP | UE8M0, 128)]


@pytest.mark.parametrize("T,H", [(64, 4096), (1024, 4096)], ids=["register", "pipelined"])
@pytest.mark.parametrize("mode,G", NORM_MODES, ids=lambda v: str(v))
@pytest.mark.parametrize("fused", [True, False], ids=["fused_add", "plain"])
def test_nonfinite_norm(T, H, mode, G, fused):
    rng = np.random.default_rng(T + mode + G)
    d = gen.norm_inputs(T, H, seed=5)
    x, w = d["x"].copy(), d["weight"]
    res = d["residual"].copy() if fused else None
    # an infinite amax has no power-of-two scale: UE8M0 gets NaN rows only
    rows = plant_norm(x, res, rng, with_inf=not (mode & UE8M0))
    g = parity.gpu_norm(x, res, w, 1e-5, mode, G, scale=0.05)
    o = parity.oracle_norm(x, res, w, 1e-5, mode, G, scale=0.05)
    parity.check_norm(g, o, mode & 0xFF)
    assert np.any(g["q"][rows] == 0x7F)


@pytest.mark.parametrize("mode,G", [(STATIC, 128), (PER_TOKEN, 128), (PER_GROUP, 128)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("T", [64, 1024], ids=["register", "pipelined"])
def test_nan_weight_and_zero_rows_without_eps(T, mode, G):
    """A NaN weight column turns only that column into NaN; with eps = 0 an
    all-zero row is 0 * (1/0) = NaN everywhere (the other rows are defined)."""
    H = 4096
    d = gen.norm_inputs(T, H, seed=6)
    w = d["weight"].copy()
    w[[3, 1000, 4095]] = NAN16
    g = parity.gpu_norm(d["x"], d["residual"], w, 1e-5, mode, G, scale=0.05)
    o = parity.oracle_norm(d["x"], d["residual"], w, 1e-5, mode, G, scale=0.05)
    parity.check_norm(g, o, mode)
    assert np.all(g["q"][:, [3, 1000, 4095]] == 0x7F)
    x = d["x"].copy()
    x[[0, T // 2, T - 1]] = 0
    g = parity.gpu_norm(x, None, d["weight"], 0.0, mode, G, scale=0.05)
    o = parity.oracle_norm(x, None, d["weight"], 0.0, mode, G, scale=0.05)
    parity.check_norm(g, o, mode)
    assert np.all(g["q"][[0, T // 2, T - 1]] == 0x7F)


def plant_silu(gu, rng, with_inf=True):
    T, two_i = gu.shape
    I = two_i // 2
    rows = rng.permutation(T)[:30]
    cols = rng.integers(0, I, rows.size)
    kinds = ["gate_nan", "up_nan", "gate_ninf", "up_inf", "gate_inf"] if with_inf \
        else ["gate_nan", "up_nan"]
    for i, (t, j) in enumerate(zip(rows, cols)):
        k = kinds[i % len(kinds)]
        if k == "gate_nan":
            gu[t, j] = NAN16
        elif k == "up_nan":
            gu[t, I + j] = NAN16
        elif k == "gate_ninf":
            gu[t, j] = NINF16           # silu(-inf) = -inf / inf = NaN
        elif k == "up_inf":
            gu[t, I + j] = PINF16       # +-inf, or NaN where the gate is 0
        else:
            gu[t, j] = PINF16           # silu(inf) = inf, times up
    return rows


SILU_MODES = [(STATIC, 128), (PER_TOKEN, 128), (PER_GROUP, 128), (PER_GROUP, 64),
              (PER_GROUP | COL_MAJOR, 128), (PER_GROUP | UE8M0, 128)]


@pytest.mark.parametrize("T,I", [(64, 4096), (400, 4096)], ids=["register", "pipelined"])
@pytest.mark.parametrize("mode,G", SILU_MODES, ids=lambda v: str(v))
def test_nonfinite_silu(T, I, mode, G):
    rng = np.random.default_rng(T + mode + G + 1)
    gu = gen.silu_inputs(T, I, seed=7)["gate_up"].copy()
    rows = plant_silu(gu, rng, with_inf=not (mode & UE8M0))
    g = parity.gpu_silu(gu, mode, G, scale=0.1)
    o = parity.oracle_silu(gu, mode, G, scale=0.1)
    parity.check_silu(g, o, mode & 0xFF)
    assert np.any(g["q"][rows] == 0x7F)
