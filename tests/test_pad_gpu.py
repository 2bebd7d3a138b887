"""Residual add + RMSNorm into a padded bf16 row: the CUDA path against the
oracle ("Fusion torch.compile passes", section "RMSNorm + Padding
(fuse_act_padding)").  The padded rows (tail included) and residual_out are
bit-exact.  Inputs are the seeded generators' bytes."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

H, HP = gen.PAD_HIDDEN, gen.PAD_PADDED


def run(T, hidden, padded, residual=True, inplace=True, eps=1e-6, seed=0, d=None):
    d = d or gen.norm_inputs(T, hidden, seed=seed)
    res = d["residual"] if residual else None
    g = parity.gpu_pad(d["x"], res, d["weight"], eps, padded, inplace=inplace)
    o = parity.oracle_pad(d["x"], res, d["weight"], eps, padded)
    parity.check_pad(g, o)
    return g, o


# decode sizes (register kernel) and T >= 4 rows per SM (the pipelined kernel)
@pytest.mark.parametrize("residual", [True, False], ids=["fused_add", "plain"])
@pytest.mark.parametrize("T", [1, 7, 64, 512, 700, 4099])
def test_pad_gpt_oss_shape(T, residual):
    run(T, H, HP, residual=residual, seed=T)


@pytest.mark.parametrize("hidden,padded,T", [
    (2880, 2880, 700),        # no padding
    (1032, 1040, 13),         # ragged chunk count, one padded chunk
    (1032, 2048, 700),        # a tail wider than one thread's share
    (8, 64, 5),               # one chunk of data, seven of padding
    (4096, 4104, 1300),
    (32768, 32776, 3),        # the widest row
    (8192, 16384, 650),       # pipelined, padded to twice the width
])
def test_pad_shapes(hidden, padded, T):
    run(T, hidden, padded, seed=hidden + padded + T)


def test_pad_out_of_place_equals_in_place():
    a, _ = run(640, H, HP, inplace=True, seed=1)
    b, _ = run(640, H, HP, inplace=False, seed=1)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["residual_out"], b["residual_out"])


def test_pad_edge_values():
    rng = np.random.default_rng(8)
    T, hidden = 8, 2880
    x = np.zeros((T, hidden), np.float32)
    x[1] = -0.0
    x[2] = 1.5
    x[3, ::5] = -2.0
    x[4] = 1e-30 * rng.standard_normal(hidden)
    x[5] = 3e4 * rng.standard_normal(hidden)
    x[6] = np.where(np.arange(hidden) % 2 == 0, 1.0, -1.0)
    x[7] = rng.standard_normal(hidden) * np.exp2(rng.integers(-20, 20, hidden))
    d = {"x": gen.to_bf16_bits(x), "residual": np.zeros((T, hidden), np.uint16),
         "weight": gen.to_bf16_bits((1 + 0.5 * rng.standard_normal(hidden)).astype(np.float32))}
    for residual in (True, False):
        run(T, hidden, HP, residual=residual, d=d)


def test_pad_prefill_full_size_sampled():
    """32768 tokens in the launch configuration the sweep times; the oracle
    checks every 37th token."""
    T = 32768
    d = gen.norm_inputs(T, H, seed=6)
    g = parity.gpu_pad(d["x"], d["residual"], d["weight"], 1e-6, HP)
    rows = np.arange(0, T, 37)
    o = parity.oracle_pad(d["x"][rows], d["residual"][rows], d["weight"], 1e-6, HP)
    parity.check_pad({"out": g["out"][rows], "residual_out": g["residual_out"][rows]}, o)
