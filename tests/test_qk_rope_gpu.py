"""Per-head QK RMSNorm + rotary embedding: the CUDA path against the oracle
("Fusion torch.compile passes", section "QK Norm + RoPE
(enable_qk_norm_rope_fusion)").  qkv is updated in place; the Q and K heads
follow the bf16 tolerance (the kernel's fp32 value is within 2^-20 of the
exact one: identical codes except one-ulp flips within 2^-19 of a bf16
midpoint, at most 0.1 %), and the V heads are untouched.  Inputs are the
seeded generators' bytes."""
import numpy as np
import pytest

import gen
import parity
import norm_activation_fp8_gb300 as vg

pytestmark = pytest.mark.gpu

HQ, HKV, D, MAXP = gen.QK_HQ, gen.QK_HKV, gen.QK_D, gen.QK_MAX_POS


def run(T, hq, hkv, head_dim, neox, max_pos=4096, eps=1e-6, seed=0, d=None):
    d = d or gen.qk_inputs(T, hq, hkv, head_dim, max_pos, seed=seed)
    g = parity.gpu_qk(d, hq, hkv, head_dim, eps, neox)
    parity.check_qk(g, parity.oracle_qk(d, hq, hkv, head_dim, eps, neox), d["qkv"], hq, hkv, head_dim)
    return g


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
@pytest.mark.parametrize("T", [1, 7, 64, 333, 2048])
def test_qk_qwen3_shape(T, neox):
    run(T, HQ, HKV, D, neox, max_pos=MAXP, seed=T)


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
@pytest.mark.parametrize("hq,hkv,head_dim,T", [
    (16, 4, 64, 301),
    (8, 1, 256, 129),
    (5, 0, 128, 33),     # query heads only
    (0, 3, 128, 17),     # key heads only (V still follows them)
    (1, 1, 64, 1),       # one head of each in a warp with dead lanes
    (64, 8, 128, 77),    # Qwen3-32B
])
def test_qk_shapes(hq, hkv, head_dim, T, neox):
    run(T, hq, hkv, head_dim, neox, seed=hq * 100 + hkv + head_dim + T)


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_qk_edge_values(neox):
    """Zero and -0 heads (inv = 1/sqrt(eps)), constant, tiny and huge heads,
    position 0 (the identity rotation) and the last position."""
    rng = np.random.default_rng(9)
    T, hq, hkv, head_dim = 6, 2, 1, 128
    row = (hq + 2 * hkv) * head_dim
    x = rng.standard_normal((T, row)).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] = 1.5
    x[3] = 1e-30 * rng.standard_normal(row)
    x[4] = 3e4 * rng.standard_normal(row)
    d = gen.qk_inputs(T, hq, hkv, head_dim, 64, seed=3)
    d["qkv"] = gen.to_bf16_bits(x)
    d["positions"] = np.array([0, 63, 5, 0, 17, 63], np.int64)
    run(T, hq, hkv, head_dim, neox, d=d)


def test_qk_bad_position_is_reported_and_skipped():
    """A position outside the cache leaves that token unchanged and sets
    VG_DEVICE_BAD_POSITION; the other tokens are still exact."""
    T = 9
    d = gen.qk_inputs(T, 4, 2, 128, 64, seed=4)
    good = np.ones(T, bool)
    d["positions"][3] = 64
    d["positions"][7] = -1
    good[[3, 7]] = False
    vg.vg_device_status(reset=True)
    g = parity.gpu_qk(d, 4, 2, 128, 1e-6, True)
    assert vg.vg_device_status(reset=True) & vg.DEVICE_BAD_POSITION
    assert np.array_equal(g[~good], d["qkv"][~good])
    ok = {k: (v[good] if k in ("qkv", "positions") else v) for k, v in d.items()}
    parity.check_qk(g[good], parity.oracle_qk(ok, 4, 2, 128, 1e-6, True), ok["qkv"], 4, 2, 128)
    assert vg.vg_device_status() == 0


def test_qk_prefill_full_size_sampled():
    """32768 tokens in the launch configuration the sweep times; the oracle
    checks every 31st token."""
    T = 32768
    d = gen.qk_inputs(T, HQ, HKV, D, MAXP, seed=7)
    g = parity.gpu_qk(d, HQ, HKV, D, 1e-6, True)
    rows = np.arange(0, T, 31)
    sub = {k: (v[rows] if k in ("qkv", "positions") else v) for k, v in d.items()}
    stats = parity.check_qk(g[rows], parity.oracle_qk(sub, HQ, HKV, D, 1e-6, True), sub["qkv"],
                            HQ, HKV, D)
    assert stats["flips"] <= 1e-3 * stats["elements"]
