"""Per-group UE8M0 (power-of-two) and column-major scales on the GPU against
the oracle, for both ops and both norm kernels.  Power-of-two scales must
equal the oracle's exactly; codes follow the FP8 code rule; a column-major
buffer's padding columns must keep their guard pattern."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

PG, UE, CM = 2, 0x100, 0x200
FLAGS = [UE, CM, UE | CM]
IDS = ["ue8m0", "colmajor", "ue8m0+colmajor"]


@pytest.mark.parametrize("flags", FLAGS, ids=IDS)
@pytest.mark.parametrize("T,H,G", [(7, 4096, 128), (333, 4096, 64), (1300, 8192, 128),
                                   (2049, 4096, 128), (5, 1024, 64)])
def test_norm_group_scale_options(T, H, G, flags):
    d = gen.norm_inputs(T, H, seed=T + H + flags)
    mode = PG | flags
    g = parity.gpu_norm(d["x"], d["residual"], d["weight"], 1e-5, mode, G)
    o = parity.oracle_norm(d["x"], d["residual"], d["weight"], 1e-5, mode, G)
    parity.check_norm(g, o, mode)
    if flags & UE:
        assert np.array_equal(g["scale"], o["scale"])


@pytest.mark.parametrize("flags", FLAGS, ids=IDS)
@pytest.mark.parametrize("T,I,G", [(8, 14336, 128), (512, 14336, 64), (2048, 5120, 128),
                                   (33, 28672, 128), (3, 1024, 64)])
def test_silu_group_scale_options(T, I, G, flags):
    d = gen.silu_inputs(T, I, seed=T + I + flags)
    mode = PG | flags
    g = parity.gpu_silu(d["gate_up"], mode, G)
    o = parity.oracle_silu(d["gate_up"], mode, G)
    parity.check_silu(g, o, mode)
    if flags & UE:
        assert np.array_equal(g["scale"], o["scale"])


def _near_boundary_pairs(n):
    """bf16 (g, u) pairs whose silu(g) * u lies within 2^-20 (relative, but
    not exactly) of 448 * 2^k for some k -- closer than the kernel's fp32
    amax can tell apart -- found by exhaustive search over bf16 values
    (fp64 arithmetic)."""
    gs = gen.to_bf16_bits(np.linspace(-8.0, 20.0, 8000, dtype=np.float32))
    us = gen.to_bf16_bits(np.geomspace(1e-4, 1e4, 8000).astype(np.float32))
    gf = parity.exact.bf16_bits_to_f64(np.unique(gs))
    uf = parity.exact.bf16_bits_to_f64(np.unique(us))
    a = (gf / (1.0 + np.exp(-gf)))[:, None] * uf[None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = a / 448.0
        k = np.round(np.log2(np.abs(r)))
        rel = np.abs(np.abs(r) / np.exp2(k) - 1.0)
    ii, jj = np.nonzero((rel < 2.0 ** -20) & (rel > 0))
    picks = [(gf[i], uf[j]) for i, j in zip(ii, jj)][:n]
    assert len(picks) >= 4, "no near-boundary pairs found"
    return picks


@pytest.mark.parametrize("flags", [UE, UE | CM], ids=["ue8m0", "ue8m0+colmajor"])
def test_silu_ue8m0_amax_at_a_power_of_two_boundary(flags):
    """Groups whose amax sits within 2^-20 of 448 * 2^k: the fp32 amax cannot
    settle the exponent, the fp64 recheck must, exactly as the oracle does."""
    picks = _near_boundary_pairs(16)
    T, I, G = len(picks), 1024, 64
    rng = np.random.default_rng(12)
    gate = rng.standard_normal((T, I)) * 0.05
    up = rng.standard_normal((T, I)) * 0.05
    for t, (gv, uv) in enumerate(picks):
        j = (t * 37) % I
        gate[t, j], up[t, j] = gv, uv
    gu = gen.to_bf16_bits(np.concatenate([gate, up], axis=1).astype(np.float32))
    g = parity.gpu_silu(gu, PG | flags, G)
    o = parity.oracle_silu(gu, PG | flags, G)
    assert np.array_equal(g["scale"], o["scale"])
    parity.check_silu(g, o, PG | flags)


def test_norm_ue8m0_colmajor_prefill_sampled():
    """The pipelined norm at 16384 x 8192 (the prefill shape) with both
    options; the oracle checks every 29th row."""
    T, H = 16384, 8192
    d = gen.norm_inputs(T, H, seed=21, x_dist="t3_outliers")
    mode = PG | UE | CM
    g = parity.gpu_norm(d["x"], d["residual"], d["weight"], 1e-5, mode, 128)
    rows = np.arange(0, T, 29)
    o = parity.oracle_norm(d["x"][rows], d["residual"][rows], d["weight"], 1e-5, mode, 128)
    parity.check_norm(g, o, mode, rows=rows)
    assert np.array_equal(g["scale"][rows], o["scale"])


def test_group_options_sweep_full_size_sampled():
    """The sweep's largest UE8M0 + column-major points (32768 tokens) in the
    launch configuration it times; the oracle checks every 41st row."""
    T = 32768
    rows = np.arange(0, T, 41)
    mode = PG | UE | CM
    w = next(x for x in gen.group_option_workloads() if x.op == "norm" and x.T == T)
    d = w.inputs()
    g = parity.gpu_norm(d["x"], d["residual"], d["weight"], w.eps, mode, 128)
    o = parity.oracle_norm(d["x"][rows], d["residual"][rows], d["weight"], w.eps, mode, 128)
    parity.check_norm(g, o, mode, rows=rows)
    assert np.array_equal(g["scale"][rows], o["scale"])
    del d, g
    w = next(x for x in gen.group_option_workloads() if x.op == "silu" and x.T == T)
    gu = w.inputs()["gate_up"]
    g = parity.gpu_silu(gu, mode, 128)
    o = parity.oracle_silu(gu[rows], mode, 128)
    parity.check_silu(g, o, mode, rows=rows)
    assert np.array_equal(g["scale"][rows], o["scale"])
