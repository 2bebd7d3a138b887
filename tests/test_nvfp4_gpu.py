"""NVFP4 outputs of both fusions: the CUDA path against the oracle ("Fusion
torch.compile passes", "Quick Reference" table: FP4 outputs of "RMSNorm +
Quantization" and "SiLU+Mul + Quantization"; the NVFP4 format: E2M1
elements, E4M3 scales per 16 columns, an fp32 per-tensor scale).

Block scale codes must be bit-exact: both kernels decide them as the exact
gs * amax / 6 rounds (the norm in double-float, the SiLU kernel in fp64 near
an E4M3 midpoint).  Element codes follow the E2M1 code rule; residual_out is
bit-exact."""
import numpy as np
import pytest

import exact
import gen
import parity

pytestmark = pytest.mark.gpu

GS = (1.0, 168.0, 123.456)


def run_norm(x, res, w, eps, gs, inplace=True):
    g = parity.gpu_nvfp4_norm(x, res, w, eps, gs, inplace=inplace)
    o = parity.oracle_nvfp4_norm(x, res, w, eps, gs)
    parity.check_nvfp4(g, o)
    return g, o


def run_silu(gu, gs):
    g = parity.gpu_nvfp4_silu(gu, gs)
    o = parity.oracle_nvfp4_silu(gu, gs)
    parity.check_nvfp4(g, o)
    return g, o


# decode-sized register plans, packed short rows, and the pipelined TMA plan
# (T >= 4 rows per SM, H >= 2048); ragged block and chunk counts
@pytest.mark.parametrize("T,H", [(1, 4096), (7, 8192), (333, 4096), (2048, 4096), (700, 8192),
                                 (4099, 2048), (5, 16), (300, 48), (1200, 1040), (650, 2896),
                                 (3, 32768), (9, 12304)])
@pytest.mark.parametrize("gs", GS)
def test_norm_nvfp4_shapes(T, H, gs):
    d = gen.norm_inputs(T, H, seed=T + H)
    run_norm(d["x"], d["residual"], d["weight"], 1e-5, gs)


@pytest.mark.parametrize("T,H", [(4, 4096), (1000, 4096), (300, 1024)])
def test_norm_nvfp4_plain_and_out_of_place(T, H):
    d = gen.norm_inputs(T, H, seed=3)
    run_norm(d["x"], None, d["weight"], 1e-6, 168.0)
    run_norm(d["x"], d["residual"], d["weight"], 1e-6, 168.0, inplace=False)


def test_norm_nvfp4_heavy_tails():
    d = gen.norm_inputs(2048, 8192, seed=4, x_dist="t3_outliers")
    run_norm(d["x"], d["residual"], d["weight"], 1e-5, 168.0)


@pytest.mark.parametrize("gs", [1e-3, 168.0, 1e5])
def test_norm_nvfp4_edge_values(gs):
    """Zero, -0, constant, sparse, tiny and huge rows; gs small enough for
    subnormal E4M3 block scales and zero blocks, and large enough to
    saturate them at 448 (elements then saturate at 6)."""
    rng = np.random.default_rng(5)
    T, H = 8, 256

    def rows(scale_rows):
        x = np.zeros((T, H), np.float32)
        x[1] = -0.0
        x[2] = 1.5
        x[3, ::7] = -2.0
        x[4] = 1e-30 * rng.standard_normal(H)
        x[5] = 3e4 * rng.standard_normal(H)
        x[6] = np.where(np.arange(H) % 2 == 0, 1.0, -1.0)
        x[7] = rng.standard_normal(H) * np.exp2(rng.integers(-20, 20, H))
        return gen.to_bf16_bits(x * scale_rows)

    x = rows(1.0)
    res = rows(0.0)
    w = gen.to_bf16_bits((1 + 0.5 * rng.standard_normal(H)).astype(np.float32))
    g, o = run_norm(x, res, w, 1e-6, gs)
    assert np.all(g["sf"][0] == 0) and np.all(g["q4"][0] == 0)  # zero row: +0 everywhere


def test_norm_nvfp4_exact_ties():
    """eps = 0 and rows of mean square 1 make inv exactly 1, so with gs = 6
    the block value gs * amax / 6 is the block's largest |r w| itself: a bf16
    number, often exactly an E4M3 midpoint.  Both sides round ties to even."""
    rng = np.random.default_rng(6)
    T, H = 64, 512
    x = gen.to_bf16_bits(np.where(rng.random((T, H)) < 0.5, 1.0, -1.0).astype(np.float32))
    # weights on E4M3 midpoints (4 significant bits, the last one set)
    mids = np.array([1.0625, 1.1875, 1.3125, 1.4375, 1.5625, 2.125, 0.53125, 0.78125], np.float32)
    w = gen.to_bf16_bits(rng.choice(mids, H))
    g, o = run_norm(x, None, w, 0.0, 6.0)
    assert np.any(o["sf"] % 2 == 0)


def _midpoints():
    """Midpoints between E4M3 neighbours: subnormal, small, near 1, large."""
    v = exact.E4M3_POS_F64
    return [(v[i] + v[i + 1]) / 2 for i in (1, 3, 30, 56, 57, 80, 100, 120)]


def _norm_y(x, res, w, eps):
    """fp64 RMSNorm rows from bf16 bits (used only to choose a gs)."""
    xf = exact.bf16_bits_to_f64(x)
    r = xf if res is None else exact.bf16_bits_to_f64(gen.to_bf16_bits(
        (xf + exact.bf16_bits_to_f64(res)).astype(np.float32)))
    inv = 1.0 / np.sqrt(np.mean(r * r, axis=1, keepdims=True) + eps)
    return r * inv * exact.bf16_bits_to_f64(w)[None, :]


def test_norm_nvfp4_block_values_on_midpoints():
    """gs chosen so that one block's gs * amax / 6 falls within 2^-24 of an
    E4M3 midpoint: the block code must still be the exact value's."""
    d = gen.norm_inputs(64, 1024, seed=8)
    y = _norm_y(d["x"], None, d["weight"], 1e-5)
    amax = np.abs(y).reshape(64, -1, 16).max(axis=2)
    for k, mid in enumerate(_midpoints()):
        t, b = divmod(37 * k + 5, amax.shape[1])
        gs = float(np.float32(mid * 6.0 / amax[t % 64, b]))
        run_norm(d["x"], None, d["weight"], 1e-5, gs)


@pytest.mark.parametrize("T,I", [(1, 14336), (5, 4096), (64, 1024), (700, 14336), (2048, 2048),
                                 (33, 16), (300, 48), (129, 1040), (9, 32768), (2100, 28672)])
@pytest.mark.parametrize("gs", GS)
def test_silu_nvfp4_shapes(T, I, gs):
    run_silu(gen.silu_inputs(T, I, seed=T + I)["gate_up"], gs)


@pytest.mark.parametrize("gs", [1e-4, 168.0, 1e6])
def test_silu_nvfp4_edge_values(gs):
    rng = np.random.default_rng(9)
    T, I = 6, 512
    g = np.zeros((T, I), np.float32)
    u = np.ones((T, I), np.float32)
    g[1] = -0.0
    g[2] = rng.standard_normal(I) * 30          # exp(-g) huge and tiny
    g[3] = -100.0                               # silu underflows toward -0
    g[4] = rng.standard_normal(I)
    u[4] = 0.0                                  # products of zero
    g[5] = rng.standard_normal(I) * np.exp2(rng.integers(-30, 8, I))
    gu = np.concatenate([gen.to_bf16_bits(g), gen.to_bf16_bits(u)], axis=1)
    run_silu(gu, gs)


def _silu_a(gu):
    g = exact.bf16_bits_to_f64(gu[:, :gu.shape[1] // 2])
    u = exact.bf16_bits_to_f64(gu[:, gu.shape[1] // 2:])
    return g / (1.0 + np.exp(-g)) * u


def test_silu_nvfp4_block_values_on_midpoints():
    """The fp32 block value lands within 2^-24 of an E4M3 midpoint, inside
    the kernel's 2^-17 window: the fp64 recomputation must give the exact
    value's code."""
    gu = gen.silu_inputs(64, 2048, seed=10)["gate_up"]
    amax = np.abs(_silu_a(gu)).reshape(64, -1, 16).max(axis=2)
    for k, mid in enumerate(_midpoints()):
        t, b = divmod(53 * k + 11, amax.shape[1])
        gs = float(np.float32(mid * 6.0 / amax[t % 64, b]))
        run_silu(gu, gs)


def test_nvfp4_full_size_sampled():
    """The sweep's largest token count in the launch configuration it times;
    the oracle checks every 37th row."""
    T = 32768
    rows = np.arange(0, T, 37)
    d = gen.norm_inputs(T, gen.NVFP4_H, seed=0)
    g = parity.gpu_nvfp4_norm(d["x"], d["residual"], d["weight"], 1e-5, gen.NVFP4_GS)
    o = parity.oracle_nvfp4_norm(d["x"][rows], d["residual"][rows], d["weight"], 1e-5, gen.NVFP4_GS)
    parity.check_nvfp4(g, o, rows=rows)
    del d, g
    gu = gen.silu_inputs(T, gen.NVFP4_I, seed=0)["gate_up"]
    g = parity.gpu_nvfp4_silu(gu, gen.NVFP4_GS)
    o = parity.oracle_nvfp4_silu(gu[rows], gen.NVFP4_GS)
    parity.check_nvfp4(g, o, rows=rows)


def test_nvfp4_graph_capture_matches_eager():
    import torch
    import norm_activation_fp8_gb300 as vg
    dev = "cuda"
    d = gen.norm_inputs(512, 4096, seed=12)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    w = torch.from_numpy(d["weight"].view(np.int16)).to(dev)
    gs = torch.tensor([168.0], device=dev)
    q4e, sfe, _ = vg.fused_add_rms_norm_nvfp4(x, None, w, 1e-5, gs)
    gu = torch.from_numpy(gen.silu_inputs(512, 4096, seed=13)["gate_up"].view(np.int16)).to(dev)
    a4e, ase = vg.silu_mul_nvfp4(gu, gs)
    q4 = torch.empty_like(q4e)
    sf = torch.empty_like(sfe)
    a4 = torch.empty_like(a4e)
    asf = torch.empty_like(ase)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        vg.vg_fused_add_rms_norm_nvfp4(q4, sf, None, x, None, w, gs, 1e-5)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        vg.vg_fused_add_rms_norm_nvfp4(q4, sf, None, x, None, w, gs, 1e-5)
        vg.vg_silu_mul_nvfp4(a4, asf, gu, gs)
    q4.zero_()
    a4.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q4, q4e) and torch.equal(sf.view(torch.uint8), sfe.view(torch.uint8))
    assert torch.equal(a4, a4e) and torch.equal(asf.view(torch.uint8), ase.view(torch.uint8))
