"""MLA dual RMSNorm: the CUDA path against the oracle ("Fusion torch.compile
passes", section "MLA Dual RMSNorm (fuse_mla_dual_rms_norm)").

bf16 outputs must be bit-exact; the fp8 q side follows the FP8 code rule and
its per-token scales agree within 1e-6 (exactly, in practice: see
test_mla_fp8_q_exact).  Inputs are the seeded generators' bytes."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

Q, KV = gen.MLA_Q_DIM, gen.MLA_KV_DIM


def run(T, q_dim, kv_dim, q_fp8, eps_q=1e-6, eps_kv=1e-6, seed=0, inputs=None, **layout):
    d = inputs or gen.mla_inputs(T, q_dim, kv_dim, seed=seed)
    g = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], eps_q, eps_kv,
                       q_fp8, **layout)
    o = parity.oracle_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], eps_q, eps_kv,
                          q_fp8)
    return g, o, parity.check_mla(g, o, q_fp8)


# decode (one token per CTA), the packed-token plan, and prefill sizes
@pytest.mark.parametrize("q_fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("T", [1, 7, 64, 333, 700, 2048, 4099])
def test_mla_deepseek_shapes(T, q_fp8):
    run(T, Q, KV, q_fp8, seed=T)


@pytest.mark.parametrize("q_fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("q_dim,kv_dim,q_pad,kv_pad,T", [
    (1544, 520, 8, 24, 5),        # ragged chunk counts, separate strided tensors
    (1544, 520, 8, 24, 700),
    (8, 8, 0, 8, 9),              # one chunk per row
    (8, 4104, 16, 0, 650),        # very unequal sides
    (4096, 2048, 16, 8, 611),     # two chunks per thread at large T
    (8192, 8192, 8, 8, 3),        # four chunks per thread
    (32768, 32768, 8, 8, 3),      # the largest rows: eight chunks per thread
    (1544, 520, 8, 24, 2100),     # too wide for one warp at large T
    (1024, 1016, 8, 8, 2100),     # the warp kernel: ragged 4 + 4 chunks per lane
    (8, 8, 0, 8, 2100),           # the warp kernel: one chunk per side
    (248, 1792, 0, 16, 3000),     # the warp kernel: 1 + 7 chunks per lane
    (1280, 768, 8, 8, 2100),      # the warp kernel: 5 + 3 (too wide for a pair)
    (1000, 400, 8, 24, 2100),     # the warp kernel: ragged 2 + 1 chunks per lane
    (1536, 512, 0, 64, 4099),     # the fixed-layout warp kernel, strided rows, ragged T
    (1536, 512, 0, 64, 6081),     # the same, more tokens than one wave of CTAs
    (1024, 1016, 8, 8, 5000),     # the warp kernel in registers, more than one wave
])
def test_mla_shapes_and_strides(q_dim, kv_dim, q_pad, kv_pad, T, q_fp8):
    run(T, q_dim, kv_dim, q_fp8, seed=q_dim + kv_dim + T, q_pad=q_pad, kv_pad=kv_pad)


@pytest.mark.parametrize("q_fp8", [False, True], ids=["bf16", "fp8"])
def test_mla_edge_values(q_fp8):
    """Zero, -0, constant, sparse, tiny and huge rows with eps = 1e-6; then
    eps = 0 on the rows where it is defined in fp32 (no all-zero row, which
    is 0/0, and no row whose squares underflow fp32), among them rows of
    mean square 1: inv is exactly 1 and bf16 ties go to even on both sides."""
    rng = np.random.default_rng(7)
    T, q_dim, kv_dim = 8, 256, 128

    def rows(n):
        x = np.zeros((T, n), np.float32)
        x[1] = -0.0
        x[2] = 1.5
        x[3, ::5] = -2.0
        x[4] = 1e-30 * rng.standard_normal(n)
        x[5] = 3e4 * rng.standard_normal(n)
        x[6] = np.where(np.arange(n) % 2 == 0, 1.0, -1.0)   # mean square 1
        x[7] = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
        return gen.to_bf16_bits(x)

    w_q = gen.to_bf16_bits((1 + 0.5 * rng.standard_normal(q_dim)).astype(np.float32))
    w_kv = gen.to_bf16_bits((-1 + 0.5 * rng.standard_normal(kv_dim)).astype(np.float32))
    d = {"q_c": rows(q_dim), "kv_c": rows(kv_dim), "q_weight": w_q, "kv_weight": w_kv}
    g, o, _ = run(T, q_dim, kv_dim, q_fp8, eps_q=1e-6, eps_kv=1e-6, inputs=d)
    if not q_fp8:
        assert np.all(g["q"][1] & 0x7FFF == 0)          # -0 rows stay zero
        assert np.any(g["q"][1] == 0x8000)
    defined = [2, 3, 5, 6, 7]
    d0 = {"q_c": d["q_c"][defined], "kv_c": d["kv_c"][defined], "q_weight": w_q, "kv_weight": w_kv}
    run(len(defined), q_dim, kv_dim, q_fp8, eps_q=0.0, eps_kv=0.0, inputs=d0)


def test_mla_fp8_q_exact():
    """The q side's scales and codes equal the oracle's bit for bit (the
    exact dynamic-scale arithmetic, as for the per-token norm)."""
    g, o, _ = run(2048, Q, KV, True, seed=11)
    assert np.array_equal(g["q_scale"], o["q_scale"])
    assert np.array_equal(g["q_fp8"], o["q_fp8"])


@pytest.mark.parametrize("q_fp8", [False, True], ids=["bf16", "fp8"])
def test_mla_prefill_full_size_sampled(q_fp8):
    """32768 tokens in the launch configuration the sweep times; the oracle
    checks every 41st token."""
    T = 32768
    d = gen.mla_inputs(T, Q, KV, seed=5)
    g = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-6, q_fp8)
    rows = np.arange(0, T, 41)
    o = parity.oracle_mla(d["q_c"][rows], d["q_weight"], d["kv_c"][rows], d["kv_weight"],
                          1e-6, 1e-6, q_fp8)
    parity.check_mla({k: v[rows] for k, v in g.items()}, o, q_fp8)


def test_mla_bf16_and_fp8_share_the_kv_side():
    """The two variants compute the same kv rows."""
    d = gen.mla_inputs(300, Q, KV, seed=3)
    a = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-5, False)
    b = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-5, True)
    assert np.array_equal(a["kv"], b["kv"])


def test_mla_graph_capture_matches_eager():
    import torch
    import norm_activation_fp8_gb300 as vg
    d = gen.mla_inputs(512, Q, KV, seed=9)
    dev = "cuda"
    qc = torch.from_numpy(d["q_c"].view(np.int16)).to(dev)
    kc = torch.from_numpy(d["kv_c"].view(np.int16)).to(dev)
    qw = torch.from_numpy(d["q_weight"].view(np.int16)).to(dev)
    kw = torch.from_numpy(d["kv_weight"].view(np.int16)).to(dev)
    eager = vg.mla_dual_rms_norm(qc, qw, kc, kw, 1e-6, 1e-6, q_fp8=True)
    s = torch.cuda.Stream()
    q8 = torch.empty(512, Q, dtype=torch.uint8, device=dev)
    sc = torch.empty(512, dtype=torch.float32, device=dev)
    kv = torch.empty(512, KV, dtype=torch.int16, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        vg.vg_fused_mla_dual_rms_norm_per_token_quant(q8, sc, kv, qc, qw, kc, kw, 1e-6, 1e-6)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        vg.vg_fused_mla_dual_rms_norm_per_token_quant(q8, sc, kv, qc, qw, kc, kw, 1e-6, 1e-6)
    q8.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q8, eager[0].view(torch.uint8))
    assert torch.equal(sc, eager[1])
    assert torch.equal(kv, eager[2])
