"""Pins for the oracle: checks against what the E4M3/bf16 definitions, closed
forms, invariants, library routines and exact-arithmetic brute force fix.

Every ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  ``tests/test_oracle_pins.py`` runs them on the committed oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and requires that at least one check fails for each.
"""
from __future__ import annotations

import os
from fractions import Fraction as F

import numpy as np
import torch

import exact

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(vals) -> np.ndarray:
    """float values -> bf16 bits (torch RNE cast; all values used here are
    exactly representable)."""
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(rng, shape, scale=1.0) -> np.ndarray:
    return _bits(rng.standard_normal(shape).astype(np.float32) * scale)


def _weight(rng, H) -> np.ndarray:
    return _bits((1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32))


# ----------------------------------------------------------------- e4m3

def load_e4m3_points():
    pts = []
    with open(os.path.join(GOLDEN, "e4m3_ofp8_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, val, *_ = line.split()
            pts.append((int(code, 16), float(val)))
    return pts


def check_e4m3_spec_points(orc):
    for code, val in load_e4m3_points():
        got = orc.e4m3_decode(np.array([code], np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got), (hex(code), got)
            assert orc.e4m3_encode(np.array([np.nan]))[0] == 0x7F
            continue
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)
        enc = orc.e4m3_encode(np.array([val]))[0]
        assert enc == code, (val, hex(enc), hex(code))


def check_e4m3_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    dec = orc.e4m3_decode(codes)
    nan = np.isnan(dec)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    # positive codes enumerate exactly the format's value set, in order
    assert np.array_equal(dec[:0x7F], exact.E4M3_POS_F64)
    assert np.array_equal(dec[0x80:0xFF], -exact.E4M3_POS_F64)
    assert np.signbit(dec[0x80]) and not np.signbit(dec[0x00])
    enc = orc.e4m3_encode(dec)
    fin = ~nan
    assert np.array_equal(enc[fin], codes[fin])


def check_e4m3_encoder_brute_force(orc):
    vals = exact.E4M3_POS_F64
    mids = (vals[:-1] + vals[1:]) / 2.0
    pts = [vals, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
           np.nextafter(vals, np.inf), np.nextafter(vals, -np.inf),
           np.array([448.0, 460.0, 463.99, 464.0, 464.01, 479.0, 480.0, 1e6, 1e300,
                     2.0 ** -10, 2.0 ** -10 * (1 + 2 ** -40), 2.0 ** -11, 1e-300])]
    rng = np.random.default_rng(7)
    pts.append(np.exp2(rng.uniform(-13, 10, 200_000)))
    v = np.concatenate(pts)
    v = np.concatenate([v, -v])
    got = orc.e4m3_encode(v)
    want = exact.e4m3_nearest_code_vec(v)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(v[i], hex(got[i]), hex(want[i])) for i in bad[:5]]
    # the vectorised search agrees with the plain exhaustive one
    for x in list(mids[::9]) + [460.0, 2.0 ** -10, 0.3, 17.0]:
        assert exact.e4m3_nearest_code(x) == orc.e4m3_encode(np.array([x]))[0], x


def check_e4m3_special_values(orc):
    enc = orc.e4m3_encode(np.array([np.inf, -np.inf, np.nan, -0.0, -1e-30, 1e-30, 0.0]))
    assert list(enc) == [0x7E, 0xFE, 0x7F, 0x80, 0x80, 0x00, 0x00], [hex(c) for c in enc]


# ----------------------------------------------------------------- bf16

def check_bf16_all_patterns(orc):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = orc.bf16_decode(codes)
    ref = exact.bf16_bits_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dec), nan)
    assert np.array_equal(dec[~nan], ref[~nan])
    assert np.array_equal(np.signbit(dec[~nan]), np.signbit(ref[~nan]))
    enc = orc.bf16_encode(dec)
    assert np.array_equal(enc[~nan], codes[~nan])
    assert np.all(np.isnan(exact.bf16_bits_to_f64(enc[nan])))


def check_bf16_encoder_brute_force(orc):
    rng = np.random.default_rng(11)
    vals = exact.BF16_POS_VALUES[:-1]
    mids = (vals[:-1] + vals[1:]) / 2.0   # exact in fp64
    pick = rng.choice(mids.size, 4000, replace=False)
    pts = np.concatenate([
        mids[pick], np.nextafter(mids[pick], np.inf), np.nextafter(mids[pick], -np.inf),
        rng.standard_normal(3000) * np.exp2(rng.integers(-140, 127, 3000)),
        np.array([3.3895313892515355e38, 3.4e38, 1e39, 1e-45, 2.0 ** -134, 2.0 ** -133 * 1.5]),
    ])
    pts = np.concatenate([pts, -pts])
    got = orc.bf16_encode(pts)
    for v, g in zip(pts, got):
        want = exact.bf16_nearest_code(v)
        assert int(g) == want, (v, hex(g), hex(want))
    # library cross-check: torch's float32 -> bfloat16 cast rounds to nearest even
    f32 = (rng.standard_normal(100_000) * np.exp2(rng.integers(-60, 60, 100_000))).astype(np.float32)
    lib = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_encode(f32.astype(np.float64)), lib)


# ------------------------------------------------------------- RMSNorm

def check_norm_constant_row(orc):
    """RMSNorm of a constant row c is c / sqrt(c^2 + eps) * w, which is
    sign(c) * w when eps = 0 (to the rounding of c * (1/|c|))."""
    rng = np.random.default_rng(1)
    H = 256
    w = _weight(rng, H)
    wf = exact.bf16_bits_to_f64(w)
    for c in (1.5, -0.375, 3.0e-3, 96.0):
        x = _bits(np.full((1, H), c))
        c = float(exact.bf16_bits_to_f64(x[0, 0]))
        for eps in (0.0, 1e-6, 1e-2):
            out = orc.fused_add_rms_norm_fp8(x, None, w, eps, STATIC, scale=1.0)
            eps32 = float(np.float32(eps))
            want = c / np.sqrt(c * c + eps32) * wf
            if eps == 0.0:
                np.testing.assert_allclose(out["v"][0], np.sign(c) * wf, rtol=1e-15)
            np.testing.assert_allclose(out["v"][0], want, rtol=1e-14)


def check_norm_h1_closed_form(orc):
    rng = np.random.default_rng(2)
    x = _rand_bf16(rng, (64, 1))
    res = _rand_bf16(rng, (64, 1))
    w = _bits([0.8125])
    out = orc.fused_add_rms_norm_fp8(x, res, w, 1e-3, STATIC, scale=0.5)
    r = exact.bf16_bits_to_f64(out["residual_out"])[:, 0]
    eps32 = float(np.float32(1e-3))
    want = r / np.sqrt(r * r + eps32) * 0.8125 / 0.5
    np.testing.assert_allclose(out["v"][:, 0], want, rtol=1e-14)


def check_norm_invariants(orc):
    """eps = 0: the row's RMS of y/w is exactly 1 (up to fp64 rounding), and
    scaling the input by 2 (exact in bf16) leaves y unchanged bit for bit."""
    rng = np.random.default_rng(3)
    T, H = 8, 384
    x = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    wf = exact.bf16_bits_to_f64(w)
    out = orc.fused_add_rms_norm_fp8(x, None, w, 0.0, STATIC, scale=1.0)
    y_over_w = out["v"] / wf
    np.testing.assert_allclose(np.sqrt(np.mean(y_over_w ** 2, axis=1)), 1.0, rtol=1e-13)
    # y_j / w_j is proportional to x_j within a row
    xf = exact.bf16_bits_to_f64(x)
    ratio = y_over_w / xf
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones_like(ratio), rtol=1e-13)
    x2 = _bits(2.0 * xf)
    out2 = orc.fused_add_rms_norm_fp8(x2, None, w, 0.0, STATIC, scale=1.0)
    assert np.array_equal(out2["v"], out["v"])


def check_norm_residual_add_library(orc):
    """residual_out = bf16(x + residual): a float32 add followed by torch's RNE
    cast gives the correctly rounded sum of two bf16 numbers; the normalised
    row is that stored residual (plain variant run on residual_out)."""
    rng = np.random.default_rng(4)
    T, H = 16, 512
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-8, 8, (T, H))))
    res = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    out = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, PER_TOKEN)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    rt = torch.from_numpy(res.view(np.int16)).view(torch.bfloat16).float()
    lib = (xt + rt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out["residual_out"], lib)
    plain = orc.fused_add_rms_norm_fp8(out["residual_out"], None, w, 1e-5, PER_TOKEN)
    assert np.array_equal(plain["q"], out["q"]) and np.array_equal(plain["scale"], out["scale"])
    # a zero residual changes nothing against the plain variant
    zero = np.zeros_like(res)
    pz = orc.fused_add_rms_norm_fp8(x, zero, w, 1e-5, PER_TOKEN)
    p0 = orc.fused_add_rms_norm_fp8(x, None, w, 1e-5, PER_TOKEN)
    assert np.array_equal(pz["q"], p0["q"]) and np.array_equal(pz["v"], p0["v"])
    assert np.array_equal(pz["residual_out"], x)


def check_norm_brute_force(orc):
    """Tiny random rows against exact rational arithmetic (60-digit sqrt)."""
    rng = np.random.default_rng(5)
    floor = orc.amax_floor()
    for H, mode, G in ((8, STATIC, 0), (16, PER_TOKEN, 0), (16, PER_GROUP, 8),
                       (12, PER_GROUP, 4), (1, PER_TOKEN, 0)):
        T = 3
        x = _rand_bf16(rng, (T, H))
        res = _rand_bf16(rng, (T, H), scale=3.0)
        w = _weight(rng, H)
        s_static = 0.0625 if mode == STATIC else None
        for residual in (res, None):
            out = orc.fused_add_rms_norm_fp8(x, residual, w, 1e-5, mode, G or 128,
                                             scale=s_static)
            for t in range(T):
                ex = exact.exact_norm_row(x[t], None if residual is None else residual[t],
                                          w, 1e-5, mode, G, s_static, floor)
                if residual is not None:
                    assert list(out["residual_out"][t]) == ex["residual_out"]
                s_row = out["scale"] if mode == STATIC else np.atleast_1d(out["scale"][t])
                assert np.array_equal(s_row, ex["scale"]), (s_row, ex["scale"])
                np.testing.assert_allclose(out["v"][t], [float(v) for v in ex["v"]], rtol=1e-13)
                assert list(out["q"][t]) == ex["q"], (H, mode, t)


# ------------------------------------------------------------- quant modes

def check_per_token_max_code(orc):
    """Dynamic per-token: every row reaches |q| = 448 (code 0x7E/0xFE), the
    scale is fp32(amax/448), and dequantisation q*s is within half an E4M3
    step of y."""
    rng = np.random.default_rng(6)
    T, H = 32, 640
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-6, 6, (T, 1))))
    res = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    out = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, PER_TOKEN)
    assert np.all(np.max(out["q"] & 0x7F, axis=1) == 0x7E)
    ref = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, STATIC, scale=1.0)
    y = ref["v"]
    amax = np.max(np.abs(y), axis=1)
    np.testing.assert_allclose(out["scale"], (amax / 448.0).astype(np.float32), rtol=1e-7)
    deq = exact.E4M3_POS_F64[out["q"] & 0x7F] * np.where(out["q"] & 0x80, -1, 1)
    deq = deq * out["scale"][:, None]
    step = np.maximum(np.abs(y) / 8.0, 2.0 ** -9 * out["scale"][:, None])
    assert np.all(np.abs(deq - y) <= step * 0.5 + 1e-12 * np.abs(y))


def check_per_group_layout(orc):
    """Per-group: each group's scale is fp32(max|y| over its G columns / 448),
    stored at [t, g]; every group reaches 448; G = H equals per-token; and a
    static run with the per-token scale of each row gives the same codes."""
    rng = np.random.default_rng(8)
    T, H = 6, 512
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-4, 4, (1, H))))
    res = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    ref = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, STATIC, scale=1.0)
    for G in (64, 128):
        out = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, PER_GROUP, G)
        assert out["scale"].shape == (T, H // G)
        amax = np.max(np.abs(ref["v"]).reshape(T, H // G, G), axis=2)
        np.testing.assert_allclose(out["scale"], (amax / 448.0).astype(np.float32), rtol=1e-7)
        assert np.all(np.max((out["q"] & 0x7F).reshape(T, H // G, G), axis=2) == 0x7E)
    full = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, PER_GROUP, H)
    tok = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, PER_TOKEN)
    assert np.array_equal(full["q"], tok["q"])
    assert np.array_equal(full["scale"].reshape(T), tok["scale"])
    for t in range(T):
        st = orc.fused_add_rms_norm_fp8(x[t:t + 1], res[t:t + 1], w, 1e-5, STATIC,
                                        scale=tok["scale"][t])
        assert np.array_equal(st["q"][0], tok["q"][t])


def check_zero_row_and_saturation(orc):
    H = 256
    w = _bits(np.ones(H))
    z = np.zeros((2, H), np.uint16)
    out = orc.fused_add_rms_norm_fp8(z, z, w, 1e-5, PER_TOKEN)
    assert np.all(out["q"] == 0)
    assert np.all(out["scale"] == np.float32(orc.amax_floor() / 448.0))
    rng = np.random.default_rng(9)
    x = _rand_bf16(rng, (2, H))
    sat = orc.fused_add_rms_norm_fp8(x, None, w, 1e-5, STATIC, scale=1e-6)
    v = sat["v"]
    big = np.abs(v) >= 448
    assert big.mean() > 0.9
    assert np.all((sat["q"][big] & 0x7F) == 0x7E)
    assert np.array_equal(sat["q"][big] >> 7, np.signbit(v[big]).astype(np.uint8))


# ------------------------------------------------------------------ SiLU

def check_silu_closed_forms(orc):
    """silu(0) = 0; silu(g) = g for g >= 40 (e^-40 is below half an fp64 ulp);
    silu(g) - silu(-g) = g; silu(g) -> -0 for g <= -745; silu(g)*u against
    scipy's logistic function."""
    from scipy.special import expit
    I = 8
    g = np.array([0.0, 40.0, 64.0, 1024.0, -746.0, -1024.0, 2.5, -2.5])
    u = np.array([1.0, 1.0, 0.5, 1.0, 1.0, 1.0, 1.0, 1.0])
    gu = _bits(np.concatenate([g, u])[None, :])
    out = orc.silu_mul_fp8(gu, STATIC, scale=1.0)
    v = out["v"][0]
    assert v[0] == 0.0 and v[1] == 40.0 and v[2] == 32.0 and v[3] == 1024.0
    assert v[4] == 0.0 and np.signbit(v[4]) and out["q"][0, 4] == 0x80
    assert abs((v[6] - v[7]) - 2.5) <= 1e-15
    rng = np.random.default_rng(10)
    T, I = 4, 512
    gate = rng.standard_normal((T, I)) * 4
    up = rng.standard_normal((T, I))
    gu = _bits(np.concatenate([gate, up], axis=1))
    gf = exact.bf16_bits_to_f64(gu[:, :I])
    uf = exact.bf16_bits_to_f64(gu[:, I:])
    out = orc.silu_mul_fp8(gu, STATIC, scale=1.0)
    np.testing.assert_allclose(out["v"], gf * expit(gf) * uf, rtol=1e-14, atol=1e-300)


def check_silu_brute_force(orc):
    rng = np.random.default_rng(12)
    floor = orc.amax_floor()
    for I, mode, G in ((8, STATIC, 0), (16, PER_TOKEN, 0), (16, PER_GROUP, 8)):
        T = 3
        gu = _rand_bf16(rng, (T, 2 * I), scale=3.0)
        s_static = 0.1 if mode == STATIC else None
        out = orc.silu_mul_fp8(gu, mode, G or 128, scale=s_static)
        for t in range(T):
            ex = exact.exact_silu_row(gu[t], mode, G, s_static, floor)
            s_row = out["scale"] if mode == STATIC else np.atleast_1d(out["scale"][t])
            assert np.array_equal(s_row, ex["scale"]), (s_row, ex["scale"])
            np.testing.assert_allclose(out["v"][t], [float(v) for v in ex["v"]], rtol=1e-13)
            assert list(out["q"][t]) == ex["q"], (I, mode, t)


def check_silu_modes(orc):
    """SiLU per-token rows reach 448; per-group G = I equals per-token."""
    rng = np.random.default_rng(13)
    T, I = 8, 256
    gu = _rand_bf16(rng, (T, 2 * I))
    tok = orc.silu_mul_fp8(gu, PER_TOKEN)
    assert np.all(np.max(tok["q"] & 0x7F, axis=1) == 0x7E)
    full = orc.silu_mul_fp8(gu, PER_GROUP, I)
    assert np.array_equal(full["q"], tok["q"])
    ref = orc.silu_mul_fp8(gu, STATIC, scale=1.0)
    G = 128
    grp = orc.silu_mul_fp8(gu, PER_GROUP, G)
    amax = np.max(np.abs(ref["v"]).reshape(T, I // G, G), axis=2)
    np.testing.assert_allclose(grp["scale"], (amax / 448.0).astype(np.float32), rtol=1e-7)


# ------------------------------------------------------- bf16 rms_norm


def check_rms_norm_bf16_closed_forms(orc):
    """With eps = 0 a constant row c gives y = sign(c) * w, so the bf16 output
    is w with c's sign; a row holding one value a among H = 4 gives
    y = sign(a) * 2 * w at that column and a signed zero elsewhere; with
    eps > 0 a constant row gives c / sqrt(c^2 + eps) * w."""
    rng = np.random.default_rng(21)
    H = 64
    w = _weight(rng, H)
    wf = exact.bf16_bits_to_f64(w)
    for c in (1.5, -0.375, 3.0e-3, -96.0):
        x = _bits(np.full((1, H), c))
        out = orc.rms_norm_bf16(x, w, 0.0)
        want = w ^ np.uint16(0x8000) if c < 0 else w
        assert np.array_equal(out["out"][0], want), c
        cb = float(exact.bf16_bits_to_f64(x[0, 0]))
        for eps in (1e-6, 0.5):
            out = orc.rms_norm_bf16(x, w, eps)
            eps32 = F(float(np.float32(eps)))
            inv = 1 / exact._sqrt(F(cb) * F(cb) + eps32)
            y = [F(cb) * inv * F(float(wj)) for wj in wf]
            assert list(out["out"][0]) == [exact.bf16_nearest_code(v) for v in y], (c, eps)
    w4 = _bits([0.75, -1.25, 3.0, -0.5])
    for a, j in ((2.5, 0), (-0.125, 2), (7.0, 3)):
        x = np.zeros((1, 4), np.uint16)
        x[0, j] = _bits([a])[0]
        out = orc.rms_norm_bf16(x, w4, 0.0)["out"][0]
        w4f = exact.bf16_bits_to_f64(w4)
        for k in range(4):
            if k == j:
                assert out[k] == _bits([np.sign(a) * 2.0 * w4f[k]])[0], (a, j)
            else:
                assert out[k] == (0x8000 if w4f[k] < 0 else 0x0000), (a, j, k)


def check_rms_norm_bf16_invariants(orc):
    """eps = 0: the RMS of y / w is 1, y / w is proportional to x within a row,
    and doubling the input (exact in bf16) changes nothing."""
    rng = np.random.default_rng(22)
    T, H = 6, 192
    x = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    wf = exact.bf16_bits_to_f64(w)
    out = orc.rms_norm_bf16(x, w, 0.0)
    y_over_w = out["y"] / wf
    np.testing.assert_allclose(np.sqrt(np.mean(y_over_w ** 2, axis=1)), 1.0, rtol=1e-13)
    ratio = y_over_w / exact.bf16_bits_to_f64(x)
    np.testing.assert_allclose(ratio, ratio[:, :1] * np.ones_like(ratio), rtol=1e-13)
    out2 = orc.rms_norm_bf16(_bits(2.0 * exact.bf16_bits_to_f64(x)), w, 0.0)
    assert np.array_equal(out2["out"], out["out"]) and np.array_equal(out2["y"], out["y"])


def check_rms_norm_bf16_brute_force(orc):
    """Tiny random rows against exact rational arithmetic: every output is
    the nearest-even bf16 of the exact normalised value."""
    rng = np.random.default_rng(23)
    for H, eps in ((1, 1e-5), (8, 1e-5), (16, 0.25), (24, 1e-6)):
        T = 3
        x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-6, 6, (T, H))))
        w = _weight(rng, H)
        out = orc.rms_norm_bf16(x, w, eps)
        for t in range(T):
            ex = exact.exact_norm_row(x[t], None, w, eps, STATIC, 0, 1.0, 1e-10)
            assert list(out["out"][t]) == [exact.bf16_nearest_code(v) for v in ex["y"]], (H, t)
            np.testing.assert_allclose(out["y"][t], [float(v) for v in ex["y"]], rtol=1e-13)


# ------------------------------------------------------------------ NVFP4


def load_e2m1_points():
    pts = []
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                code, val, *_ = line.split()
                pts.append((int(code, 16), float(val)))
    return pts


def check_e2m1_codec(orc):
    """The OCP MX spec's E2M1 points; all 16 codes decode to the value set
    enumerated as significand x 2^k and round-trip; the encoder equals an
    exhaustive nearest-value search (ties to the even code, saturation at 6)
    on every midpoint, midpoint +- 1 ulp and random values of both signs."""
    for code, val in load_e2m1_points():
        got = orc.e2m1_decode(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)
        assert orc.e2m1_encode(np.array([val]))[0] == code, (val, code)
    codes = np.arange(16, dtype=np.uint8)
    dec = orc.e2m1_decode(codes)
    want = [float(v) for v in exact.E2M1_POS]
    assert list(dec[:8]) == want and list(-dec[8:]) == want
    assert np.array_equal(orc.e2m1_encode(dec), codes)
    pos = [float(v) for v in exact.E2M1_POS]
    mids = [(a + b) / 2 for a, b in zip(pos, pos[1:])] + [7.0, 6.0, 100.0]
    rng = np.random.default_rng(29)
    probe = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 100),
                            rng.uniform(0, 8, 2000)])
    probe = np.concatenate([probe, -probe])
    got = orc.e2m1_encode(probe)
    assert list(got) == [exact.e2m1_nearest_code(float(p)) for p in probe]


def check_nvfp4_rows(orc):
    """Tiny rows of both ops against exact rationals: E4M3 block scale codes
    of gs*amax/6, E2M1 codes of y*gs/scale, two codes a byte (column 2i in
    the low nibble); an all-zero block gives scale code 0 and zero codes."""
    rng = np.random.default_rng(30)
    floor = orc.amax_floor()
    T, H = 3, 48
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-3, 3, (T, H))))
    x[1, 16:32] = 0                                   # an all-zero block
    res = _rand_bf16(rng, (T, H))
    res[1, 16:32] = 0
    w = _weight(rng, H)
    gs = 448.0 * 6.0 / 5.0
    out = orc.fused_add_rms_norm_nvfp4(x, res, w, 1e-5, gs)
    for t in range(T):
        ex = exact.exact_norm_row(x[t], res[t], w, 1e-5, STATIC, 0, 1.0, floor)
        sf, v, codes = exact.exact_nvfp4(ex["y"], gs)
        assert list(out["sf"][t]) == sf, t
        lo, hi = out["q4"][t] & 0xF, out["q4"][t] >> 4
        got = np.empty(H, np.int64)
        got[0::2], got[1::2] = lo, hi
        assert list(got) == codes, t
        np.testing.assert_allclose(out["v"][t], [float(z) for z in v], rtol=1e-13)
    assert out["sf"][1, 1] == 0 and np.all(out["q4"][1, 8:16] == 0)
    gu = _rand_bf16(rng, (T, 2 * H), scale=2.0)
    sout = orc.silu_mul_nvfp4(gu, 3.0)
    for t in range(T):
        ex = exact.exact_silu_row(gu[t], STATIC, 0, 1.0, floor)
        sf, v, codes = exact.exact_nvfp4(ex["y"], 3.0)
        got = np.empty(H, np.int64)
        got[0::2], got[1::2] = sout["q4"][t] & 0xF, sout["q4"][t] >> 4
        assert list(sout["sf"][t]) == sf and list(got) == codes, t


# ------------------------------------- UE8M0 / column-major group scales

UE8M0, COL_MAJOR = 0x100, 0x200


def check_group_scale_options(orc):
    """UE8M0 scales are the powers of two that bracket each group's amax/448
    (exact rationals on tiny rows, codes included, both ops); the
    column-major layout holds the row-major scales transposed, T padded to a
    multiple of 4 with the padding left alone; the options need per-group."""
    rng = np.random.default_rng(28)
    floor = orc.amax_floor()
    T, H, G = 3, 16, 8
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-5, 5, (T, H))))
    w = _weight(rng, H)
    out = orc.fused_add_rms_norm_fp8(x, None, w, 1e-5, PER_GROUP | UE8M0, G)
    for t in range(T):
        ex = exact.exact_norm_row(x[t], None, w, 1e-5, PER_GROUP, G, None, floor, ue8m0=True)
        assert np.array_equal(out["scale"][t], ex["scale"]), t
        assert list(out["q"][t]) == ex["q"], t
    s = out["scale"].astype(np.float64)
    assert np.all(np.exp2(np.round(np.log2(s))) == s)          # powers of two
    gu = _rand_bf16(rng, (T, 2 * H), scale=3.0)
    sout = orc.silu_mul_fp8(gu, PER_GROUP | UE8M0, G)
    for t in range(T):
        ex = exact.exact_silu_row(gu[t], PER_GROUP, G, None, floor, ue8m0=True)
        assert np.array_equal(sout["scale"][t], ex["scale"]) and list(sout["q"][t]) == ex["q"], t
    # layout: a larger T so that the padding is visible (T4 = 8 for T = 5)
    T = 5
    d = _rand_bf16(rng, (T, 256))
    w = _weight(rng, 256)
    for extra in (0, UE8M0):
        row = orc.fused_add_rms_norm_fp8(d, None, w, 1e-5, PER_GROUP | extra, 64)
        col = orc.fused_add_rms_norm_fp8(d, None, w, 1e-5, PER_GROUP | extra | COL_MAJOR, 64)
        assert col["scale"].shape == (4, 8)
        assert np.array_equal(col["scale"][:, :T], row["scale"].T)
        assert np.all(col["scale"][:, T:] == -1.0)              # padding not written
        assert np.array_equal(col["q"], row["q"])
    # an all-zero group: the floored amax, so the power of two at A_MIN/448
    z = d.copy()
    z[1, :64] = 0
    zo = orc.fused_add_rms_norm_fp8(z, None, w, 1e-5, PER_GROUP | UE8M0, 64)
    assert zo["scale"][1, 0] == np.float32(float(exact.pow2_at_least(F(floor) / 448)))
    assert np.all(zo["q"][1, :64] == 0)
    for bad in (STATIC | UE8M0, PER_TOKEN | COL_MAJOR, PER_GROUP | 0x400):
        try:
            orc.fused_add_rms_norm_fp8(d, None, w, 1e-5, bad, 64, scale=1.0)
        except ValueError:
            continue
        raise AssertionError(f"mode {bad:#x} accepted")


# ----------------------------------------------------- act padding


def check_norm_pad(orc):
    """The padded tail is zero; the first H columns are the bf16 rms_norm of
    the stored residual (pinned above); residual_out is torch's bf16 add; the
    plain variant equals the bf16 rms_norm of x; padded = H adds nothing."""
    rng = np.random.default_rng(24)
    T, H, Hp = 5, 360, 384
    x = _rand_bf16(rng, (T, H), scale=np.exp2(rng.integers(-4, 4, (T, H))))
    res = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    out = orc.fused_add_rms_norm_pad(x, res, w, 1e-6, Hp)
    assert out["out"].shape == (T, Hp)
    assert np.all(out["out"][:, H:] == 0)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    rt = torch.from_numpy(res.view(np.int16)).view(torch.bfloat16).float()
    lib = (xt + rt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out["residual_out"], lib)
    ref = orc.rms_norm_bf16(out["residual_out"], w, 1e-6)
    assert np.array_equal(out["out"][:, :H], ref["out"])
    plain = orc.fused_add_rms_norm_pad(x, None, w, 1e-6, Hp)
    assert plain["residual_out"] is None
    assert np.array_equal(plain["out"][:, :H], orc.rms_norm_bf16(x, w, 1e-6)["out"])
    big = orc.fused_add_rms_norm_pad(x, res, w, 0.5, Hp)  # an eps that matters
    assert np.array_equal(big["out"][:, :H], orc.rms_norm_bf16(big["residual_out"], w, 0.5)["out"])
    assert not np.array_equal(big["out"], out["out"])
    same = orc.fused_add_rms_norm_pad(x, res, w, 1e-6, H)
    assert np.array_equal(same["out"], out["out"][:, :H])
    for t in range(2):
        ex = exact.exact_norm_row(x[t], res[t], w, 1e-6, STATIC, 0, 1.0, 1e-10)
        assert list(out["out"][t, :H]) == [exact.bf16_nearest_code(v) for v in ex["y"]]


# ------------------------------------------------------- QK norm + RoPE


def _qk_case(rng, T, Hq, Hkv, D):
    qkv = _rand_bf16(rng, (T, (Hq + 2 * Hkv) * D), scale=np.exp2(rng.integers(-3, 3, (T, (Hq + 2 * Hkv) * D))))
    return qkv, _weight(rng, D), _bits(0.5 + rng.random(D))


def check_qk_norm_rope_rotations(orc):
    """Cache rows of exact rotations: the identity gives the pinned bf16
    rms_norm of every head; a quarter turn swaps the pair members with one
    sign flipped; a half turn negates; V columns are never touched."""
    rng = np.random.default_rng(25)
    T, Hq, Hkv, D = 3, 3, 2, 16
    qkv, qw, kw = _qk_case(rng, T, Hq, Hkv, D)
    cache = np.zeros((3, D), np.float32)
    cache[0, :D // 2] = 1.0                     # cos 1, sin 0
    cache[1, D // 2:] = 1.0                     # cos 0, sin 1
    cache[2, :D // 2] = -1.0                    # cos -1, sin 0
    nq = Hq * D
    heads = qkv[:, :(Hq + Hkv) * D].reshape(T, Hq + Hkv, D)
    ref = np.empty_like(heads)
    for h in range(Hq + Hkv):
        ref[:, h] = orc.rms_norm_bf16(heads[:, h], qw if h < Hq else kw, 1e-6)["out"]
    sign = np.uint16(0x8000)
    for neox in (True, False):
        for row in range(3):
            out = orc.qk_norm_rope(qkv, qw, kw, cache, np.full(T, row), Hq, Hkv, D, 1e-6, neox)
            got = out["qkv"][:, :(Hq + Hkv) * D].reshape(T, Hq + Hkv, D)
            if row == 0:
                want = ref
            elif row == 2:
                want = ref ^ sign
            else:
                want = np.empty_like(ref)
                a = np.arange(D // 2) if neox else 2 * np.arange(D // 2)
                b = a + D // 2 if neox else a + 1
                want[..., a] = ref[..., b] ^ sign
                want[..., b] = ref[..., a]
            assert np.array_equal(got, want), (neox, row)
            assert np.array_equal(out["qkv"][:, (Hq + Hkv) * D:], qkv[:, (Hq + Hkv) * D:])
            assert out["qkv"][:, nq:].shape[1] == 2 * Hkv * D


def check_qk_norm_rope_pairings(orc):
    """neox on a head equals gptj on the same head with its columns
    interleaved (column i -> 2i, column i + D/2 -> 2i + 1), weights likewise."""
    rng = np.random.default_rng(26)
    T, Hq, Hkv, D = 4, 2, 1, 16
    qkv, qw, kw = _qk_case(rng, T, Hq, Hkv, D)
    cache = (rng.random((5, D)) * 2 - 1).astype(np.float32)
    pos = np.array([4, 0, 2, 2])
    perm = np.empty(D, np.int64)
    perm[2 * np.arange(D // 2)] = np.arange(D // 2)
    perm[2 * np.arange(D // 2) + 1] = np.arange(D // 2) + D // 2   # gptj column k holds neox column perm[k]
    heads = qkv.reshape(T, Hq + 2 * Hkv, D)
    qkv_g = heads[:, :, perm].reshape(T, -1)
    a = orc.qk_norm_rope(qkv, qw, kw, cache, pos, Hq, Hkv, D, 1e-5, True)["qkv"]
    b = orc.qk_norm_rope(qkv_g, qw[perm], kw[perm], cache, pos, Hq, Hkv, D, 1e-5, False)["qkv"]
    assert np.array_equal(a.reshape(T, -1, D)[:, :, perm], b.reshape(T, -1, D))


def check_qk_norm_rope_brute_force(orc):
    """Tiny heads against exact rational arithmetic (fp32 cache values taken
    exactly, 60-digit sqrt): every output is the nearest-even bf16."""
    rng = np.random.default_rng(27)
    T, Hq, Hkv, D = 2, 1, 1, 8
    for neox in (True, False):
        qkv, qw, kw = _qk_case(rng, T, Hq, Hkv, D)
        cache = (rng.random((4, D)) * 2 - 1).astype(np.float32)
        pos = np.array([3, 1])
        out = orc.qk_norm_rope(qkv, qw, kw, cache, pos, Hq, Hkv, D, 1e-4, neox)["qkv"]
        for t in range(T):
            for h in range(Hq + Hkv):
                x = [F(float(v)) for v in exact.bf16_bits_to_f64(qkv[t, h * D:(h + 1) * D])]
                w = [F(float(v)) for v in exact.bf16_bits_to_f64(qw if h < Hq else kw)]
                inv = 1 / exact._sqrt(sum(v * v for v in x) / D + F(float(np.float32(1e-4))))
                y = [x[j] * inv * w[j] for j in range(D)]
                o = [None] * D
                for i in range(D // 2):
                    a, b = (i, i + D // 2) if neox else (2 * i, 2 * i + 1)
                    c, sn = F(float(cache[pos[t], i])), F(float(cache[pos[t], D // 2 + i]))
                    o[a] = y[a] * c - y[b] * sn
                    o[b] = y[b] * c + y[a] * sn
                assert list(out[t, h * D:(h + 1) * D]) == [exact.bf16_nearest_code(v) for v in o], \
                    (neox, t, h)


# ------------------------------------------------------- NaN and infinity
#
# The reading for non-finite inputs: every formula is evaluated in IEEE
# arithmetic as written, and the amax of a row or group is the largest |y|
# among its non-NaN elements (a NaN never wins the comparison; 0 when there
# is none), floored at A_MIN as usual.  Consequences fixed here without the
# oracle's own arithmetic:
#   a NaN anywhere in r makes sum(r^2), inv and every y NaN: every code 0x7F,
#     every dynamic scale fp32(A_MIN / 448);
#   an infinity in r (and no NaN) makes sum(r^2) = inf and inv = 0: y = +-0
#     (the sign of r w) at finite r and NaN at the infinite one, so the codes
#     are 0x00 / 0x80 and 0x7F there, and every dynamic scale is the floor;
#   eps = 0 with an all-zero row: inv = 1/0 = inf and y = 0 * inf = NaN;
#   a NaN in the weight turns only its own column into NaN;
#   SiLU: silu(g) u with a NaN operand, or silu(-inf) = -inf / inf, is NaN
#     (code 0x7F, left out of the amax); an infinite a saturates to +-448
#     under a static scale and makes its row's or group's dynamic scale
#     +inf, so its own code is 0x7F (inf / inf) and its finite neighbours
#     code as +-0.

_NAN16, _PINF16, _NINF16 = 0x7FC0, 0x7F80, 0xFF80


def _is_nan16(b):
    b = np.asarray(b, np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def check_nonfinite_norm(orc):
    rng = np.random.default_rng(31)
    T, H, G = 6, 256, 128
    x = _rand_bf16(rng, (T, H))
    res = _rand_bf16(rng, (T, H))
    w = _weight(rng, H)
    x[0, 5] = _NAN16                        # NaN in x
    x[1, 7] = _PINF16                       # +inf in x
    res[2, 200] = _NINF16                   # -inf in the residual
    x[3, 9], res[3, 9] = _PINF16, _NINF16   # inf + (-inf) = NaN
    floor = np.float32(orc.amax_floor() / 448.0)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    rt = torch.from_numpy(res.view(np.int16)).view(torch.bfloat16).float()
    lib = (xt + rt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wf = exact.bf16_bits_to_f64(w)
    control = {m: orc.fused_add_rms_norm_fp8(x[5:6], res[5:6], w, 1e-5, m, G, scale=0.05)
               for m in (STATIC, PER_TOKEN, PER_GROUP)}
    for mode in (STATIC, PER_TOKEN, PER_GROUP, PER_GROUP | 0x100):
        out = orc.fused_add_rms_norm_fp8(x, res, w, 1e-5, mode, G, scale=0.05)
        ro = out["residual_out"]
        nan = _is_nan16(ro)
        assert np.array_equal(np.argwhere(nan), [[0, 5], [3, 9]])
        assert np.array_equal(ro[~nan], lib[~nan])
        assert ro[1, 7] == _PINF16 and ro[2, 200] == _NINF16
        q = out["q"]
        # the floored scale: fp32(A_MIN / 448), or the power of two above it
        fl = np.float32(exact.pow2_at_least(F(float(orc.amax_floor())) / 448)) if mode & 0x100 \
            else floor
        for t in (0, 3):  # NaN rows
            assert np.all(q[t] == 0x7F), (mode, t)
            if mode != STATIC:
                assert np.all(out["scale"][t] == fl), (mode, t)
        if mode & 0x100:
            continue  # an infinite amax has no power-of-two scale; NaN rows only
        for t, j in ((1, 7), (2, 200)):  # infinite rows
            assert q[t, j] == 0x7F
            r = exact.bf16_bits_to_f64(ro[t])
            sign = np.signbit(r * wf).astype(np.uint8) << 7
            keep = np.arange(H) != j
            assert np.array_equal(q[t, keep], sign[keep]), (mode, t)
            if mode != STATIC:
                assert np.all(out["scale"][t] == floor), (mode, t)
        if mode in control:  # a finite row next to them is unaffected
            assert np.array_equal(q[5], control[mode]["q"][0])
            if mode != STATIC:
                assert np.array_equal(out["scale"][5], control[mode]["scale"][0])
    # a NaN weight column: 0x7F in that column only; elsewhere as with w = 0 there
    wn, w0 = w.copy(), w.copy()
    wn[3], w0[3] = _NAN16, 0
    for mode in (STATIC, PER_TOKEN, PER_GROUP):
        a = orc.fused_add_rms_norm_fp8(x[4:6], res[4:6], wn, 1e-5, mode, G, scale=0.05)
        b = orc.fused_add_rms_norm_fp8(x[4:6], res[4:6], w0, 1e-5, mode, G, scale=0.05)
        assert np.all(a["q"][:, 3] == 0x7F)
        keep = np.arange(H) != 3
        assert np.array_equal(a["q"][:, keep], b["q"][:, keep]), mode
        if mode != STATIC:
            assert np.array_equal(a["scale"], b["scale"]), mode
    # eps = 0 with an all-zero row: 0 * (1/0) is NaN everywhere
    z = np.zeros((1, H), np.uint16)
    for mode in (STATIC, PER_TOKEN, PER_GROUP):
        out = orc.fused_add_rms_norm_fp8(z, None, w, 0.0, mode, G, scale=0.05)
        assert np.all(out["q"] == 0x7F), mode
        if mode != STATIC:
            assert np.all(out["scale"] == floor), mode


def check_nonfinite_silu(orc):
    rng = np.random.default_rng(32)
    T, I, G = 6, 256, 128
    gu = _rand_bf16(rng, (T, 2 * I))
    marks = {0: (4, _NAN16, None),              # NaN gate
             1: (10, _bits([1.0])[0], _PINF16),  # silu(1) * inf = +inf
             2: (20, _PINF16, _bits([-1.5])[0]), # silu(inf) * -1.5 = -inf
             3: (30, _NINF16, None),             # silu(-inf) = -inf / inf = NaN
             4: (40, None, _NAN16)}              # NaN up
    zeroed = gu.copy()
    for t, (j, g, u) in marks.items():
        if g is not None:
            gu[t, j] = g
        if u is not None:
            gu[t, I + j] = u
        zeroed[t, j] = zeroed[t, I + j] = 0     # a_j = 0 in the reference row
    nan_rows, inf_rows = (0, 3, 4), (1, 2)
    for mode in (STATIC, PER_TOKEN, PER_GROUP, PER_GROUP | 0x100):
        out = orc.silu_mul_fp8(gu, mode, G, scale=0.1)
        ref = orc.silu_mul_fp8(zeroed, mode, G, scale=0.1)
        q, rq = out["q"], ref["q"]
        for t in range(T):
            j = marks[t][0] if t in marks else None
            keep = np.arange(I) != j if j is not None else np.ones(I, bool)
            if t in inf_rows and mode & 0x100:
                continue  # an infinite amax has no power-of-two scale
            if mode == STATIC:
                assert np.array_equal(q[t, keep], rq[t, keep]), (mode, t)
                if t in nan_rows:
                    assert q[t, j] == 0x7F
                elif t in inf_rows:
                    assert q[t, j] == (0x7E if t == 1 else 0xFE)
                continue
            srow = out["scale"][t] if mode == PER_TOKEN else out["scale"][t]
            rrow = ref["scale"][t]
            if t in nan_rows or t == 5:
                assert np.array_equal(srow, rrow), (mode, t)
                assert np.array_equal(q[t, keep], rq[t, keep]), (mode, t)
                if j is not None:
                    assert q[t, j] == 0x7F
                continue
            # an infinite activation: its row (per-token) or group gets scale inf
            assert q[t, j] == 0x7F
            width = I if mode == PER_TOKEN else G
            g0 = j // width
            cols = np.arange(g0 * width, (g0 + 1) * width)
            cols = cols[cols != j]
            sign = (np.signbit(ref["v"][t, cols]).astype(np.uint8) << 7)
            assert np.array_equal(q[t, cols], sign), (mode, t)
            if mode == PER_TOKEN:
                assert np.isposinf(srow)
            else:
                assert np.isposinf(srow[g0])
                other = np.arange(I // G) != g0
                assert np.array_equal(srow[other], rrow[other])
                rest = np.ones(I, bool)
                rest[g0 * G:(g0 + 1) * G] = False
                assert np.array_equal(q[t, rest], rq[t, rest])


ALL_CHECKS = [
    check_e4m3_spec_points, check_e4m3_all_codes, check_e4m3_encoder_brute_force,
    check_e4m3_special_values, check_bf16_all_patterns, check_bf16_encoder_brute_force,
    check_norm_constant_row, check_norm_h1_closed_form, check_norm_invariants,
    check_norm_residual_add_library, check_norm_brute_force, check_per_token_max_code,
    check_per_group_layout, check_zero_row_and_saturation, check_silu_closed_forms,
    check_silu_brute_force, check_silu_modes, check_rms_norm_bf16_closed_forms,
    check_rms_norm_bf16_invariants, check_rms_norm_bf16_brute_force, check_norm_pad,
    check_qk_norm_rope_rotations, check_qk_norm_rope_pairings, check_qk_norm_rope_brute_force,
    check_group_scale_options, check_e2m1_codec, check_nvfp4_rows,
    check_nonfinite_norm, check_nonfinite_silu,
]
