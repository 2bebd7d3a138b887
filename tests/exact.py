"""Exact-arithmetic brute force used to pin the oracle (test helper).

Nothing here is taken from the oracle: the value sets of bf16 and e4m3 are
enumerated from the formats' definitions (significand times a power of two,
or numpy's own float32 view of bf16 bits), nearest values are found by
exhaustive search with exact rational comparisons, and the row computations
use Python ``fractions`` plus ``decimal`` square roots and exponentials at
60 significant digits.
"""
from __future__ import annotations

from decimal import Decimal, localcontext
from fractions import Fraction as F

import numpy as np

# --------------------------------------------------------------- e4m3 values


def e4m3_positive_values() -> list[F]:
    """The 127 finite non-negative E4M3 values in increasing order, listed as
    significand x 2^k: subnormals k/512 (k = 0..7), then 1.m x 2^e for
    e = -6..8 and m = 0..7, stopping at the largest finite value 448."""
    vals = [F(k, 512) for k in range(8)]
    for e in range(-6, 9):
        for m in range(8):
            v = F(8 + m, 8) * (F(2) ** e)
            if v <= 448:
                vals.append(v)
    return vals


E4M3_POS = e4m3_positive_values()
E4M3_POS_F64 = np.array([float(v) for v in E4M3_POS])


def e4m3_nearest_code(v: F | float) -> int:
    """Brute-force RNE-with-saturation to E4M3: search every finite value;
    on an exact tie take the even code index (= even mantissa), and clamp
    magnitudes above 448 to 448."""
    v = F(v)
    sign = 0x80 if v < 0 else 0x00
    a = abs(v)
    if a >= E4M3_POS[-1]:
        return sign | (len(E4M3_POS) - 1)
    best = None
    for k, c in enumerate(E4M3_POS):
        d = abs(a - c)
        if best is None or d < best[0] or (d == best[0] and k % 2 == 0):
            best = (d, k)
    return sign | best[1]


def e4m3_nearest_code_vec(v: np.ndarray) -> np.ndarray:
    """Vectorised form of the same search for fp64 inputs: the candidates are
    the two neighbours from a sorted search, compared against their exact
    midpoint (midpoints of E4M3 values are exact in fp64)."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    vals = E4M3_POS_F64
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, len(vals) - 1)
    lo = hi - 1
    mid = (vals[lo] + vals[hi]) / 2.0
    pick = np.where(a < mid, lo, np.where(a > mid, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= vals[-1], len(vals) - 1, pick)
    sign = np.where(np.signbit(v), 0x80, 0x00)
    return (sign | pick).astype(np.uint8)


# --------------------------------------------------------------- e2m1 values


def e2m1_positive_values() -> list[F]:
    """The 8 non-negative E2M1 values in increasing order, listed as
    significand x 2^k: the subnormal 0.5 (and zero), then 1.m x 2^e for
    e = 0..2, m = 0..1."""
    vals = [F(0), F(1, 2)]
    for e in range(3):
        for m in range(2):
            vals.append(F(2 + m, 2) * F(2) ** e)
    return vals


E2M1_POS = e2m1_positive_values()


def e2m1_nearest_code(v: F | float) -> int:
    """Brute-force RNE-with-saturation to E2M1: the nearest value, ties to
    the even code index (even mantissa), magnitudes above 6 clamped to 6."""
    v = F(v)
    sign = 0x8 if v < 0 else 0x0
    a = abs(v)
    if a >= E2M1_POS[-1]:
        return sign | (len(E2M1_POS) - 1)
    best = None
    for k, c in enumerate(E2M1_POS):
        d = abs(a - c)
        if best is None or d < best[0] or (d == best[0] and k % 2 == 0):
            best = (d, k)
    return sign | best[1]


def exact_nvfp4(y: list[F], gs: float):
    """Block codes, (v, code) of one row under NVFP4 with per-tensor scale gs:
    sf = e4m3(gs * amax / 6) per 16 columns, v = y gs / decode(sf)."""
    gs = F(float(np.float32(gs)))
    sf, v, codes = [], [], []
    for b in range(len(y) // 16):
        blk = y[16 * b:16 * b + 16]
        code = e4m3_nearest_code(gs * max(abs(t) for t in blk) / 6)
        sf.append(code)
        s = E4M3_POS[code & 0x7F]
        for t in blk:
            vj = t * gs / s if s > 0 else F(0)
            v.append(vj)
            codes.append(e2m1_nearest_code(vj))
    return sf, v, codes


# --------------------------------------------------------------- bf16 values


def bf16_bits_to_f64(bits) -> np.ndarray:
    """numpy's float32 view of (bits << 16)."""
    b = (np.asarray(bits, np.uint32) << 16).astype(np.uint32)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def _bf16_positive_table():
    codes = np.arange(0x0000, 0x7F81, dtype=np.uint32)  # +0 .. +inf
    return codes, bf16_bits_to_f64(codes)


BF16_POS_CODES, BF16_POS_VALUES = _bf16_positive_table()  # last entry is +inf
_BF16_MAX_F = F(float(BF16_POS_VALUES[-2]))
_BF16_OVERFLOW = _BF16_MAX_F + F(2) ** (127 - 8)  # max + half an ulp of the top binade


def bf16_nearest_code(v: F | float) -> int:
    """Exact RNE of a rational to bf16 (overflow to infinity at the IEEE
    threshold), by bisection over the sorted positive values and an exact
    midpoint comparison; ties go to the even code."""
    v = F(v)
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a >= _BF16_OVERFLOW:
        return sign | 0x7F80
    fa = float(a)
    k = int(np.searchsorted(BF16_POS_VALUES, fa))
    k = min(max(k, 1), len(BF16_POS_VALUES) - 2)
    cands = [j for j in (k - 1, k, k + 1) if 0 <= j < len(BF16_POS_VALUES) - 1]
    best = None
    for j in cands:
        d = abs(a - F(float(BF16_POS_VALUES[j])))
        if best is None or d < best[0] or (d == best[0] and BF16_POS_CODES[j] % 2 == 0):
            best = (d, j)
    return sign | int(BF16_POS_CODES[best[1]])


def fp32_nearest(v: F) -> np.float32:
    """Exact RNE of a rational to binary32."""
    d = np.float32(float(v))
    cands = [d, np.nextafter(d, np.float32(np.inf)), np.nextafter(d, np.float32(-np.inf))]
    best = None
    for c in cands:
        dist = abs(F(float(c)) - v)
        even = (np.array(c, np.float32).view(np.uint32) % 2) == 0
        if best is None or dist < best[0] or (dist == best[0] and even):
            best = (dist, c)
    return np.float32(best[1])


# ------------------------------------------------------------- exact rows


def _sqrt(x: F) -> F:
    with localcontext() as ctx:
        ctx.prec = 60
        d = Decimal(x.numerator) / Decimal(x.denominator)
        return F(d.sqrt())


def _exp(x: F) -> F:
    with localcontext() as ctx:
        ctx.prec = 60
        d = Decimal(x.numerator) / Decimal(x.denominator)
        return F(d.exp())


def pow2_at_least(x: F) -> F:
    """The smallest power of two >= x > 0, by exact comparison."""
    k = int(np.floor(np.log2(float(x))))
    while F(2) ** k < x:
        k += 1
    while F(2) ** (k - 1) >= x:
        k -= 1
    return F(2) ** k


def exact_quantize(y: list[F], mode: int, group: int, static_scale, amax_floor: float,
                   ue8m0: bool = False):
    """Scales and (v, code) pairs of one row, every step exact except the
    fp32 rounding of a dynamic scale, which is exact RNE (with ``ue8m0`` the
    scale is the smallest power of two >= amax/448 instead)."""
    n = len(y)
    if mode == 0:
        s_list = [np.float32(static_scale)]
        width = n
    else:
        width = n if mode == 1 else group
        s_list = []
        for g in range(n // width):
            amax = max(abs(t) for t in y[g * width:(g + 1) * width])
            amax = max(amax, F(amax_floor))
            s_list.append(np.float32(float(pow2_at_least(amax / 448))) if ue8m0
                          else fp32_nearest(amax / 448))
    v, codes = [], []
    for j, yj in enumerate(y):
        s = F(float(s_list[0 if mode == 0 else j // width]))
        vj = yj / s
        v.append(vj)
        codes.append(e4m3_nearest_code(vj))
    return np.array(s_list, np.float32), v, codes


def exact_norm_row(x_bits, res_bits, w_bits, eps: float, mode: int, group: int,
                   static_scale, amax_floor: float, ue8m0: bool = False):
    xs = [F(float(t)) for t in bf16_bits_to_f64(x_bits)]
    ws = [F(float(t)) for t in bf16_bits_to_f64(w_bits)]
    if res_bits is None:
        r_codes = None
        r = xs
    else:
        rs = [F(float(t)) for t in bf16_bits_to_f64(res_bits)]
        r_codes = [bf16_nearest_code(a + b) for a, b in zip(xs, rs)]
        r = [F(float(t)) for t in bf16_bits_to_f64(np.array(r_codes))]
    H = len(r)
    ms = sum(t * t for t in r) / H
    inv = 1 / _sqrt(ms + F(float(np.float32(eps))))
    y = [rj * inv * wj for rj, wj in zip(r, ws)]
    s, v, codes = exact_quantize(y, mode, group, static_scale, amax_floor, ue8m0)
    return {"residual_out": r_codes, "y": y, "scale": s, "v": v, "q": codes}


def exact_silu_row(gu_bits, mode: int, group: int, static_scale, amax_floor: float,
                   ue8m0: bool = False):
    vals = [F(float(t)) for t in bf16_bits_to_f64(gu_bits)]
    n = len(vals) // 2
    y = [vals[j] / (1 + _exp(-vals[j])) * vals[n + j] for j in range(n)]
    s, v, codes = exact_quantize(y, mode, group, static_scale, amax_floor, ue8m0)
    return {"y": y, "scale": s, "v": v, "q": codes}

