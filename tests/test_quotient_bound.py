"""Host check of the two-multiply dynamic quotient used by the GPU kernels.

Under a per-token or per-group scale the norm kernels (where the launch
allows it) and the MLA dual norm's FP8 q row code each element from
v = fp32(fp32(448 t) * rf), rf = fp32(fp32(1/amax) * (1 +- 2^-22)), where t
and amax are exact products of two bf16 numbers and the sign of the factor
is the direction in which the stored scale was rounded.  The claim: v gets
the E4M3 code of the exact quotient Q = 448 t / amax whenever Q is not an
E4M3 rounding midpoint, and the code on the recorded side when it is one.

The argument rests on a gap: a non-midpoint Q sits more than 8.3 u
(u = 2^-24, the unit roundoff; relative) from every midpoint, while the three fp32 roundings
and the factor move v between u and 7u off Q.  This test emulates the fp32
steps with numpy float32 (IEEE round-to-nearest-even, as on the GPU) over
every product of two 8-bit significands against a set of divisors, and
compares the codes with exact decisions.  It also shows that the factor is
neither too small (2^-23 misplaces exact ties) nor too large (2^-20 moves
non-ties across a midpoint).
"""
from __future__ import annotations

import numpy as np

import exact

U = 2.0 ** -24
# the sorted E4M3 rounding midpoints (exact in fp64)
MIDS = (exact.E4M3_POS_F64[:-1] + exact.E4M3_POS_F64[1:]) / 2


def _cases():
    """(t, amax) pairs: every product of two 8-bit significands, scaled by
    2^0 .. 2^-11, against divisors drawn from the same products plus ones
    built to make many exact ties (7 x a power of two)."""
    sig = np.arange(128, 256, dtype=np.int64)
    prods = np.unique((sig[:, None] * sig[None, :]).ravel())
    rng = np.random.default_rng(1234)
    divisors = np.concatenate([rng.choice(prods, 48, replace=False),
                               [65025, 16384, 28672, 7 * 4096, 224 * 255, 254 * 255]])
    ts, As = [], []
    for A in divisors:
        for s in range(0, -12, -1):
            t = prods * 2.0 ** s
            t = t[t <= A]
            ts.append(t)
            As.append(np.full(t.shape, float(A)))
    return np.concatenate(ts), np.concatenate(As)


def _codes(t, A, tie_factor, away):
    """Magnitude code indices of the emulated GPU value and of the exact
    decision, for one tie direction."""
    t32 = t.astype(np.float32)
    A32 = A.astype(np.float32)
    assert np.array_equal(t32.astype(np.float64), t) and np.array_equal(A32.astype(np.float64), A)
    T = np.float32(448.0) * t32                      # exact: <= 19 significant bits
    ra = np.float32(1.0) / A32                       # correctly rounded reciprocal
    f = np.float32(1.0 + tie_factor) if away else np.float32(1.0 - tie_factor)
    rf = ra * f
    v = (T * rf).astype(np.float64)
    got = exact.e4m3_nearest_code_vec(v) & 0x7F

    q = 448.0 * t / A    # fp64: equals a midpoint exactly iff Q does (gap >> 2^-53)
    want = exact.e4m3_nearest_code_vec(q) & 0x7F
    idx = np.searchsorted(MIDS, q)
    tie = (idx < len(MIDS)) & (MIDS[np.minimum(idx, len(MIDS) - 1)] == q)
    # a midpoint between values k and k + 1 (magnitude indices) goes to k + 1
    # away from zero, to k toward zero
    want = np.where(tie, idx + (1 if away else 0), want)
    return got, want, tie


def test_gap_and_two_multiply_codes():
    t, A = _cases()
    q = 448.0 * t / A
    idx = np.searchsorted(MIDS, q)
    gaps = []
    for j in (idx - 1, idx):
        ok = (j >= 0) & (j < len(MIDS))
        m = MIDS[np.clip(j, 0, len(MIDS) - 1)]
        g = np.abs(q - m) / m
        gaps.append(g[ok & (g > 0)])
    gmin = np.concatenate(gaps).min()
    assert gmin > 8.3 * U, gmin / U  # the bound 1 / (31 * 65025)

    for away in (True, False):
        got, want, tie = _codes(t, A, 2.0 ** -22, away)
        assert tie.sum() > 1000  # the divisor set makes many exact ties
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (away, t[bad[:5]], A[bad[:5]])


def test_tie_factor_is_neither_too_small_nor_too_large():
    t, A = _cases()

    def mismatches(factor):
        n = 0
        for away in (True, False):
            got, want, _ = _codes(t, A, factor, away)
            n += int((got != want).sum())
        return n

    assert mismatches(2.0 ** -23) > 0  # too small: exact ties land on either side
    assert mismatches(2.0 ** -20) > 0  # too large: non-ties cross a midpoint
