"""The tolerance checker accepts exactly what the tolerance allows (CPU)."""
import numpy as np
import pytest

import oracle
import parity


def _case(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n) * 50
    return v, oracle.e4m3_encode(v)


def test_identical_codes_pass():
    v, q = _case()
    assert parity.compare_codes(q, q, v)["mismatch"] == 0


def test_near_midpoint_flip_passes():
    v, q = _case()
    g = q.copy()
    # a value sitting just above the midpoint of codes 0x50 and 0x51
    lo, hi = oracle.e4m3_decode(np.array([0x50, 0x51], np.uint8))
    v[0] = (lo + hi) / 2 * (1 + 1e-7)
    q[0] = 0x51
    g[0] = 0x50
    st = parity.compare_codes(g, q, v)
    assert st["flips"] == 1 and st["max_flip_rel_dist"] < 1e-6


def test_flip_far_from_midpoint_fails():
    v, q = _case()
    g = q.copy()
    k = int(np.flatnonzero((q & 0x7F) > 0x20)[0])
    g[k] = q[k] + 1 if (q[k] & 0x7F) < 0x7E else q[k] - 1
    with pytest.raises(parity.ParityError, match="outside tolerance"):
        parity.compare_codes(g, q, v)


def test_non_adjacent_or_sign_flip_fails():
    v, q = _case()
    lo, hi = oracle.e4m3_decode(np.array([0x50, 0x51], np.uint8))
    v[0] = (lo + hi) / 2
    q[0] = 0x51
    for bad in (0x4F, 0xD1, 0xD0):
        g = q.copy()
        g[0] = bad
        with pytest.raises(parity.ParityError):
            parity.compare_codes(g, q, v)


def test_saturated_values_must_agree():
    v, q = _case()
    v[0], q[0] = 1000.0, 0x7E
    g = q.copy()
    g[0] = 0x7D
    with pytest.raises(parity.ParityError):
        parity.compare_codes(g, q, v)


def test_too_many_flips_fail():
    n = 20000
    lo, hi = oracle.e4m3_decode(np.array([0x50, 0x51], np.uint8))
    v = np.full(n, (lo + hi) / 2 * (1 + 1e-7))
    q = np.full(n, 0x51, np.uint8)
    g = q.copy()
    g[:2] = 0x50            # 2 flips = 0.01 % of 20000: allowed
    parity.compare_codes(g, q, v)
    g[:3] = 0x50            # 3 flips: over the budget
    with pytest.raises(parity.ParityError, match="near-midpoint flips"):
        parity.compare_codes(g, q, v)


def test_scale_tolerance():
    s = np.array([1.0, 2.5e-3, 7.0], np.float32)
    parity.compare_scales(s * np.float32(1 + 5e-7), s)
    with pytest.raises(parity.ParityError):
        parity.compare_scales(s * np.float32(1 + 3e-6), s)


def test_residual_bit_exact():
    a = np.arange(10, dtype=np.uint16)
    parity.compare_exact(a, a.copy(), "residual_out")
    b = a.copy()
    b[3] ^= 1
    with pytest.raises(parity.ParityError):
        parity.compare_exact(b, a, "residual_out")


def test_bf16_checker_accepts_near_midpoint_flips_only():
    import exact as ex
    o = np.full(3000, 0x3F80, np.uint16)                    # 1.0 ...
    o[1], o[2] = 0x3F81, 0xBF80                             # 1.0078125, -1.0
    mid = (1.0 + 1.0078125) / 2
    v = np.ones(3000)
    v[0], v[1], v[2] = mid * (1 - 2.0 ** -21), 1.0078125, -1.0
    g = o.copy()
    g[0] = 0x3F81                                           # one ulp, v near the midpoint: allowed
    assert parity.compare_bf16(g, o, v)["flips"] == 1
    v_far = v.copy()
    v_far[0] = 1.001                                        # far from the midpoint: rejected
    with pytest.raises(parity.ParityError):
        parity.compare_bf16(g, o, v_far)
    g2 = o.copy()
    g2[0] = 0x3F82                                          # two ulps: rejected
    with pytest.raises(parity.ParityError):
        parity.compare_bf16(g2, o, v)
    g3 = o.copy()
    g3[2] = 0xBF81                                          # sign kept, v not near: rejected
    with pytest.raises(parity.ParityError):
        parity.compare_bf16(g3, o, v)
    assert ex.bf16_bits_to_f64(np.array([0x3F81], np.uint16))[0] == 1.0078125


def _e2m1_case(n=40000, seed=1):
    """Oracle-coded E2M1 values, packed the NVFP4 way, and their v."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n) * 2.5
    codes = oracle.e2m1_encode(v)
    return v, codes, (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def _pack(codes):
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def test_e2m1_unpack_order():
    assert parity.unpack_e2m1(np.array([0x71], np.uint8)).tolist() == [1, 7]


def test_e2m1_checker():
    v, c, q4 = _e2m1_case()
    assert parity.compare_e2m1(q4, q4, v)["flips"] == 0
    # near the 1.0 / 1.5 midpoint (1.25): an adjacent flip passes
    v2, g = v.copy(), c.copy()
    v2[0], c2 = 1.25 * (1 + 1e-6), c.copy()
    c2[0], g[0] = 0x3, 0x2
    assert parity.compare_e2m1(_pack(g), _pack(c2), v2)["flips"] == 1
    # far from a midpoint, two codes apart, across the sign, or saturated: fail
    for vk, ok_code, bad_code in ((1.4, 0x3, 0x2), (1.25, 0x3, 0x1), (0.1, 0x0, 0x8),
                                  (6.5, 0x7, 0x6), (-1.25 * (1 + 1e-6), 0xB, 0x3)):
        v3, o, g = v.copy(), c.copy(), c.copy()
        v3[0], o[0], g[0] = vk, ok_code, bad_code
        with pytest.raises(parity.ParityError, match="outside tolerance"):
            parity.compare_e2m1(_pack(g), _pack(o), v3)
    # too many flips
    near = np.flatnonzero(np.isin(c & 7, [2, 3]))[:20]
    v4, o, g = v.copy(), c.copy(), c.copy()
    v4[near] = np.sign(v4[near]) * 1.25
    o[near] = (c[near] & 8) | 2
    g[near] = (c[near] & 8) | 3
    with pytest.raises(parity.ParityError, match="flips"):
        parity.compare_e2m1(_pack(g), _pack(o), v4)


def test_bf16_nan_payloads_match_but_not_numbers():
    a = np.array([0x7FC0, 0x3F80, 0xFF80], np.uint16)
    parity.compare_bf16_exact(np.array([0x7FFF, 0x3F80, 0xFF80], np.uint16), a, "r")
    with pytest.raises(parity.ParityError):
        parity.compare_bf16_exact(np.array([0x7F80, 0x3F80, 0xFF80], np.uint16), a, "r")
    with pytest.raises(parity.ParityError):
        parity.compare_bf16_exact(np.array([0x7FC0, 0x3F81, 0xFF80], np.uint16), a, "r")


def test_non_finite_scales_must_match_exactly():
    o = np.array([np.inf, 1.0, np.nan], np.float32)
    parity.compare_scales(np.array([np.inf, 1.0 + 5e-7, np.nan], np.float32), o)
    for g in ([3e38, 1.0, np.nan], [np.inf, np.inf, np.nan], [np.inf, 1.0, 1.0],
              [-np.inf, 1.0, np.nan]):
        with pytest.raises(parity.ParityError):
            parity.compare_scales(np.array(g, np.float32), o)
