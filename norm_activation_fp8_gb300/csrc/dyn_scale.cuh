// dyn_scale.cuh -- the dynamic-scale arithmetic shared by the norm kernels.
//
// Per-token and per-group scales divide by the stored fp32 scale
// s = fp32(amax * inv / 448).  Since y/s = 448 t / amax up to the rounding of
// s, and t = r*w and amax are exact products of bf16 numbers, some elements
// sit exactly on an e4m3 rounding midpoint; the direction in which s was
// rounded decides them.  make_dyn_scale rounds s correctly from a
// double-float inv and records that direction; dyn_values8_fast and
// dyn_values8_exact apply it.
//
// Why two multiplies an element are enough.  With t = P 2^e and
// amax = A 2^e' (P, A < 2^16: products of two 8-bit significands), an e4m3
// midpoint is M = N 2^k with N odd, N <= 31.  448 t and M amax are both
// integer multiples of the smaller of their two powers of two, so a quotient
// Q = 448 t / amax that is not exactly M differs from it by at least
// min(1/(N A), 1/(7 P)) >= 1/(31 * 65025) > 8.3 u relative (u = 2^-24).
// v = fp32(fp32(448 t) * rf), rf = fp32(fp32(1/amax) (1 +- 4u)), is Q times
// (1 +- 4u) up to three roundings of at most u each, so it lies between u and
// 7u (relative) on the recorded side of Q: an exact tie goes the recorded
// way, and every other quotient stays on its own side of every midpoint
// (8.3u > 7u), so its code is Q's code.  Where no direction is recorded (X
// exactly 448 s, the floored scale, a non-finite row) ties go to even, and
// the correctly rounded quotient is formed instead (dyn_values8_exact, which
// also serves launches that keep the quotient form throughout: measured on
// GB300, the persistent norm kernel with 256-thread rows runs 4-6 % faster
// back to back with it, although it issues more instructions).
#pragma once

#include "common.cuh"

namespace vg {

constexpr float kInv448 = 1.0f / 448.0f;
// fp32(A_MIN / 448), the scale of a row or group whose amax is floored.
constexpr float kFloorScale = (float)((double)kAmaxFloor / 448.0);
constexpr float kTieAway = 1.0f + 0x1p-22f;    // 1 + 4u: ties away from zero
constexpr float kTieToward = 1.0f - 0x1p-22f;  // 1 - 4u: ties toward zero

// Per row (or group) quantities of the dynamic path.
struct DynScale {
  float s;   // stored dequantisation scale
  float a;   // divisor: v = 448 t / a (a = amax, or the floored equivalent)
  float ra;  // correctly rounded 1/a
  float rf;  // fp32(ra * (1 +- 4u)) in the tie direction; == ra: no direction
};

__device__ __forceinline__ float next_up(float x) { return __uint_as_float(__float_as_uint(x) + 1u); }
__device__ __forceinline__ float next_down(float x) { return __uint_as_float(__float_as_uint(x) - 1u); }

// amax: max |r*w| of the row or group; inv = y + dy, a normalised
// double-float (|dy| <= half an ulp of y).
__device__ __forceinline__ DynScale make_dyn_scale(float amax, float y, float dy) {
  const float xh = amax * y;
  const float xl = fmaf(amax, y, -xh) + amax * dy;  // X = xh + xl, |xl| <~ ulp(xh)/2
  DynScale d;
  if (xh >= kAmaxFloor) {
    // s = fp32(X / 448): start from xh * fp32(1/448) (within two ulps) and
    // step by the sign of D = X - 448 s against half an ulp (448/2 ulp(s));
    // the FMA part of D is exact because 448 s is within a few ulps of xh.
    float s = xh * kInv448;
#pragma unroll
    for (int it = 0; it < 3; ++it) {
      const float D = fmaf(-448.0f, s, xh) + xl;
      const float half = 224.0f * (next_up(s) - s);
      s = D > half ? next_up(s) : (D < -half ? next_down(s) : s);
    }
    const float D = fmaf(-448.0f, s, xh) + xl;
    d.s = s;
    d.a = amax;
    d.ra = __frcp_rn(amax);
    d.rf = D != 0.f ? d.ra * (D > 0.f ? kTieAway : kTieToward) : d.ra;
  } else {
    // amax floored, or X not a number (a NaN in the row, or inv = 0 from an
    // infinite sum of squares): v = t * inv / s, no exact ties to resolve.
    // inv = 0 takes a = 1 and 1/a = 0, so that v = t * 0 is the IEEE +-0, or
    // NaN for an infinite t; a NaN inv makes every v NaN.
    d.s = kFloorScale;
    d.a = y == 0.f ? 1.0f : 448.0f * kFloorScale / y;
    d.ra = y == 0.f ? 0.f : __frcp_rn(d.a);
    d.rf = d.ra;
  }
  return d;
}

// UE8M0 (power-of-two) scale of a row or group: the smallest s = 2^k with
// 448 s >= X = max(amax * inv, A_MIN), inv = y + dy.  The comparisons with
// 448 * 2^k are exact (an FMA difference of nearby fp32 numbers, then the
// sign of the double-float remainder).  Returns s in .s and the element
// multiplier y / s in .ra (v = t * ra; .a = 0 marks the power-of-two form).
__device__ __forceinline__ bool df_at_most(float xh, float xl, float p) {
  const float d = xh - p;  // exact when xh and p are within a factor of two
  return d < 0.f || (d == 0.f && xl <= 0.f);
}

// The smallest k with 448 * 2^k >= a, for a normal fp32 a > 0, from its
// bits: 448 = 1.75 * 2^8, so with a = m * 2^e (1 <= m < 2), k = e - 8 when
// m <= 1.75 and e - 7 otherwise.  Exact.
__device__ __forceinline__ int pow2_exponent_448(float a) {
  const uint32_t b = __float_as_uint(a);
  return (int)(b >> 23) - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}

// Whether a lies within 2^-18 (relative) of a boundary 448 * 2^k: its
// significand within 56 units of the last place of 1.75.
__device__ __forceinline__ bool near_pow2_boundary_448(float a) {
  const int d = (int)(__float_as_uint(a) & 0x7FFFFFu) - 0x600000;
  return d >= -56 && d <= 56;
}

// 2^k for -126 <= k <= 127.
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

__device__ __forceinline__ DynScale make_pow2_scale(float amax, float y, float dy) {
  float xh = amax * y;
  float xl = fmaf(amax, y, -xh) + amax * dy;
  if (!(xh >= kAmaxFloor)) {  // floored (the equal case rounds to the floor too; NaN too)
    xh = kAmaxFloor;
    xl = 0.f;
  }
  // X = xh + xl with |xl| <= ulp(xh) / 2 and every boundary representable:
  // only an xh exactly on a boundary lets xl decide
  int k = pow2_exponent_448(xh);
  if ((__float_as_uint(xh) & 0x7FFFFFu) == 0x600000u && xl > 0.f) ++k;
  DynScale d;
  d.s = exp2i(k);
  d.a = 0.f;
  d.ra = y * exp2i(-k);  // exact: a power-of-two scaling
  d.rf = d.ra;
  return d;
}

// Whether a row or group's codes may take the two-multiply form: it has a
// tie direction, and 1/a is far from the subnormal range (where rf would be
// rounded with less than fp32 precision).
__device__ __forceinline__ bool two_multiply_ok(const DynScale &d) {
  return d.rf != d.ra && d.ra >= 0x1p-100f;
}

// A chunk of 8 in the two-multiply form: v = fp32(fp32(448 t) rf).
__device__ __forceinline__ void dyn_values8_fast(const float2 (&t)[4], float rf, float (&v)[8]) {
  const float2 k448 = make_float2(kE4M3Max, kE4M3Max), r = make_float2(rf, rf);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = f2_mul(f2_mul(t[i], k448), r);  // 448 t is exact
    v[2 * i] = q.x;
    v[2 * i + 1] = q.y;
  }
}

// A chunk of 8 in the quotient form, valid for every row: the correctly
// rounded q = 448 t / a (one FMA correction of the product with the
// correctly rounded reciprocal), so that an exact tie lands exactly on its
// midpoint, then multiplied by 1 + 2^-23 (ties away from zero) or 1 - 2^-24
// (toward zero) in the recorded direction, or left on the midpoint (ties to
// even) where none is recorded.  A non-tie quotient lies more than 8 u from
// every midpoint, so the factor cannot change its code.
__device__ __forceinline__ void dyn_values8_exact(const float2 (&t)[4], const DynScale &d,
                                                  float (&v)[8]) {
  const float2 k448 = make_float2(kE4M3Max, kE4M3Max);
  const float f = d.rf > d.ra ? 1.0f + 0x1p-23f : (d.rf < d.ra ? 1.0f - 0x1p-24f : 1.0f);
  const float2 ra = make_float2(d.ra, d.ra), na = make_float2(-d.a, -d.a), ff = make_float2(f, f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 T = f2_mul(t[i], k448);
    const float2 q0 = f2_mul(T, ra);
    const float2 q1 = f2_mul(f2_fma(f2_fma(q0, na, T), ra, q0), ff);
    // the correction step turns a -0 quotient into +0 ((+0) + (-0) = +0);
    // the quotient has the sign of t (a > 0)
    v[2 * i] = copysignf(q1.x, t[i].x);
    v[2 * i + 1] = copysignf(q1.y, t[i].y);
  }
}

}  // namespace vg
