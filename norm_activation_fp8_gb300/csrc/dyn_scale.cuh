// dyn_scale.cuh -- the dynamic-scale arithmetic shared by the norm kernels.
//
// Per-token and per-group scales divide by the stored fp32 scale
// s = fp32(amax * inv / 448).  Since y/s = 448 t / amax up to the rounding of
// s, and t = r*w and amax are exact products of bf16 numbers, some elements
// sit exactly on an e4m3 rounding midpoint; the direction in which s was
// rounded decides them.  make_dyn_scale rounds s correctly from a
// double-float inv and records that direction; dyn_values applies it.
#pragma once

#include "common.cuh"

namespace vg {

constexpr float kInv448 = 1.0f / 448.0f;
// fp32(A_MIN / 448), the scale of a row or group whose amax is floored.
constexpr float kFloorScale = (float)((double)kAmaxFloor / 448.0);
constexpr float kAwayOneUlp = 1.0f + 1.0f / 8388608.0f;    // 1 + 2^-23
constexpr float kTowardOneUlp = 1.0f - 1.0f / 16777216.0f; // 1 - 2^-24

// Per row (or group) quantities of the dynamic path.
struct DynScale {
  float s;   // stored dequantisation scale
  float a;   // divisor: v = 448 t / a (a = amax, or the floored equivalent)
  float ra;  // correctly rounded 1/a
  float f;   // tie direction: 1 + 2^-23 (away from zero), 1 - 2^-24 or 1
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
    d.f = D > 0.f ? kAwayOneUlp : (D < 0.f ? kTowardOneUlp : 1.0f);
    d.a = amax;
    d.ra = __frcp_rn(amax);
  } else {
    // amax floored, or X not a number (a NaN in the row, or inv = 0 from an
    // infinite sum of squares): v = t * inv / s, no exact ties to resolve.
    // inv = 0 takes a = 1 and 1/a = 0, so that v = t * 0 is the IEEE +-0, or
    // NaN for an infinite t; a NaN inv makes every v NaN.
    d.s = kFloorScale;
    d.f = 1.0f;
    d.a = y == 0.f ? 1.0f : 448.0f * kFloorScale / y;
    d.ra = y == 0.f ? 0.f : __frcp_rn(d.a);
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
  d.f = 1.0f;
  return d;
}

// Two elements: v = (448 t / a correctly rounded) * f.  For an exact tie the
// quotient is exactly a midpoint and f moves it off, in the direction the
// stored scale was rounded; every other quotient lies at least 2^-22
// (relative) from any midpoint, further than f can move it, so its code is
// unchanged.
__device__ __forceinline__ float2 dyn_values(float2 t, const DynScale &d) {
  const float2 T = f2_mul(t, make_float2(kE4M3Max, kE4M3Max));  // exact
  const float2 ra = make_float2(d.ra, d.ra);
  const float2 q0 = f2_mul(T, ra);
  const float2 q1 = f2_fma(f2_fma(q0, make_float2(-d.a, -d.a), T), ra, q0);
  const float2 v = f2_mul(q1, make_float2(d.f, d.f));
  // the correction step turns a -0 quotient into +0 ((+0) + (-0) = +0);
  // the quotient has the sign of t (a > 0)
  return make_float2(copysignf(v.x, t.x), copysignf(v.y, t.y));
}

}  // namespace vg
