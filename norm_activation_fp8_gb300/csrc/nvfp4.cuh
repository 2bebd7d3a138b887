// nvfp4.cuh -- the NVFP4 output format (NVIDIA's public NVFP4; E2M1 from the
// OCP Microscaling spec): E2M1 element codes (+-{0, 0.5, 1, 1.5, 2, 3, 4,
// 6}), blocks of 16 columns, an E4M3 scale code per block
// sf = e4m3(gs * amax / 6) with an fp32 per-tensor scale gs, elements
// e2m1(y * gs / decode(sf)), two codes a byte with column 2i in the low
// nibble.
#pragma once

#include "common.cuh"

namespace vg {

constexpr float kE2M1Max = 6.0f;
constexpr int kNvfp4Block = 16;  // columns per block scale (two 16-byte chunks)

// Eight E2M1 codes (RNE, saturating at 6) packed into 32 bits, element k in
// bits 4k..4k+3.  cvt...e2m1x2 puts its first source in the upper nibble.
__device__ __forceinline__ uint32_t quant_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// The value of a non-negative E4M3 code (0..0x7E), exactly: every E4M3
// value is an fp16 value, so E4M3 -> f16 -> f32 loses nothing.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  float r;
  asm("{\n\t.reg .b32 h2;\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.f16x2.e4m3x2 h2, %1;\n\t"
      "mov.b32 {lo, hi}, h2;\n\t"
      "cvt.f32.f16 %0, lo;\n\t}"
      : "=f"(r)
      : "h"((uint16_t)c));
  return r;
}

// E4M3 code of a non-negative fp32 value, RNE with saturation at 448.
__device__ __forceinline__ uint32_t e4m3_code(float x) { return cvt_e4m3x2(x, 0.f) & 0xFFu; }

// E4M3 code (RNE, saturating) of the non-negative double-float X = xh + xl
// (|xl| <= half an ulp of xh), decided exactly: the two codes around xh and
// the sign of X minus their midpoint (xh - m is exact: Sterbenz).
__device__ __forceinline__ uint32_t e4m3_code_df(float xh, float xl) {
  if (!(xh < kE4M3Max)) return 0x7Eu;  // saturated (and any overflow to inf)
  // |xl| <= 2^-24 xh: when xh (1 -+ 2^-20) round alike, so does X
  const uint32_t cc = cvt_e4m3x2(xh * (1.0f - 1.0f / 1048576.0f), xh * (1.0f + 1.0f / 1048576.0f));
  if ((cc >> 8) == (cc & 0xFFu)) return cc & 0xFFu;
  const uint32_t c = e4m3_code(xh);
  const float v = e4m3_value(c);
  if (v == xh || c == 0x7Eu && xh > v) return c;  // on a value, or saturated
  const uint32_t lo = v < xh ? c : c - 1, hi = lo + 1;
  const float mid = 0.5f * (e4m3_value(lo) + e4m3_value(hi));  // exact
  const float d = xh - mid;
  if (d > 0.f || (d == 0.f && xl > 0.f)) return hi;
  if (d < 0.f || xl < 0.f) return lo;
  return (lo & 1u) ? hi : lo;  // an exact tie: even code
}

// The E4M3 code of an fp32 estimate x whose relative error is below
// 2^-18 / 4: exact (`exact` is called) only where x lies within 2^-18 of a
// midpoint, i.e. where x (1 -+ 2^-18) round to different codes.
template <class Exact>
__device__ __forceinline__ uint32_t e4m3_code_settled(float x, Exact exact) {
  const uint32_t cc = cvt_e4m3x2(x * (1.0f - 1.0f / 262144.0f), x * (1.0f + 1.0f / 262144.0f));
  return (cc >> 8) == (cc & 0xFFu) ? (cc & 0xFFu) : exact();
}

}  // namespace vg
