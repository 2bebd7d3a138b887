// row_norm.cuh -- pass 1 of an RMSNorm row, shared by the norm kernels.
//
// Per chunk of 8 bf16: r = bf16(x + residual) (or x), t = r * w (exact in
// fp32: two 8-bit significands), the chunk's amax |t|, and sum r^2 (exact
// squares; summed in double-float with TwoSum for the dynamic-scale and
// exact-rounding paths).
#pragma once

#include "common.cuh"

namespace vg {

struct RowAcc {
  float2 ss = make_float2(0.f, 0.f);  // sum r^2 (two lanes)
  float2 lo = make_float2(0.f, 0.f);  // its TwoSum error terms (dynamic modes)
};

// Pass 1 over one chunk: r = bf16(x + residual) (returned packed, for
// residual_out), t = r * w, the chunk's amax |t|, and sum r^2.
template <bool DYN, bool RES>
__device__ __forceinline__ uint4 pass1_chunk(const uint4 &xv, const uint4 &rv, const uint4 &wv,
                                             float2 (&t)[4], float &cmax, RowAcc &acc) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
  const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
  const float2 neg1 = make_float2(-1.f, -1.f);
  uint32_t ow[4];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (RES) {
      const float2 s2 = f2_add(bf16x2_to_f2(xw[i]), bf16x2_to_f2(rw[i]));
      ow[i] = pack_bf16x2_rn(s2.x, s2.y);
    } else {
      ow[i] = xw[i];
    }
    const float2 r = bf16x2_to_f2(ow[i]);
    if (DYN) {  // packed TwoSum of r^2 into (ss, lo)
      const float2 x = f2_mul(r, r);
      const float2 s = f2_add(acc.ss, x);
      const float2 bp = f2_fma(acc.ss, neg1, s);
      const float2 e = f2_add(f2_fma(f2_fma(bp, neg1, s), neg1, acc.ss), f2_fma(bp, neg1, x));
      acc.ss = s;
      acc.lo = f2_add(acc.lo, e);
    } else {
      acc.ss = f2_fma(r, r, acc.ss);
    }
    t[i] = f2_mul(r, bf16x2_to_f2(ww[i]));
    m = fmaxf(m, fmaxf(fabsf(t[i].x), fabsf(t[i].y)));
  }
  cmax = m;
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

}  // namespace vg
