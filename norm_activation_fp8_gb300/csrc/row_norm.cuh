// row_norm.cuh -- pass 1 of an RMSNorm row, shared by the norm kernels.
//
// Per chunk of 8 bf16: r = bf16(x + residual) (or x), t = r * w (exact in
// fp32: two 8-bit significands), the chunk's amax |t|, and sum r^2 (exact
// squares; summed in double-float with TwoSum for the dynamic-scale and
// exact-rounding paths).  Also the correctly rounded bf16 of t * inv for the
// norms whose output stays bf16.
#pragma once

#include "common.cuh"

namespace vg {

struct RowAcc {
  float2 ss = make_float2(0.f, 0.f);  // sum r^2 (two lanes)
  float2 lo = make_float2(0.f, 0.f);  // its TwoSum error terms (dynamic modes)
};

// Pass 1 over one chunk: r = bf16(x + residual) (returned packed, for
// residual_out), t = r * w, the chunk's amax |t|, and sum r^2.  The weight
// comes as four fp32 pairs.  PADD: the residual add as one packed bf16 add
// a pair (the exact sum rounded once); otherwise an fp32 add and a
// conversion, which give the same bits.  Measured on GB300: the packed add
// is 1-3 % faster in the register kernel, the fp32 form 5-8 % faster in the
// persistent kernel at H = 8192.
template <bool DYN, bool RES, bool PADD = false>
__device__ __forceinline__ uint4 pass1_chunk(const uint4 &xv, const uint4 &rv, const float2 (&wf)[4],
                                             float2 (&t)[4], float &cmax, RowAcc &acc) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
  const float2 neg1 = make_float2(-1.f, -1.f);
  uint32_t ow[4];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (RES && PADD) {
      ow[i] = add_bf16x2_rn(xw[i], rw[i]);
    } else if (RES) {
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
    t[i] = f2_mul(r, wf[i]);
    m = fmax3(m, fabsf(t[i].x), fabsf(t[i].y));
  }
  cmax = m;
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// The same with the weight as a packed bf16 chunk.
template <bool DYN, bool RES, bool PADD = false>
__device__ __forceinline__ uint4 pass1_chunk(const uint4 &xv, const uint4 &rv, const uint4 &wv,
                                             float2 (&t)[4], float &cmax, RowAcc &acc) {
  const float2 wf[4] = {bf16x2_to_f2(wv.x), bf16x2_to_f2(wv.y), bf16x2_to_f2(wv.z),
                        bf16x2_to_f2(wv.w)};
  return pass1_chunk<DYN, RES, PADD>(xv, rv, wf, t, cmax, acc);
}

// bf16(t * (y + dy)) for two elements, rounded as the exact product would
// be (y + dy normalised, |dy| <= half an ulp of y).
__device__ __forceinline__ uint32_t bf16x2_product_rn(float2 t, float y, float dy) {
  float out[2];
  const float tv[2] = {t.x, t.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float p = tv[i] * y;
    const float e = fmaf(tv[i], y, -p) + tv[i] * dy;  // t (y + dy) = p + e to ~2^-44
    const float hi = p + e;                             // |e| < ulp(p): Fast2Sum
    const float lo = e - (hi - p);
    const uint32_t b = __float_as_uint(hi);
    // a hi exactly on a bf16 midpoint is decided by the sign of lo
    const float r = ((b & 0xFFFFu) == 0x8000u && lo != 0.f)
                        ? __uint_as_float(((lo > 0.f) != (b >> 31 != 0u)) ? b + 1u : b - 1u)
                        : hi;
    // y > 0, so the product has the sign of t; this keeps a -0 that the
    // additions above turn into +0
    out[i] = copysignf(r, tv[i]);
  }
  return pack_bf16x2_rn(out[0], out[1]);
}

// bf16 of t * (y + dy) for a chunk of 8.  p = fp32(t * y) lies within
// 2^-23 |p| (normal p) or 2^-149 (subnormal p) of the exact product E.  The
// bracket b <= E <= a (or a <= E <= b for negative p) with
//   a = fp32(p (1 + 2^-22) + 2^-149),   b = fp32(p (1 - 2^-22) - 2^-149)
// holds after the roundings of a and b, and rounding is monotonic: wherever
// bf16(a) and bf16(b) have the same magnitude, every value between them --
// E included -- rounds to that magnitude, and bf16(p) carries E's sign (the
// sign of t; a zero p keeps its sign).  Only chunks with an element whose
// bracket straddles a bf16 rounding boundary (about 1 in 1000) take the
// double-float path.  Three packed conversions and one logic op a pair,
// instead of a bit test per element: this keeps the integer pipe free.
static __device__ __noinline__ uint4 bf16x8_product_rn_slow(float2 t0, float2 t1, float2 t2, float2 t3,
                                                     float y, float dy) {
  return make_uint4(bf16x2_product_rn(t0, y, dy), bf16x2_product_rn(t1, y, dy),
                    bf16x2_product_rn(t2, y, dy), bf16x2_product_rn(t3, y, dy));
}

__device__ __forceinline__ uint4 bf16x8_product_rn(const float2 (&t)[4], float y, float dy) {
  const float2 yy = make_float2(y, y);
  const float2 ku = make_float2(1.0f + 0x1p-22f, 1.0f + 0x1p-22f);
  const float2 kd = make_float2(1.0f - 0x1p-22f, 1.0f - 0x1p-22f);
  const float2 eu = make_float2(0x1p-149f, 0x1p-149f);
  const float2 ed = make_float2(-0x1p-149f, -0x1p-149f);
  uint32_t o[4], diff = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = f2_mul(t[i], yy);
    const float2 a = f2_fma(p, ku, eu);
    const float2 b = f2_fma(p, kd, ed);
    diff |= pack_bf16x2_rn(a.x, a.y) ^ pack_bf16x2_rn(b.x, b.y);
    o[i] = pack_bf16x2_rn(p.x, p.y);
  }
  if (diff & 0x7FFF7FFFu)  // rare: out of line, so it costs the common path no registers
    return bf16x8_product_rn_slow(t[0], t[1], t[2], t[3], y, dy);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace vg
