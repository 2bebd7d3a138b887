// norm_fp8.cu -- residual add + RMSNorm -> FP8 e4m3, one pass over HBM.
//
// Implements "RMSNorm + Quantization (fuse_norm_quant)" of the "Fusion
// torch.compile passes" page: fused_add_rms_norm(x, residual) (residual
// updated in place) or rms_norm(x), followed by quant_fp8 with a static,
// per-token or per-token-group scale, in one kernel.  The normalised row is
// never written: it lives in registers between the two halves of the kernel.
//
// Per row (n = H, chunks of 8 bf16):
//   1. 16-byte loads of x, residual and weight for every chunk the thread
//      owns, all issued before any is used;
//   2. r = bf16(x + residual) (fp32 add, RNE) -> residual_out; t = r*w
//      (exact in fp32: 8-bit x 8-bit significands) kept in registers;
//      sum(r^2); amax of |t| per chunk;
//   3. one reduction over the row's threads: warp butterflies, then shared
//      memory across the row's warps;
//   4. y = t * inv with inv = 1/sqrt(sum/H + eps); scale; q = e4m3(y / s)
//      packed with cvt.rn.satfinite.e4m3x2 into 8-byte stores.
//
// Static scale: inv in fp32 (rsqrt), v = t * (inv / s).
//
// Dynamic scales (per token, per group): y/s = 448 t/amax up to the fp32
// rounding of the stored scale s = fp32(amax inv / 448), and t and amax are
// both products of two bf16 numbers, so a small fraction of elements fall
// exactly on an e4m3 rounding midpoint.  Their correct code is decided by
// the direction in which the stored scale was rounded, so the dynamic path
//   - sums r^2 in double-float (TwoSum; r^2 is exact in fp32) and gets
//     inv as a double-float (rsqrt_df), all in fp32 arithmetic;
//   - forms X = amax * inv exactly enough to round s = fp32(X / 448)
//     correctly and to know the sign of X - 448 s (an FMA residual that
//     is exact);
//   - per element computes q1 = 448 t / amax correctly rounded (one FMA
//     correction of the product with the correctly rounded reciprocal), and
//     where an exact FMA remainder shows q1 is the exact quotient -- the
//     only case in which it can sit on a midpoint -- moves it one or two
//     ulps in the direction of that sign before the conversion.  Elements
//     that are not exact ties lie at least 2^-22 (relative) from every
//     midpoint, so the move never changes their code.
#include "common.cuh"
#include "launch.h"

namespace vg {
namespace {

// fp32(A_MIN / 448), the scale of a row or group whose amax is floored.
constexpr float kFloorScale = (float)((double)kAmaxFloor / 448.0);
constexpr float kAwayOneUlp = 1.0f + 1.0f / 8388608.0f;    // 1 + 2^-23
constexpr float kTowardOneUlp = 1.0f - 1.0f / 16777216.0f; // 1 - 2^-24

// Per row (or group) quantities of the dynamic path.
struct DynScale {
  float s;   // stored dequantisation scale
  float a;   // divisor: v = 448 t / a (a = amax, or the floored equivalent)
  float ra;  // correctly rounded 1/a
  float f;   // multiplier applied to an exact quotient (tie direction)
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
    // s = fp32(X / 448): the correctly rounded xh/448 is within one ulp of
    // it; D = X - 448 s (the FMA part is exact) decides the last step.
    float s = __fdiv_rn(xh, 448.0f);
    float D = fmaf(-448.0f, s, xh) + xl;
    const float half = 224.0f * (next_up(s) - s);
    if (D > half) {
      s = next_up(s);
      D = fmaf(-448.0f, s, xh) + xl;
    } else if (D < -half) {
      s = next_down(s);
      D = fmaf(-448.0f, s, xh) + xl;
    }
    d.s = s;
    d.f = D > 0.f ? kAwayOneUlp : (D < 0.f ? kTowardOneUlp : 1.0f);
    d.a = amax;
  } else {  // amax floored: v = t * inv / s, no exact ties to resolve
    d.s = kFloorScale;
    d.f = 1.0f;
    d.a = amax > 0.f ? 448.0f * kFloorScale / y : 1.0f;
  }
  d.ra = __frcp_rn(d.a);
  return d;
}

// Two elements: v = 448 t / a correctly rounded, exact quotients scaled by f.
__device__ __forceinline__ float2 dyn_values(float2 t, const DynScale &d) {
  const float2 T = f2_mul(t, make_float2(kE4M3Max, kE4M3Max));  // exact
  const float2 ra = make_float2(d.ra, d.ra);
  const float2 na = make_float2(-d.a, -d.a);
  const float2 q0 = f2_mul(T, ra);
  const float2 q1 = f2_fma(f2_fma(q0, na, T), ra, q0);
  const float2 e1 = f2_fma(q1, na, T);
  const float2 m = make_float2(e1.x == 0.f ? d.f : 1.0f, e1.y == 0.f ? d.f : 1.0f);
  return f2_mul(q1, m);
}

template <int VPT, int MODE, int GCH, bool RES>
__global__ void __launch_bounds__(512) norm_fp8_kernel(const NormArgs a) {
  constexpr bool DYN = MODE != kStatic;
  __shared__ float4 red[16];  // per-warp partials; blockDim <= 512

  const int tid = threadIdx.x;
  const int slot = tid / a.ntr;       // row slot inside the CTA
  const int lr = tid - slot * a.ntr;  // thread index inside the row
  const int lane = tid & 31;
  const int64_t row = (int64_t)blockIdx.x * a.rpc + slot;
  const bool live = row < a.T;
  const int64_t base = live ? row * a.H : 0;

  uint4 xv[VPT], rv[VPT], wv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    if (live && c < a.nch) {
      xv[k] = ld_stream_ro(a.x + base + c * kElemsPerChunk);
      if (RES) rv[k] = ld_stream(a.res + base + c * kElemsPerChunk);
      wv[k] = ld_keep(a.w + c * kElemsPerChunk);
    } else {
      xv[k] = make_uint4(0, 0, 0, 0);
      rv[k] = make_uint4(0, 0, 0, 0);
      wv[k] = make_uint4(0, 0, 0, 0);
    }
  }

  // r = bf16(x + residual) -> residual_out; t = r*w; sum r^2; amax |t|.
  float2 t[VPT][4];
  float cmax[VPT];
  float2 ss = make_float2(0.f, 0.f), ss_lo = make_float2(0.f, 0.f);
  const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const uint32_t xw[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
    const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
    const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
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
      if (DYN) {  // packed TwoSum of r^2 into (ss, ss_lo)
        const float2 x = f2_mul(r, r);
        const float2 s = f2_add(ss, x);
        const float2 bp = f2_fma(ss, neg1, s);
        const float2 e = f2_add(f2_fma(f2_fma(bp, neg1, s), neg1, ss), f2_fma(bp, neg1, x));
        ss = s;
        ss_lo = f2_add(ss_lo, e);
      } else {
        ss = f2_fma(r, r, ss);
      }
      t[k][i] = f2_mul(r, bf16x2_to_f2(ww[i]));
      m = fmaxf(m, fmaxf(fabsf(t[k][i].x), fabsf(t[k][i].y)));
    }
    cmax[k] = m;
    const int c = lr + k * a.ntr;
    if (RES && live && c < a.nch)
      st_stream(a.res_out + base + c * kElemsPerChunk, make_uint4(ow[0], ow[1], ow[2], ow[3]));
  }

  float mult = 0.f;
  DynScale dk[VPT];
  if (!DYN) {
    float sum = ss.x + ss.y;
    sum = warp_sum(sum);
    if (a.ntr > 32) {  // uniform over the CTA
      const int nw = a.ntr >> 5;
      if (lane == 0) red[slot * nw + (lr >> 5)] = make_float4(sum, 0.f, 0.f, 0.f);
      __syncthreads();
      sum = 0.f;
      for (int i = 0; i < nw; ++i) sum += red[slot * nw + i].x;
    }
    const float inv = rsqrtf(fmaf(sum, a.inv_h, a.eps));
    mult = inv * __frcp_rn(__ldg(a.scale));
  } else {
    float hi = ss.x, lo = ss_lo.x + ss_lo.y;
    two_sum_acc(hi, lo, ss.y);
    lanes_sum2(hi, lo, 32);
    float am = 0.f;
    if (MODE == kPerToken) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) am = fmaxf(am, cmax[k]);
      am = warp_max(am);
    }
    if (a.ntr > 32) {  // uniform over the CTA
      const int nw = a.ntr >> 5;
      if (lane == 0) red[slot * nw + (lr >> 5)] = make_float4(hi, lo, am, 0.f);
      __syncthreads();
      // every warp folds the row's partials the same way: lane i takes
      // partial i, then one butterfly (identical result in every lane)
      const float4 p = lane < nw ? red[slot * nw + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      hi = p.x;
      lo = p.y;
      lanes_sum2(hi, lo, 32);
      if (MODE == kPerToken) am = warp_max(p.z);
    }
    float y, dy;
    rsqrt_df(hi, lo, (float)a.H, a.inv_h, a.eps, y, dy);
    if (MODE == kPerToken) {
      const DynScale d = make_dyn_scale(am, y, dy);
      if (live && lr == 0) a.scale[row] = d.s;
#pragma unroll
      for (int k = 0; k < VPT; ++k) dk[k] = d;
    } else {
      // Per group: the group's GCH chunks sit on GCH consecutive lanes.
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const float gmax = lanes_max(cmax[k], GCH);
        dk[k] = make_dyn_scale(gmax, y, dy);
        const int c = lr + k * a.ntr;
        if (live && c < a.nch && (lane & (GCH - 1)) == 0)
          a.scale[row * a.ngroups + c / GCH] = dk[k].s;
      }
    }
  }

  // q = e4m3(y / s).
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q = DYN ? dyn_values(t[k][i], dk[k]) : f2_mul(t[k][i], make_float2(mult, mult));
      v[2 * i] = q.x;
      v[2 * i + 1] = q.y;
    }
    if (live && c < a.nch) st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
  }
}

template <int VPT, int MODE, int GCH>
cudaError_t launch_res(const NormArgs &a, const RowPlan &p, cudaStream_t s) {
  if (a.res != nullptr)
    norm_fp8_kernel<VPT, MODE, GCH, true><<<(unsigned)p.grid, p.block(), 0, s>>>(a);
  else
    norm_fp8_kernel<VPT, MODE, GCH, false><<<(unsigned)p.grid, p.block(), 0, s>>>(a);
  return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_mode(const NormArgs &a, int mode, const RowPlan &p, cudaStream_t s) {
  switch (mode) {
    case kStatic: return launch_res<VPT, kStatic, 1>(a, p, s);
    case kPerToken: return launch_res<VPT, kPerToken, 1>(a, p, s);
    default:
      return a.gch == 8 ? launch_res<VPT, kPerGroup, 8>(a, p, s)
                        : launch_res<VPT, kPerGroup, 16>(a, p, s);
  }
}

}  // namespace

cudaError_t launch_norm_fp8(NormArgs a, int mode, const RowPlan &p, cudaStream_t s) {
  a.ntr = p.ntr;
  a.rpc = p.rpc;
  switch (p.vpt) {
    case 1: return launch_mode<1>(a, mode, p, s);
    case 2: return launch_mode<2>(a, mode, p, s);
    case 4: return launch_mode<4>(a, mode, p, s);
    default: return launch_mode<8>(a, mode, p, s);
  }
}

}  // namespace vg
