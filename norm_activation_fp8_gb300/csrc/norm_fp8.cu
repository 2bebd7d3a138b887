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
//   2. r = bf16(x + residual) (fp32 add, RNE) -> residual_out; accumulate
//      sum(r^2) and the amax of |r*w| (exact in fp32: 8-bit x 8-bit
//      significands) per chunk;
//   3. one reduction over the row's threads of (sum r^2, max |r*w|):
//      warp butterflies, then shared memory across the row's warps;
//   4. inv = rsqrt(sum/H + eps); y = r*w*inv; scale from the amax
//      (per-group: a butterfly over the 8 or 16 lanes holding the group);
//   5. q = e4m3(y * (1/s)) packed with cvt.rn.satfinite.e4m3x2, 8-byte stores.
#include "common.cuh"
#include "launch.h"

namespace vg {
namespace {

template <int VPT, int MODE, bool RES>
__global__ void __launch_bounds__(512) norm_fp8_kernel(const NormArgs a) {
  __shared__ float2 red[16];  // one (sum, amax) per warp; blockDim <= 512

  const int tid = threadIdx.x;
  const int slot = tid / a.ntr;        // row slot inside the CTA
  const int lr = tid - slot * a.ntr;   // thread index inside the row
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

  // r = bf16(x + residual); sum of squares; amax of |r*w| per chunk.
  float ss = 0.f, am = 0.f;
  float cmax[VPT];
  uint4 rb[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const uint32_t xw[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
    const uint32_t rw[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
    const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
    uint32_t ow[4];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ow[i] = RES ? pack_bf16x2_rn(bf16_lo(xw[i]) + bf16_lo(rw[i]), bf16_hi(xw[i]) + bf16_hi(rw[i]))
                  : xw[i];
      const float r0 = bf16_lo(ow[i]), r1 = bf16_hi(ow[i]);
      ss = fmaf(r0, r0, ss);
      ss = fmaf(r1, r1, ss);
      m = fmaxf(m, fmaxf(fabsf(r0 * bf16_lo(ww[i])), fabsf(r1 * bf16_hi(ww[i]))));
    }
    rb[k] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    cmax[k] = m;
    am = fmaxf(am, m);
    const int c = lr + k * a.ntr;
    if (RES && live && c < a.nch) st_stream(a.res_out + base + c * kElemsPerChunk, rb[k]);
  }

  // Row reduction of (sum r^2, max |r*w|).
  ss = warp_sum(ss);
  if (MODE == kPerToken) am = warp_max(am);
  if (a.ntr > 32) {  // uniform over the CTA
    const int nw = a.ntr >> 5;
    if ((lr & 31) == 0) red[slot * nw + (lr >> 5)] = make_float2(ss, am);
    __syncthreads();
    ss = 0.f;
    am = 0.f;
    for (int i = 0; i < nw; ++i) {
      const float2 p = red[slot * nw + i];
      ss += p.x;
      am = fmaxf(am, p.y);
    }
  }
  const float inv = rsqrtf(fmaf(ss, a.inv_h, a.eps));

  // Multiplier taking r*w to y/s, per row or per chunk's group.
  float mult[VPT];
  if (MODE == kStatic) {
    const float m = inv * __frcp_rn(__ldg(a.scale));
#pragma unroll
    for (int k = 0; k < VPT; ++k) mult[k] = m;
  } else if (MODE == kPerToken) {
    const float s = dynamic_scale(am * inv);
    if (live && lr == 0) a.scale[row] = s;
    const float m = inv * __frcp_rn(s);
#pragma unroll
    for (int k = 0; k < VPT; ++k) mult[k] = m;
  } else {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const float s = dynamic_scale(lanes_max(cmax[k], a.gch) * inv);
      const int c = lr + k * a.ntr;
      if (live && c < a.nch && (c % a.gch) == 0)
        a.scale[row * a.ngroups + c / a.gch] = s;
      mult[k] = inv * __frcp_rn(s);
    }
  }

  // q = e4m3(r * w * mult).
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    const uint32_t ow[4] = {rb[k].x, rb[k].y, rb[k].z, rb[k].w};
    const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_lo(ow[i]) * bf16_lo(ww[i]) * mult[k];
      v[2 * i + 1] = bf16_hi(ow[i]) * bf16_hi(ww[i]) * mult[k];
    }
    if (live && c < a.nch) st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
  }
}

template <int VPT, int MODE>
cudaError_t launch_res(const NormArgs &a, const RowPlan &p, cudaStream_t s) {
  if (a.res != nullptr)
    norm_fp8_kernel<VPT, MODE, true><<<(unsigned)p.grid, p.block(), 0, s>>>(a);
  else
    norm_fp8_kernel<VPT, MODE, false><<<(unsigned)p.grid, p.block(), 0, s>>>(a);
  return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_mode(const NormArgs &a, int mode, const RowPlan &p, cudaStream_t s) {
  switch (mode) {
    case kStatic: return launch_res<VPT, kStatic>(a, p, s);
    case kPerToken: return launch_res<VPT, kPerToken>(a, p, s);
    default: return launch_res<VPT, kPerGroup>(a, p, s);
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
