// silu_fp8.cu -- SiLU(gate) * up -> FP8 e4m3, one pass over HBM.
//
// Implements "SiLU+Mul + Quantization (fuse_act_quant)" of the "Fusion
// torch.compile passes" page: silu_and_mul of the gate-up projection
// followed by quant_fp8, in one kernel, without materialising the
// post-activation tensor.
//
// Row layout: gate_up[t] = [gate (I) | up (I)].  A thread owns the same
// chunk index c in both halves, so its 16-byte loads of gate and up are both
// coalesced across the warp.  a = g * sigmoid(g) * u in fp32:
//   sigmoid(g) = rcp(1 + __expf(-g))   (rcp.approx: 1 ulp; a huge
//                denominator flushes the reciprocal to +0 and the product
//                keeps the sign of g, as the exact -0 would)
// Static and per-group modes need no row-wide reduction: each chunk is
// quantised and stored as soon as its group's amax (a butterfly over 8 or 16
// lanes) is known.  Per-token keeps the row's activations in registers until
// the row amax is reduced.
//
// Dynamic scales: s = fp32(amax * fp32(1/448)) and v = a * rcp(s).  The
// activations are transcendental, so no element sits exactly on an e4m3
// midpoint and an ulp or two in s or 1/s only moves codes whose value is
// within ~1e-6 of a midpoint (both are far inside the parity tolerance:
// scales within 1e-6, near-midpoint flips rare).
#include "common.cuh"
#include "launch.h"

namespace vg {
namespace {

__device__ __forceinline__ float fast_rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Two elements of silu(g) * u = g * rcp(1 + exp(-g)) * u.
__device__ __forceinline__ float2 silu_mul2(uint32_t gw, uint32_t uw) {
  const float2 g = bf16x2_to_f2(gw);
  const float2 e = make_float2(__expf(-g.x), __expf(-g.y));
  const float2 d = f2_add(e, make_float2(1.0f, 1.0f));
  return f2_mul(f2_mul(g, make_float2(fast_rcp(d.x), fast_rcp(d.y))), bf16x2_to_f2(uw));
}

__device__ __forceinline__ void silu_chunk(const uint4 &gv, const uint4 &uv, float (&v)[8]) {
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = silu_mul2(gw[i], uw[i]);
    v[2 * i] = a.x;
    v[2 * i + 1] = a.y;
  }
}

__device__ __forceinline__ void scale8(float (&v)[8], float m) {
  const float2 mm = make_float2(m, m);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = f2_mul(make_float2(v[2 * i], v[2 * i + 1]), mm);
    v[2 * i] = p.x;
    v[2 * i + 1] = p.y;
  }
}

// fp32(max(amax, floor) / 448) to within an ulp: one multiply.
__device__ __forceinline__ float silu_scale(float amax) {
  return fmaxf(amax, kAmaxFloor) * (1.0f / kE4M3Max);
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// A row is covered by ntr * VPT chunks per CTA.  Static and per-group modes
// keep no row state, so longer rows are split into column segments
// (blockIdx.y), independent CTAs.  Per-token needs the amax of the whole row
// in one CTA: up to 1024 threads (BIG) with four chunks each.
//
// Register budget: static and per-group chunks hold no row state between
// loads and stores, so they fit three 512-thread CTAs per SM; per-token
// keeps its row's activations and fits two 512-thread or one 1024-thread
// CTA.
template <int VPT, int MODE, int GCH, bool BIG>
__global__ void __launch_bounds__(BIG ? 1024 : 512, BIG ? 1 : (MODE == kPerToken ? 2 : 3))
    silu_fp8_kernel(const SiluArgs a) {
  __shared__ float red[32];

  const int tid = threadIdx.x;
  const int slot = tid / a.ntr;
  const int lr0 = tid - slot * a.ntr;
  const int lr = lr0 + (int)blockIdx.y * a.ntr * VPT;  // chunk offset of the segment
  const int64_t row = (int64_t)blockIdx.x * a.rpc + slot;
  const bool live = row < a.T;
  const int64_t in_base = live ? row * 2 * a.I : 0;
  const int64_t out_base = live ? row * a.I : 0;

  uint4 gv[VPT], uv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    if (live && c < a.nch) {
      gv[k] = ld_stream_ro(a.gate_up + in_base + c * kElemsPerChunk);
      uv[k] = ld_stream_ro(a.gate_up + in_base + a.I + c * kElemsPerChunk);
    } else {
      gv[k] = make_uint4(0, 0, 0, 0);
      uv[k] = make_uint4(0, 0, 0, 0);
    }
  }

  if (MODE != kPerToken) {
    const float inv_static = (MODE == kStatic) ? __frcp_rn(__ldg(a.scale)) : 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      float v[8];
      silu_chunk(gv[k], uv[k], v);
      float m = inv_static;
      if (MODE == kPerGroup) {
        const float s = silu_scale(lanes_max(amax8(v), GCH));
        if (live && c < a.nch && (c & (GCH - 1)) == 0) a.scale[row * a.ngroups + c / GCH] = s;
        m = fast_rcp(s);
      }
      scale8(v, m);
      if (live && c < a.nch) st_stream(a.q + out_base + c * kElemsPerChunk, quant8(v));
    }
    return;
  }

  // Per-token: activations stay in registers until the row amax is known.
  float act[VPT][8];
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    silu_chunk(gv[k], uv[k], act[k]);
    am = fmaxf(am, amax8(act[k]));
  }
  am = warp_max(am);
  if (a.ntr > 32) {
    const int nw = a.ntr >> 5;
    if ((lr0 & 31) == 0) red[slot * nw + (lr0 >> 5)] = am;
    __syncthreads();
    am = 0.f;
    for (int i = 0; i < nw; ++i) am = fmaxf(am, red[slot * nw + i]);
  }
  const float s = silu_scale(am);
  if (live && lr == 0) a.scale[row] = s;
  const float m = fast_rcp(s);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    scale8(act[k], m);
    if (live && c < a.nch) st_stream(a.q + out_base + c * kElemsPerChunk, quant8(act[k]));
  }
}

template <int VPT>
cudaError_t launch_mode(const SiluArgs &a, int mode, const RowPlan &p, cudaStream_t s) {
  const dim3 g((unsigned)p.grid, (unsigned)p.segs), b((unsigned)p.block());
  switch (mode) {
    case kStatic: silu_fp8_kernel<VPT, kStatic, 1, false><<<g, b, 0, s>>>(a); break;
    case kPerToken:
      if (p.block() > 512)
        silu_fp8_kernel<VPT, kPerToken, 1, true><<<g, b, 0, s>>>(a);
      else
        silu_fp8_kernel<VPT, kPerToken, 1, false><<<g, b, 0, s>>>(a);
      break;
    default:
      if (a.gch == 8)
        silu_fp8_kernel<VPT, kPerGroup, 8, false><<<g, b, 0, s>>>(a);
      else
        silu_fp8_kernel<VPT, kPerGroup, 16, false><<<g, b, 0, s>>>(a);
      break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_silu_fp8(SiluArgs a, int mode, const RowPlan &p, cudaStream_t s) {
  a.ntr = p.ntr;
  a.rpc = p.rpc;
  switch (p.vpt) {
    case 1: return launch_mode<1>(a, mode, p, s);
    case 2: return launch_mode<2>(a, mode, p, s);
    default: return launch_mode<4>(a, mode, p, s);
  }
}

}  // namespace vg
