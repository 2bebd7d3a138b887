// mla_norm.cu -- the MLA dual RMSNorm, one launch for both norms.
//
// Implements "MLA Dual RMSNorm (fuse_mla_dual_rms_norm)" of the "Fusion
// torch.compile passes" page: MLA attention's paired q_c and kv_c RMSNorms,
// each with its own weight and eps, in one kernel.  q_c and kv_c are column
// slices of one projected tensor, so each is read through its own row
// stride.  Two output forms:
//   bf16 (fused_mla_dual_rms_norm): q_normed and kv_normed in bf16;
//   fp8  (fused_mla_dual_rms_norm_per_token_quant): q to FP8 e4m3 with a
//        dynamic per-token scale, kv_normed in bf16.
//
// Layout of a CTA: `rpc` tokens, and per token thr[0] threads on the q row
// followed by thr[1] threads on the kv row (each a whole number of warps).
// A thread owns chunks c = lr + k * thr[side], k < VPT, of its row, keeps
// t = x * w in registers, and the row's sum of squares is reduced in
// double-float (warp butterflies, then the side's warps through shared
// memory), so inv = 1/sqrt(mean + eps) is known to ~2^-44.
//
// bf16 outputs are correctly rounded: t * inv is formed as a double-float
// hi + lo and only hi is rounded, after hi has been moved one fp32 ulp toward
// lo when it sits exactly on a bf16 midpoint.  The fp8 q row uses the exact
// dynamic-scale arithmetic of dyn_scale.cuh.
#include "common.cuh"
#include "dyn_scale.cuh"
#include "launch.h"
#include "row_norm.cuh"

namespace vg {

namespace {

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

// Up to four chunks per thread a token takes at most 512 threads (register
// room for the fp8 q row's state); eight per thread allow 1024.
template <int VPT, bool QFP8>
__global__ void __launch_bounds__(VPT < 8 ? 512 : 1024) mla_dual_norm_kernel(const MlaArgs a) {
  __shared__ float4 red[32];      // per warp: sum hi, sum lo, amax
  __shared__ float2 inv[32][2];   // per token slot and side: y, dy
  __shared__ DynScale dq[32];     // per token slot: the q row's fp8 scale

  const int per_tok = a.thr[0] + a.thr[1];
  const int tid = threadIdx.x;
  const int slot = tid / per_tok;
  const int lt = tid - slot * per_tok;
  const int side = lt < a.thr[0] ? 0 : 1;  // warp-uniform
  const int lr = side == 0 ? lt : lt - a.thr[0];
  const int ntr = a.thr[side];
  const int nch = a.nch[side];
  const int64_t row = (int64_t)blockIdx.x * a.rpc + slot;
  const bool live = row < a.T;
  const uint16_t *src = a.src[side] + (live ? row * a.stride[side] : 0);
  const uint16_t *w = a.w[side];
  const bool fp8_row = QFP8 && side == 0;

  uint4 xv[VPT], wv[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * ntr;
    if (live && c < nch) {
      xv[k] = ld_stream_ro(src + c * kElemsPerChunk);
      wv[k] = ld_keep(w + c * kElemsPerChunk);
    } else {
      xv[k] = make_uint4(0, 0, 0, 0);
      wv[k] = make_uint4(0, 0, 0, 0);
    }
  }
  float2 t[VPT][4];
  float cmax[VPT];
  RowAcc acc;
#pragma unroll
  for (int k = 0; k < VPT; ++k) pass1_chunk<true, false>(xv[k], xv[k], wv[k], t[k], cmax[k], acc);

  float hi = acc.ss.x, lo = acc.lo.x + acc.lo.y;
  two_sum_acc(hi, lo, acc.ss.y);
  lanes_sum2(hi, lo, 32);
  float am = 0.f;
  if (fp8_row) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) am = fmaxf(am, cmax[k]);
    am = warp_max(am);
  }
  if ((tid & 31) == 0) red[tid >> 5] = make_float4(hi, lo, am, 0.f);
  __syncthreads();
  if (lr == 0) {  // one thread per token slot and side
    const int w0 = (slot * per_tok + (side ? a.thr[0] : 0)) >> 5;
    float h = 0.f, l = 0.f, amr = 0.f;
    for (int i = 0; i < (ntr >> 5); ++i) {  // the same order for every row
      const float4 p = red[w0 + i];
      two_sum_acc(h, l, p.x);
      l += p.y;
      amr = fmaxf(amr, p.z);
    }
    float y, dy;
    rsqrt_df(h, l, a.n[side], a.inv_n[side], a.eps[side], y, dy);
    if (fp8_row) {
      const DynScale d = make_dyn_scale(amr, y, dy);
      dq[slot] = d;
      if (live) a.q_scale[row] = d.s;
    } else {
      inv[slot][side] = make_float2(y, dy);
    }
  }
  __syncthreads();

  if (fp8_row) {
    const DynScale d = dq[slot];
    uint8_t *out = a.q8 + (live ? row * (int64_t)nch * kElemsPerChunk : 0);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * ntr;
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 q = dyn_values(t[k][i], d);
        v[2 * i] = q.x;
        v[2 * i + 1] = q.y;
      }
      if (live && c < nch) st_stream(out + c * kElemsPerChunk, quant8(v));
    }
  } else {
    const float2 yd = inv[slot][side];
    uint16_t *out = a.out[side] + (live ? row * (int64_t)nch * kElemsPerChunk : 0);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * ntr;
      uint4 o;
      o.x = bf16x2_product_rn(t[k][0], yd.x, yd.y);
      o.y = bf16x2_product_rn(t[k][1], yd.x, yd.y);
      o.z = bf16x2_product_rn(t[k][2], yd.x, yd.y);
      o.w = bf16x2_product_rn(t[k][3], yd.x, yd.y);
      if (live && c < nch) st_stream(out + c * kElemsPerChunk, o);
    }
  }
}

template <int VPT>
cudaError_t launch_vpt(const MlaArgs &a, bool q_fp8, const MlaPlan &p, cudaStream_t s) {
  if (q_fp8)
    mla_dual_norm_kernel<VPT, true><<<(unsigned)p.grid, p.block, 0, s>>>(a);
  else
    mla_dual_norm_kernel<VPT, false><<<(unsigned)p.grid, p.block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla_dual_norm(MlaArgs a, bool q_fp8, const MlaPlan &p, cudaStream_t s) {
  a.thr[0] = p.thr[0];
  a.thr[1] = p.thr[1];
  a.rpc = p.rpc;
  switch (p.vpt) {
    case 1: return launch_vpt<1>(a, q_fp8, p, s);
    case 2: return launch_vpt<2>(a, q_fp8, p, s);
    case 4: return launch_vpt<4>(a, q_fp8, p, s);
    default: return launch_vpt<8>(a, q_fp8, p, s);
  }
}

}  // namespace vg
