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
// Two kernels:
//   mla_dual_norm_kernel       a token's rows spread over a group of warps
//                              (the shortest chain per token: few tokens);
//   mla_dual_norm_warp_kernel  one warp per token (the fewest instructions
//                              and no barrier per token: many tokens).
//
// Layout of a CTA of the first: `rpc` tokens, and per token thr[0] threads on the q row
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
#include <type_traits>

#include "common.cuh"
#include "dyn_scale.cuh"
#include "launch.h"
#include "row_norm.cuh"
#include "tma.cuh"

namespace vg {

// Status word of this translation unit's kernels (kErrBounds, debug builds).
__device__ uint32_t g_mla_status;

namespace {

// Extents in bytes of the outputs (debug checks).
[[maybe_unused]] __device__ __forceinline__ uint64_t out_extent(const MlaArgs &a, int side) {
  return VG_ROWS(a.T) * 16ull * (uint64_t)a.nch[side];
}
[[maybe_unused]] __device__ __forceinline__ uint64_t q8_extent(const MlaArgs &a) {
  return VG_ROWS(a.T) * 8ull * (uint64_t)a.nch[0];
}

// The body of the warp-group kernel (wrappers below).
template <int VPT, bool QFP8>
__device__ __forceinline__ void mla_dual_norm_rows(const MlaArgs &a) {
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

  // Launched with programmatic dependent launch: nothing in global memory
  // before the previous grid has finished (the row is only asked into L2);
  // the next grid may be scheduled once this one's loads are out.
  if (lr == 0 && live && (int)blockIdx.x < a.pf_ctas) prefetch_l2(src, 16u * (uint32_t)nch);
  pdl_wait();
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
  pdl_launch_dependents();
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
      if (live && VG_ACCESS_OK(g_mla_status, a.q_scale + row, 4, a.q_scale, 4 * VG_ROWS(a.T)))
        a.q_scale[row] = d.s;
    } else {
      inv[slot][side] = make_float2(y, dy);
    }
  }
  __syncthreads();

  if (fp8_row) {
    const DynScale d = dq[slot];
    uint8_t *out = a.q8 + (live ? row * (int64_t)nch * kElemsPerChunk : 0);
    if (two_multiply_ok(d)) {  // all but degenerate rows
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int c = lr + k * ntr;
        float v[8];
        dyn_values8_fast(t[k], d.rf, v);
        if (live && c < nch && VG_ACCESS_OK(g_mla_status, out + c * kElemsPerChunk, 8, a.q8, q8_extent(a)))
          st_stream(out + c * kElemsPerChunk, quant8(v));
      }
    } else {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int c = lr + k * ntr;
        float v[8];
        dyn_values8_exact(t[k], d, v);
        if (live && c < nch && VG_ACCESS_OK(g_mla_status, out + c * kElemsPerChunk, 8, a.q8, q8_extent(a)))
          st_stream(out + c * kElemsPerChunk, quant8(v));
      }
    }
  } else {
    const float2 yd = inv[slot][side];
    uint16_t *out = a.out[side] + (live ? row * (int64_t)nch * kElemsPerChunk : 0);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * ntr;
      const uint4 o = bf16x8_product_rn(t[k], yd.x, yd.y);
      if (live && c < nch &&
          VG_ACCESS_OK(g_mla_status, out + c * kElemsPerChunk, 16, a.out[side], out_extent(a, side)))
        st_stream(out + c * kElemsPerChunk, o);
    }
  }
}

// CTAs of up to 512 threads leave room for the fp8 q row's state at up to
// eight chunks per thread; a token wider than 512 threads takes a CTA of
// 1024 (one per SM, so up to 64 registers a thread).
template <int VPT, bool QFP8>
__global__ void __launch_bounds__(512) mla_dual_norm_kernel(const MlaArgs a) {
  mla_dual_norm_rows<VPT, QFP8>(a);
}
template <int VPT, bool QFP8>
__global__ void __launch_bounds__(1024, 1) mla_dual_norm_kernel_big(const MlaArgs a) {
  mla_dual_norm_rows<VPT, QFP8>(a);
}

// ----------------------------------------------------------- warp kernel
//
// One warp per token when the token's two rows fit 8 chunks per lane
// (q_dim + kv_dim <= 2048 after rounding each side to 32 chunks; DeepSeek's
// 1536 + 512 is exactly 8): lane l holds chunks l, l+32, ... of the q row
// (kq per lane) then of the kv row (kk per lane) as raw bf16.  Both sums of
// squares reduce by shuffles, every lane computes the scales (the same
// arithmetic in every lane, so no shared memory and no barrier), and pass 2
// recomputes t = x * w from the registers.  Warps run independent tokens, so
// one token's reduction latency hides behind the loads of others.

// t = x * w with the weight as fp32 pairs.
__device__ __forceinline__ void chunk_t(const uint4 &xv, const float2 (&wf)[4], float2 (&t)[4]) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) t[i] = f2_mul(bf16x2_to_f2(xw[i]), wf[i]);
}

constexpr int kMlaWarpChunks = 8;  // chunks per lane over both rows of a token
constexpr int kMlaWeightChunks = kMlaWarpChunks * 32;  // both weights, at most

// Both weights of the warp kernel sit in shared memory as fp32, converted
// once per CTA, so that neither pass unpacks them again: the kernel is bound
// by the integer pipe, which does the unpacking.  Two planes (elements 0-3
// of every chunk, then elements 4-7), so that the lanes of a warp, which read
// consecutive chunks, read consecutive 16-byte words without bank conflicts.
__device__ __forceinline__ void stage_weights_f32(float4 *ws, const MlaArgs &a) {
  for (int i = threadIdx.x; i < a.nch[0] + a.nch[1]; i += blockDim.x) {
    const uint4 wb = i < a.nch[0] ? ld_keep(a.w[0] + i * kElemsPerChunk)
                                  : ld_keep(a.w[1] + (i - a.nch[0]) * kElemsPerChunk);
    ws[i] = make_float4(bf16_lo(wb.x), bf16_hi(wb.x), bf16_lo(wb.y), bf16_hi(wb.y));
    ws[kMlaWeightChunks + i] = make_float4(bf16_lo(wb.z), bf16_hi(wb.z), bf16_lo(wb.w), bf16_hi(wb.w));
  }
}

// Chunk i of the staged weights (zeros past the row).
__device__ __forceinline__ void weights_f32(const float4 *ws, int i, bool in_row, float2 (&wf)[4]) {
  const float4 w0 = in_row ? ws[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 w1 = in_row ? ws[kMlaWeightChunks + i] : make_float4(0.f, 0.f, 0.f, 0.f);
  wf[0] = make_float2(w0.x, w0.y);
  wf[1] = make_float2(w0.z, w0.w);
  wf[2] = make_float2(w1.x, w1.y);
  wf[3] = make_float2(w1.z, w1.w);
}

// 16-byte asynchronous copy global -> shared (no register staging); a
// source size of 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src, bool full) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src),
               "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// KQ > 0: the rows are exactly KQ * 32 (q) and (8 - KQ) * 32 (kv) chunks
// wide, known at compile time, so no chunk needs a bounds check or a
// run-time choice of row (DeepSeek's 1536 + 512 is KQ = 6).  KQ = 0: any
// widths that fit, with `kq` q chunks per lane at run time.
// STAGE (DeepSeek's widths): the token's chunks go to shared memory by
// asynchronous copies and both passes read them there, instead of 32
// registers a lane holding them from the loads to the stores, so that more
// warps fit on an SM (five CTAs instead of four).
// Warp w of CTA b takes token b * 8 + w, or with SPREAD (one wave of CTAs,
// every resident slot filled) token b + w * grid, so that the tokens of a
// single wave are dealt evenly over the SMs.
template <bool QFP8, int KQ, bool STAGE, bool SPREAD>
__global__ void __launch_bounds__(256, STAGE ? 5 : 4)
    mla_dual_norm_warp_kernel(const MlaArgs a, const int kq_rt) {
  const int kq = KQ > 0 ? KQ : kq_rt;
  __shared__ float4 ws[kMlaWeightChunks * 2];  // both weights as fp32: q chunks, then kv; two planes
  __shared__ uint4 xs[STAGE ? 8 : 1][kMlaWarpChunks][32];  // STAGE: per warp, per chunk, per lane
  const int lane = threadIdx.x & 31;
  const int64_t row = SPREAD ? (int64_t)blockIdx.x + (int64_t)(threadIdx.x >> 5) * gridDim.x
                             : (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool live = row < a.T;  // warp-uniform
  // (side is a run-time value of the unrolled index: selects, not indexing,
  // keep everything in registers)
  const uint16_t *src_q = a.src[0] + (live ? row * a.stride[0] : 0);
  const uint16_t *src_kv = a.src[1] + (live ? row * a.stride[1] : 0);

  // the token's loads go out first, then the CTA stages the weights, so the
  // two round trips overlap
  if (lane == 0 && live && (int)blockIdx.x < a.pf_ctas) {  // both rows into L2 before the wait
    prefetch_l2(src_q, 16u * (uint32_t)a.nch[0]);
    prefetch_l2(src_kv, 16u * (uint32_t)a.nch[1]);
  }
  pdl_wait();  // programmatic dependent launch, as the kernel above
  uint4 xv[STAGE ? 1 : kMlaWarpChunks];
  uint4 (&xw)[kMlaWarpChunks][32] = xs[STAGE ? threadIdx.x >> 5 : 0];
#pragma unroll
  for (int j = 0; j < kMlaWarpChunks; ++j) {
    const bool q = j < kq;
    const int c = (q ? j : j - kq) * 32 + lane;
    const bool in = live && (KQ > 0 || c < (q ? a.nch[0] : a.nch[1]));
    const uint16_t *src = (q ? src_q : src_kv) + (in ? c * kElemsPerChunk : 0);
    if constexpr (STAGE)
      cp_async16(&xw[j][lane], src, in);
    else
      xv[j] = in ? ld_stream_ro(src) : make_uint4(0, 0, 0, 0);
  }
  stage_weights_f32(ws, a);
  pdl_launch_dependents();
  if constexpr (STAGE) cp_async_wait_all();  // this lane's own copies
  __syncthreads();
  if (!live) return;  // whole warps leave together
  // chunk j of this lane: from registers, or from its own slots in shared memory
  auto chunk = [&](int j) -> uint4 {
    if constexpr (STAGE) return lds128(&xw[j][lane]);
    else return xv[j];
  };
  RowAcc acc_q, acc_kv;
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < kMlaWarpChunks; ++j) {
    const bool q = j < kq;
    const int c = (q ? j : j - kq) * 32 + lane;
    float2 wv[4];
    weights_f32(ws, q ? c : a.nch[0] + c, KQ > 0 || c < (q ? a.nch[0] : a.nch[1]), wv);
    float2 t[4];
    float cmax;
    const uint4 x = chunk(j);
    if (q) {
      pass1_chunk<true, false>(x, x, wv, t, cmax, acc_q);
      am = fmaxf(am, cmax);
    } else {
      pass1_chunk<true, false>(x, x, wv, t, cmax, acc_kv);
    }
  }
  // Both sums of squares in one butterfly: after one exchange across the
  // half-warps, lanes 0-15 hold partial q sums and lanes 16-31 partial kv
  // sums; each half reduces its row (the same double-float steps in every
  // lane of a half, so all its lanes agree) and computes that row's inv.
  // Lane 0 then holds q's, lane 16 kv's.
  float yq, dyq, ykv, dykv;
  {
    float hq = acc_q.ss.x, lq = acc_q.lo.x + acc_q.lo.y;
    two_sum_acc(hq, lq, acc_q.ss.y);
    float hk = acc_kv.ss.x, lk = acc_kv.lo.x + acc_kv.lo.y;
    two_sum_acc(hk, lk, acc_kv.ss.y);
    const int side = lane >> 4;  // 0: q, 1: kv
    float h = side ? hk : hq, l = side ? lk : lq;
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, side ? hq : hk, 16);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, side ? lq : lk, 16);
    two_sum_acc(h, l, oh);
    l += ol;
    lanes_sum2(h, l, 16);
    float y, dy;
    rsqrt_df(h, l, a.n[side], a.inv_n[side], a.eps[side], y, dy);
    yq = __shfl_sync(0xFFFFFFFFu, y, 0);
    dyq = __shfl_sync(0xFFFFFFFFu, dy, 0);
    ykv = __shfl_sync(0xFFFFFFFFu, y, 16);
    dykv = __shfl_sync(0xFFFFFFFFu, dy, 16);
  }
  DynScale d;
  if (QFP8) {
    d = make_dyn_scale(warp_max(am), yq, dyq);
    if (lane == 0 && VG_ACCESS_OK(g_mla_status, a.q_scale + row, 4, a.q_scale, 4 * VG_ROWS(a.T)))
      a.q_scale[row] = d.s;
  }
  // Pass 2, with the q row's FP8 codes in the two-multiply form when the
  // token's scale has a tie direction (all but degenerate rows; the choice
  // is made once, so that the common loop has no branch).
  auto pass2 = [&](auto fast) {
#pragma unroll
    for (int j = 0; j < kMlaWarpChunks; ++j) {
      const bool q = j < kq;
      const int c = (q ? j : j - kq) * 32 + lane;
      const int nch = q ? a.nch[0] : a.nch[1];
      if (KQ == 0 && c >= nch) continue;
      float2 wv[4], t[4];
      weights_f32(ws, q ? c : a.nch[0] + c, true, wv);
      chunk_t(chunk(j), wv, t);
      const int64_t off = (row * nch + c) * kElemsPerChunk;
      if (QFP8 && q) {
        float v[8];
        if (decltype(fast)::value)
          dyn_values8_fast(t, d.rf, v);
        else
          dyn_values8_exact(t, d, v);
        if (VG_ACCESS_OK(g_mla_status, a.q8 + off, 8, a.q8, q8_extent(a))) st_stream(a.q8 + off, quant8(v));
      } else {
        uint16_t *op = (q ? a.out[0] : a.out[1]) + off;
        if (VG_ACCESS_OK(g_mla_status, op, 16, q ? a.out[0] : a.out[1], out_extent(a, q ? 0 : 1)))
          st_stream(op, bf16x8_product_rn(t, q ? yq : ykv, q ? dyq : dykv));
      }
    }
  };
  if (QFP8 && two_multiply_ok(d))
    pass2(std::true_type{});
  else
    pass2(std::false_type{});
}

template <int KQ, bool STAGE, bool SPREAD>
cudaError_t launch_warp(const MlaArgs &a, bool q_fp8, dim3 g, dim3 b, cudaStream_t s, int kq) {
  return q_fp8 ? launch_pdl(mla_dual_norm_warp_kernel<true, KQ, STAGE, SPREAD>, g, b, 0, s, a, kq)
               : launch_pdl(mla_dual_norm_warp_kernel<false, KQ, STAGE, SPREAD>, g, b, 0, s, a, kq);
}

template <int VPT, bool BIG>
cudaError_t launch_vpt(const MlaArgs &a, bool q_fp8, const MlaPlan &p, cudaStream_t s) {
  const dim3 g((unsigned)p.grid), b((unsigned)p.block);
  if constexpr (BIG)
    return q_fp8 ? launch_pdl(mla_dual_norm_kernel_big<VPT, true>, g, b, 0, s, a)
                 : launch_pdl(mla_dual_norm_kernel_big<VPT, false>, g, b, 0, s, a);
  else
    return q_fp8 ? launch_pdl(mla_dual_norm_kernel<VPT, true>, g, b, 0, s, a)
                 : launch_pdl(mla_dual_norm_kernel<VPT, false>, g, b, 0, s, a);
}

}  // namespace

uint32_t read_mla_status(bool reset) {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mla_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_mla_status, &zero, sizeof(zero)) != cudaSuccess) return 0xFFFFFFFFu;
  }
  return v;
}

cudaError_t launch_mla_dual_norm(MlaArgs a, bool q_fp8, const MlaPlan &p, cudaStream_t s) {
  a.thr[0] = p.thr[0];
  a.thr[1] = p.thr[1];
  a.rpc = p.rpc;
  const dim3 g((unsigned)p.grid), b((unsigned)p.block);
  if (p.vpt == 0) {  // one warp per token
    const int kq = (a.nch[0] + 31) / 32;
    if (a.nch[0] == 6 * 32 && a.nch[1] == 2 * 32)  // DeepSeek's latent widths
      return p.spread ? launch_warp<6, true, true>(a, q_fp8, g, b, s, kq)
                      : launch_warp<6, true, false>(a, q_fp8, g, b, s, kq);
    return p.spread ? launch_warp<0, false, true>(a, q_fp8, g, b, s, kq)
                    : launch_warp<0, false, false>(a, q_fp8, g, b, s, kq);
  }
  switch (p.vpt) {
    case 1: return launch_vpt<1, false>(a, q_fp8, p, s);
    case 2: return launch_vpt<2, false>(a, q_fp8, p, s);
    case 4: return launch_vpt<4, false>(a, q_fp8, p, s);
    default: return p.block > 512 ? launch_vpt<8, true>(a, q_fp8, p, s)
                                  : launch_vpt<8, false>(a, q_fp8, p, s);
  }
}

}  // namespace vg
