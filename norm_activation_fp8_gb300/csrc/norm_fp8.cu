// norm_fp8.cu -- residual add + RMSNorm -> FP8 e4m3, one pass over HBM.
//
// Implements "RMSNorm + Quantization (fuse_norm_quant)" of the "Fusion
// torch.compile passes" page: fused_add_rms_norm(x, residual) (residual
// updated in place) or rms_norm(x), followed by quant_fp8 with a static,
// per-token or per-token-group scale, in one kernel.  The normalised row is
// never written: t = r*w stays in registers between the two halves.
//
// Per row (n = H, chunks of 8 bf16; a row's ntr threads own chunks
// c = lr + k*ntr, k < VPT):
//   1. r = bf16(x + residual) (fp32 add, RNE) -> residual_out; t = r*w
//      (exact in fp32: 8-bit x 8-bit significands); sum(r^2); amax |t| per
//      chunk;
//   2. one reduction over the row's threads: warp butterflies, then shared
//      memory across the row's warps;
//   3. y = t * inv with inv = 1/sqrt(sum/H + eps); scale; q = e4m3(y / s)
//      packed with cvt.rn.satfinite.e4m3x2 into 8-byte stores.
//
// Static scale: inv in fp32 (rsqrt), v = t * (inv / s).
// Dynamic scales: see dyn_scale.cuh.  Each scale slot (group, or row) is
// computed once, by the slot's own thread, through shared memory; r^2 is
// summed in double-float (TwoSum; r^2 is exact in fp32).
//
// The same row logic writes three more outputs (internal modes):
//   kBf16Pad    bf16(y), correctly rounded, into a zero-padded row
//               ("RMSNorm + Padding (fuse_act_padding)");
//   kPerGroupX  per-group scales as powers of two (UE8M0) and/or stored
//               column-major: the scale formats sm100 FP8 GEMMs read;
//   kNvfp4      NVFP4: E4M3 scale codes per 16 columns under a per-tensor
//               scale, E2M1 element codes two a byte (nvfp4.cuh).
//
// Two kernels share that row logic:
//   norm_fp8_kernel      one CTA per row group, inputs loaded straight into
//                        registers with 16-byte loads issued up front (small
//                        T: lowest latency);
//   norm_fp8_tma_kernel  persistent CTAs, one row at a time, the next rows'
//                        x and residual staged into shared memory by bulk
//                        TMA copies on a ring of mbarrier-tracked stages, the
//                        weight staged once per CTA (large T: HBM stays busy
//                        while a CTA reduces, scales and stores a row).
#include <atomic>

#include "common.cuh"
#include "dyn_scale.cuh"
#include "launch.h"
#include "nvfp4.cuh"
#include "row_norm.cuh"
#include "tma.cuh"

namespace vg {

// Status word of this translation unit's kernels (kErrWaitTimeout, and
// kErrBounds in debug builds).
__device__ uint32_t g_norm_status;

// Extents in bytes of the tensors a launch touches (debug checks).
__device__ __forceinline__ uint64_t q_extent(const NormArgs &a, int mode) {
  return VG_ROWS(a.T) * (uint64_t)(mode == kNvfp4 ? a.H / 2 : a.H);
}
__device__ __forceinline__ uint64_t row_extent(const NormArgs &a) {  // x, residual, residual_out
  return VG_ROWS(a.T) * 2ull * (uint64_t)a.H;
}
__device__ __forceinline__ uint64_t scale_extent(const NormArgs &a, int mode) {
  const uint64_t rows = VG_ROWS(a.T);
  if (mode == kPerToken) return 4 * rows;
  return rows == 0 ? 0 : 4 * ((rows - 1) * (uint64_t)a.s_ts + (uint64_t)(a.ngroups - 1) * a.s_gs + 1);
}

namespace {

// ---------------------------------------------------------------- row logic

// Shared memory a row group needs for the reduction and the scales.
struct RowSmem {
  float4 *red;    // [2][16] per-warp partials, double-buffered by row parity
  float *cmax;    // [rpc][ntr * VPT] chunk amax (per-group)
  DynScale *dyn;  // [rpc][nslots]; NVFP4 keeps float2 {s, gs * inv / s} per block
};

// Row reduction, scales and pass 2 (quantise + store q).  Called by every
// thread of the CTA.
template <int VPT, int MODE, int GCH>
__device__ __forceinline__ void finish_rows(const NormArgs &a, const float2 (&t)[VPT][4],
                                            const float (&cmax)[VPT], const RowAcc &acc,
                                            const RowSmem &sm, int parity, int slot, int lr,
                                            int64_t row, bool live, int64_t base) {
  constexpr bool DYN = MODE != kStatic;
  const int lane = threadIdx.x & 31;
  const int nw = a.ntr >> 5;
  float4 *red = sm.red + parity * 16;

  if (!DYN) {
    float sum = warp_sum(acc.ss.x + acc.ss.y);
    if (lane == 0) red[slot * nw + (lr >> 5)] = make_float4(sum, 0.f, 0.f, 0.f);
    __syncthreads();
    sum = 0.f;
    for (int i = 0; i < nw; ++i) sum += red[slot * nw + i].x;
    const float inv = rsqrtf(fmaf(sum, a.inv_h, a.eps));
    const float mult = inv * __frcp_rn(__ldg(a.scale));
    const float2 m2 = make_float2(mult, mult);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 q = f2_mul(t[k][i], m2);
        v[2 * i] = q.x;
        v[2 * i + 1] = q.y;
      }
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, a.q + base + c * kElemsPerChunk, 8, a.q, q_extent(a, MODE)))
        st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
    }
    return;
  }

  // Dynamic scales: each scale slot (group, or the row) is computed once,
  // by the slot's thread, from the warp partials and chunk amaxes.  The bf16
  // output has one slot per row holding inv = y + dy.
  const int row_chunks = a.ntr * VPT;
  constexpr bool PG = MODE == kPerGroup || MODE == kPerGroupX || MODE == kNvfp4;
  const int nslots = PG ? a.ngroups : 1;
  float hi = acc.ss.x, lo = acc.lo.x + acc.lo.y;
  two_sum_acc(hi, lo, acc.ss.y);
  lanes_sum2(hi, lo, 32);
  float am = 0.f;
  if (MODE == kPerToken) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) am = fmaxf(am, cmax[k]);
    am = warp_max(am);
  } else if (PG) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) sm.cmax[slot * row_chunks + lr + k * a.ntr] = cmax[k];
  }
  if (lane == 0) red[slot * nw + (lr >> 5)] = make_float4(hi, lo, am, 0.f);
  __syncthreads();
  if (lr < nslots) {
    float h = 0.f, l = 0.f, amr = 0.f;
    for (int i = 0; i < nw; ++i) {  // same order in every slot thread
      const float4 p = red[slot * nw + i];
      two_sum_acc(h, l, p.x);
      l += p.y;
      amr = fmaxf(amr, p.z);
    }
    float y, dy;
    rsqrt_df(h, l, (float)a.H, a.inv_h, a.eps, y, dy);
    if (MODE == kBf16Pad) {
      sm.dyn[slot] = DynScale{y, dy, 0.f, 0.f};
    } else if (MODE == kNvfp4) {
      // a block scale for every 16 columns: more blocks than threads when a
      // thread holds more than two chunks.  x = amax * (y gs / 6) in fp32 is
      // within 2^-22 of X = gs * amax * inv / 6; a block whose x lies near an
      // E4M3 midpoint gets the code of X in double-float.
      const float gs = __ldg(a.scale);
      const float ygs = y * gs, ygs6 = ygs * (1.0f / 6.0f);
      for (int g = lr; g < nslots; g += a.ntr) {
        float bm = 0.f;
#pragma unroll
        for (int i = 0; i < GCH; ++i) bm = fmaxf(bm, sm.cmax[slot * row_chunks + g * GCH + i]);
        const uint32_t code = e4m3_code_settled(bm * ygs6, [&] {
          // amax * gs exactly, times y + dy, then a division by 6 with its
          // exact remainder
          const float p = bm * gs, pe = fmaf(bm, gs, -p);
          const float xh = p * y, xl = fmaf(p, y, -xh) + (p * dy + pe * y);
          const float qh = __fdiv_rn(xh, 6.0f);
          const float ql = __fdiv_rn(fmaf(-qh, 6.0f, xh) + xl, 6.0f);
          const float qs = qh + ql;
          return e4m3_code_df(qs, ql - (qs - qh));
        });
        const float sv = e4m3_value(code);
        if (live && VG_ACCESS_OK(g_norm_status, a.sf8 + row * nslots + g, 1, a.sf8,
                                 VG_ROWS(a.T) * (uint64_t)nslots))
          a.sf8[row * nslots + g] = (uint8_t)code;
        reinterpret_cast<float2 *>(sm.dyn)[slot * nslots + g] =
            make_float2(sv, sv > 0.f ? ygs * __frcp_rn(sv) : 0.f);
      }
    } else {
      if (PG) {
        amr = 0.f;
#pragma unroll
        for (int i = 0; i < GCH; ++i) amr = fmaxf(amr, sm.cmax[slot * row_chunks + lr * GCH + i]);
      }
      const DynScale d = MODE == kPerGroupX && a.ue8m0 ? make_pow2_scale(amr, y, dy)
                                                       : make_dyn_scale(amr, y, dy);
      sm.dyn[slot * nslots + lr] = d;
      float *sp = MODE == kPerGroupX ? a.scale + row * a.s_ts + (int64_t)lr * a.s_gs
                                     : a.scale + row * nslots + lr;
      if (live && VG_ACCESS_OK(g_norm_status, sp, 4, a.scale, scale_extent(a, MODE))) *sp = d.s;
    }
  }
  __syncthreads();
  if (MODE == kNvfp4) {  // v = t * y * gs / s, E2M1 codes; a zero scale gives +0 codes
    uint8_t *out = a.q + (live ? row * (int64_t)(a.H / 2) : 0);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      const float2 d = reinterpret_cast<const float2 *>(sm.dyn)[slot * nslots + (c >= a.nch ? 0 : c / GCH)];
      const float2 m2 = make_float2(d.y, d.y);
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 q = f2_mul(t[k][i], m2);
        v[2 * i] = q.x;
        v[2 * i + 1] = q.y;
      }
      const uint32_t codes = quant_e2m1x8(v) & (d.x > 0.f ? 0xFFFFFFFFu : 0u);  // +0 codes
      if (live && c < a.nch && VG_ACCESS_OK(g_norm_status, out + c * 4, 4, a.q, q_extent(a, MODE)))
        st_stream(out + c * 4, codes);
    }
    return;
  }
  if (MODE == kBf16Pad) {
    const DynScale d = sm.dyn[slot];  // s = y, a = dy
    uint16_t *out = a.out16 + (live ? row * (int64_t)a.nch_pad * kElemsPerChunk : 0);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      const uint4 o = bf16x8_product_rn(t[k], d.s, d.a);
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, out + c * kElemsPerChunk, 16, a.out16,
                       VG_ROWS(a.T) * 16ull * (uint64_t)a.nch_pad))
        st_stream(out + c * kElemsPerChunk, o);
    }
    // the padded tail is zero
    for (int c = a.nch + lr; live && c < a.nch_pad; c += a.ntr)
      if (VG_ACCESS_OK(g_norm_status, out + c * kElemsPerChunk, 16, a.out16,
                       VG_ROWS(a.T) * 16ull * (uint64_t)a.nch_pad))
        st_stream(out + c * kElemsPerChunk, make_uint4(0, 0, 0, 0));
    return;
  }
  // padding chunks (c >= nch) read slot 0 and store nothing
  auto scale_of = [&](int c) -> const DynScale & {
    return sm.dyn[slot * nslots + (MODE == kPerToken || c >= a.nch ? 0 : c / GCH)];
  };
  if (MODE == kPerGroupX && a.ue8m0) {  // v = t * y / 2^k (ulp-level, no exact ties)
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      const DynScale d = scale_of(c);
      const float2 m2 = make_float2(d.ra, d.ra);
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 q = f2_mul(t[k][i], m2);
        v[2 * i] = q.x;
        v[2 * i + 1] = q.y;
      }
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, a.q + base + c * kElemsPerChunk, 8, a.q, q_extent(a, MODE)))
        st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
    }
    return;
  }
  // FP8 codes under the dynamic scales: the two-multiply form when the
  // launch asks for it and every chunk of this thread allows it (all but
  // degenerate rows), decided once so that the common loop is straight-line
  // code; otherwise the quotient form.  The scale-option instance keeps the
  // quotient form only (measured on GB300: UE8M0 column-major 32768 x 8192
  // 315 -> 303 us without the second form compiled in).
  float rf[VPT];
  bool fast = false;
  if (MODE != kPerGroupX && a.fastq) {
    fast = true;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const DynScale &d = scale_of(lr + k * a.ntr);
      rf[k] = d.rf;
      fast = fast && two_multiply_ok(d);
    }
  }
  if (fast) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      float v[8];
      dyn_values8_fast(t[k], rf[k], v);
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, a.q + base + c * kElemsPerChunk, 8, a.q, q_extent(a, MODE)))
        st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
    }
  } else {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      const DynScale d = scale_of(c);
      float v[8];
      dyn_values8_exact(t[k], d, v);
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, a.q + base + c * kElemsPerChunk, 8, a.q, q_extent(a, MODE)))
        st_stream(a.q + base + c * kElemsPerChunk, quant8(v));
    }
  }
}

__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

// DynScale-sized entries a row needs for its scales (NVFP4's float2 pairs
// take half an entry each).
__host__ __device__ inline int scale_slots(int mode, int ngroups) {
  return mode == kStatic ? 0
                         : (mode == kPerGroup || mode == kPerGroupX ? ngroups
                                                                    : (mode == kNvfp4 ? (ngroups + 1) / 2 : 1));
}

// Dynamic shared memory of the row logic: red, cmax, dyn.
__host__ __device__ inline size_t row_smem_bytes(int block, int vpt, int slots) {
  return 2 * 16 * sizeof(float4) + align128((size_t)block * vpt * 4) +
         align128((size_t)slots * sizeof(DynScale));
}

__device__ inline RowSmem carve_row_smem(unsigned char *p, int block, int vpt) {
  RowSmem sm;
  sm.red = reinterpret_cast<float4 *>(p);
  p += 2 * 16 * sizeof(float4);
  sm.cmax = reinterpret_cast<float *>(p);
  p += align128((size_t)block * vpt * 4);
  sm.dyn = reinterpret_cast<DynScale *>(p);
  return sm;
}

// ------------------------------------------------------- register kernel

template <int VPT, int MODE, int GCH, bool RES>
__global__ void __launch_bounds__(512) norm_fp8_kernel(const NormArgs a) {
  constexpr bool DYN = MODE != kStatic;
  extern __shared__ __align__(128) unsigned char dsm[];
  const RowSmem sm = carve_row_smem(dsm, blockDim.x, VPT);

  const int tid = threadIdx.x;
  const int slot = tid / a.ntr;       // row slot inside the CTA
  const int lr = tid - slot * a.ntr;  // thread index inside the row
  const int64_t row = (int64_t)blockIdx.x * a.rpc + slot;
  const bool live = row < a.T;
  const int64_t base = live ? row * a.H : 0;
  if (lr == 0 && live && (int)blockIdx.x < a.pf_ctas) {
    prefetch_l2(a.x + base, 2u * (uint32_t)a.H);
    if (RES) prefetch_l2(a.res + base, 2u * (uint32_t)a.H);
  }
  pdl_wait();

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
  pdl_launch_dependents();

  float2 t[VPT][4];
  float cmax[VPT];
  RowAcc acc;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const uint4 ow = pass1_chunk<DYN, RES, true>(xv[k], rv[k], wv[k], t[k], cmax[k], acc);
    const int c = lr + k * a.ntr;
    if (RES && live && c < a.nch &&
        VG_ACCESS_OK(g_norm_status, a.res_out + base + c * kElemsPerChunk, 16, a.res_out, row_extent(a)))
      st_stream(a.res_out + base + c * kElemsPerChunk, ow);
  }
  finish_rows<VPT, MODE, GCH>(a, t, cmax, acc, sm, 0, slot, lr, row, live, base);
}

// ------------------------------------------------------------ TMA kernel
//
// Dynamic shared memory: stages[S] (x row, then residual row), the weight
// row, the row logic's buffers, then S + 1 mbarriers (full[S], weight).

struct TmaLayout {
  size_t stage_bytes, w_off, row_off, bar_off, total;
  __host__ __device__ TmaLayout(int H, bool res, int stages, int block, int vpt, int slots) {
    stage_bytes = align128((size_t)(res ? 4 : 2) * H);
    w_off = stage_bytes * stages;
    row_off = w_off + align128((size_t)2 * H);
    bar_off = row_off + align128(row_smem_bytes(block, vpt, slots));
    total = bar_off + (size_t)(stages + 1) * 8;
  }
};

template <int VPT, int MODE, int GCH, bool RES>
__global__ void __launch_bounds__(512) norm_fp8_tma_kernel(const NormArgs a, const int stages) {
  constexpr bool DYN = MODE != kStatic;
  extern __shared__ __align__(128) unsigned char dsm[];
  const int slots = scale_slots(MODE, a.ngroups);
  const TmaLayout L(a.H, RES, stages, blockDim.x, VPT, slots);
  const RowSmem sm = carve_row_smem(dsm + L.row_off, blockDim.x, VPT);
  unsigned char *wbuf = dsm + L.w_off;
  uint64_t *full = reinterpret_cast<uint64_t *>(dsm + L.bar_off);
  uint64_t *wbar = full + stages;
  const uint32_t row_bytes = 2u * (uint32_t)a.H;

  const int lr = threadIdx.x;  // one row at a time: ntr == blockDim.x
  const int64_t first = blockIdx.x, stride = gridDim.x;

  auto issue = [&](int s, int64_t row) {
    unsigned char *st = dsm + (size_t)s * L.stage_bytes;
    // (debug builds: a copy whose source is out of range is replaced by a
    // plain arrival, so that the stage's wait still completes)
    if (!VG_ACCESS_OK(g_norm_status, a.x + row * a.H, row_bytes, a.x, row_extent(a)) ||
        (RES && !VG_ACCESS_OK(g_norm_status, a.res + row * a.H, row_bytes, a.res, row_extent(a)))) {
      mbar_arrive(&full[s]);
      return;
    }
    mbar_arrive_expect_tx(&full[s], RES ? 2 * row_bytes : row_bytes);
    tma_load_bulk(st, a.x + row * a.H, row_bytes, &full[s]);
    if (RES) tma_load_bulk(st + row_bytes, a.res + row * a.H, row_bytes, &full[s]);
  };

  VG_NEVER_BARRIER;
  if (lr == 0) {
    for (int s = 0; s <= stages; ++s) mbar_init(&full[s], 1);
    VG_NEVER_BARRIER_INIT();
    fence_mbar_init();
  }
  __syncthreads();
  // Launched with programmatic dependent launch: the barriers above are set
  // up while the previous grid drains; nothing in global memory is touched
  // before it has finished.  The next grid may then be scheduled: its CTAs
  // take the slots of CTAs of this one as they exit (the plan's shared
  // memory keeps exactly its CTAs on an SM).  The rows of the first stages
  // and the weight are asked into L2 before the wait.
  if (lr == 0 && a.pf_ctas > 0) {
    prefetch_l2(a.w, row_bytes);
    for (int s = 0; s < stages; ++s)
      if (first + s * stride < a.T) {
        prefetch_l2(a.x + (first + s * stride) * a.H, row_bytes);
        if (RES) prefetch_l2(a.res + (first + s * stride) * a.H, row_bytes);
      }
  }
  pdl_wait();
  if (lr == 0) {
    mbar_arrive_expect_tx(wbar, row_bytes);
    tma_load_bulk(wbuf, a.w, row_bytes, wbar);
    for (int s = 0; s < stages; ++s)
      if (first + s * stride < a.T) issue(s, first + s * stride);
  }
  pdl_launch_dependents();
  bool failed = __syncthreads_or(!mbar_wait_bounded(wbar, 0));

  int64_t i = 0;
  for (int64_t row = first; row < a.T && !failed; row += stride, ++i) {
    const int s = (int)(i % stages);
    const unsigned char *st = dsm + (size_t)s * L.stage_bytes;
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((i / stages) & 1)) && !VG_FORCED_TIMEOUT(i == 0);
    const int64_t base = row * a.H;

    float2 t[VPT][4];
    float cmax[VPT];
    RowAcc acc;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      uint4 xv = make_uint4(0, 0, 0, 0), rv = xv, wv = xv;
      if (ok && c < a.nch) {
        xv = lds128(st + c * 16);
        if (RES) rv = lds128(st + row_bytes + c * 16);
        wv = lds128(wbuf + c * 16);
      }
      const uint4 ow = pass1_chunk<DYN, RES>(xv, rv, wv, t[k], cmax[k], acc);
      if (RES && ok && c < a.nch &&
          VG_ACCESS_OK(g_norm_status, a.res_out + base + c * kElemsPerChunk, 16, a.res_out, row_extent(a)))
        st_stream(a.res_out + base + c * kElemsPerChunk, ow);
    }
    // Every thread has read stage s once this barrier is passed, so its
    // refill goes out now; a timed-out wait anywhere in the CTA ends the
    // loop for all threads.
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (lr == 0) {
      const int64_t next = row + (int64_t)stages * stride;
      if (next < a.T) {
        fence_proxy_async_smem();
        issue(s, next);
      }
    }
    finish_rows<VPT, MODE, GCH>(a, t, cmax, acc, sm, (int)(i & 1), 0, lr, row, true, base);
  }
  if (failed && lr == 0) {
    atomicOr(&g_norm_status, kErrWaitTimeout);
    // wait (bounded) for the copies this CTA may still have in flight
    for (int64_t k = i; k < i + stages; ++k)
      if (first + k * stride < a.T) mbar_wait_bounded(&full[k % stages], (uint32_t)((k / stages) & 1));
  }
}

// ------------------------------------------------------------ launchers

template <int VPT, int MODE, int GCH>
cudaError_t launch_res(const NormArgs &a, const RowPlan &p, cudaStream_t s) {
  const int slots = scale_slots(MODE, a.ngroups) * p.rpc;
  const size_t smem = row_smem_bytes(p.block(), VPT, slots);
  // row CTAs: the next grid may be scheduled while this one drains
  const dim3 g((unsigned)p.grid), b((unsigned)p.block());
  return a.res != nullptr ? launch_pdl(norm_fp8_kernel<VPT, MODE, GCH, true>, g, b, smem, s, a)
                          : launch_pdl(norm_fp8_kernel<VPT, MODE, GCH, false>, g, b, smem, s, a);
}

template <int VPT, int MODE, int GCH, bool RES>
cudaError_t launch_tma_res(const NormArgs &a, const TmaPlan &p, cudaStream_t s) {
  const int slots = scale_slots(MODE, a.ngroups);
  const TmaLayout L(a.H, RES, p.stages, p.block, VPT, slots);
  auto kern = norm_fp8_tma_kernel<VPT, MODE, GCH, RES>;
  // opt in to large dynamic shared memory once per instantiation and device
  static std::atomic<uint64_t> opted_in{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(opted_in.load(std::memory_order_acquire) & bit)) {
    e = opt_in_dynamic_smem(reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit, std::memory_order_release);
  }
  return launch_pdl(kern, dim3((unsigned)p.grid), dim3((unsigned)p.block),
                    p.smem > L.total ? p.smem : L.total, s, a, p.stages);
}

template <int VPT, int MODE, int GCH>
cudaError_t launch_tma_mode(const NormArgs &a, const TmaPlan &p, cudaStream_t s) {
  return a.res != nullptr ? launch_tma_res<VPT, MODE, GCH, true>(a, p, s)
                          : launch_tma_res<VPT, MODE, GCH, false>(a, p, s);
}

template <int VPT>
cudaError_t launch_mode(const NormArgs &a, int mode, const RowPlan &p, cudaStream_t s) {
  switch (mode) {
    case kStatic: return launch_res<VPT, kStatic, 1>(a, p, s);
    case kPerToken: return launch_res<VPT, kPerToken, 1>(a, p, s);
    case kBf16Pad: return launch_res<VPT, kBf16Pad, 1>(a, p, s);
    case kNvfp4: return launch_res<VPT, kNvfp4, 2>(a, p, s);
    default:
      if (a.ue8m0 || a.s_gs != 1)
        return a.gch == 8 ? launch_res<VPT, kPerGroupX, 8>(a, p, s)
                          : launch_res<VPT, kPerGroupX, 16>(a, p, s);
      return a.gch == 8 ? launch_res<VPT, kPerGroup, 8>(a, p, s)
                        : launch_res<VPT, kPerGroup, 16>(a, p, s);
  }
}

// (static scales never take the TMA kernel: the register kernel streams at
// the copy roofline there)
template <int VPT>
cudaError_t launch_tma_vpt(const NormArgs &a, int mode, const TmaPlan &p, cudaStream_t s) {
  switch (mode) {
    case kPerToken: return launch_tma_mode<VPT, kPerToken, 1>(a, p, s);
    case kBf16Pad: return launch_tma_mode<VPT, kBf16Pad, 1>(a, p, s);
    case kNvfp4: return launch_tma_mode<VPT, kNvfp4, 2>(a, p, s);
    default:
      if (a.ue8m0 || a.s_gs != 1)
        return a.gch == 8 ? launch_tma_mode<VPT, kPerGroupX, 8>(a, p, s)
                          : launch_tma_mode<VPT, kPerGroupX, 16>(a, p, s);
      return a.gch == 8 ? launch_tma_mode<VPT, kPerGroup, 8>(a, p, s)
                        : launch_tma_mode<VPT, kPerGroup, 16>(a, p, s);
  }
}

}  // namespace

cudaError_t launch_norm_fp8(NormArgs a, int mode, const RowPlan &p, cudaStream_t s) {
  a.ntr = p.ntr;
  a.rpc = p.rpc;
  a.fastq = 1;
  switch (p.vpt) {
    case 1: return launch_mode<1>(a, mode, p, s);
    case 2: return launch_mode<2>(a, mode, p, s);
    case 4: return launch_mode<4>(a, mode, p, s);
    default: return launch_mode<8>(a, mode, p, s);
  }
}

size_t norm_tma_smem_bytes(int H, bool res, int stages, int block, int vpt, int slots) {
  return TmaLayout(H, res, stages, block, vpt, slots).total;
}

cudaError_t launch_norm_fp8_tma(NormArgs a, int mode, const TmaPlan &p, cudaStream_t s) {
  a.ntr = p.block;
  a.rpc = 1;
  // The two-multiply codes for rows of up to 128 threads (measured on
  // GB300, back to back: 5-6 % faster at H = 4096); rows of 256 threads run
  // 4-6 % faster with the quotient form (H = 8192).
  a.fastq = p.block < 256 ? 1 : 0;
  switch (p.vpt) {
    case 2: return launch_tma_vpt<2>(a, mode, p, s);
    case 4: return launch_tma_vpt<4>(a, mode, p, s);
    default: return launch_tma_vpt<8>(a, mode, p, s);
  }
}

uint32_t read_norm_status(bool reset) {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_norm_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_norm_status, &zero, sizeof(zero)) != cudaSuccess) return 0xFFFFFFFFu;
  }
  return v;
}

}  // namespace vg
