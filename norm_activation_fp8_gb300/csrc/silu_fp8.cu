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
//   sigmoid(g) = rcp(1 + 2^(-g log2 e))   (ex2.approx and rcp.approx, each
//                an ulp or two; a huge denominator flushes the reciprocal
//                to +0 and the product keeps the sign of g, as the exact -0
//                would)
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
//
// Decisions the pages' formats make exactly -- a power-of-two (UE8M0)
// group exponent, an NVFP4 block's E4M3 scale code -- are taken from the
// fp32 values wherever those are far enough from the decision boundary; the
// rare groups or blocks that are not are settled in fp64 after the chunk
// loop (the warp reloads their chunks and rewrites them), so that the fp64
// work and its registers stay off the streaming path.
#include <atomic>

#include "common.cuh"
#include "dyn_scale.cuh"
#include "launch.h"
#include "nvfp4.cuh"
#include "tma.cuh"

namespace vg {

// Status word of this translation unit's kernels (kErrWaitTimeout, and
// kErrBounds in debug builds).
__device__ uint32_t g_silu_status;

namespace {

// Extents in bytes of the tensors a launch touches (debug checks).
__device__ __forceinline__ uint64_t q_extent(const SiluArgs &a, bool fp4) {
  return VG_ROWS(a.T) * (uint64_t)(fp4 ? a.I / 2 : a.I);
}
__device__ __forceinline__ uint64_t scale_extent(const SiluArgs &a, int mode) {
  const uint64_t rows = VG_ROWS(a.T);
  if (mode == kPerToken) return 4 * rows;
  return rows == 0 ? 0 : 4 * ((rows - 1) * (uint64_t)a.s_ts + (uint64_t)(a.ngroups - 1) * a.s_gs + 1);
}

__device__ __forceinline__ float fast_rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// 2^x by the hardware approximation (ex2.approx, ~2 ulp), flushing
// subnormal inputs and results to zero: here every result is added to 1, so
// a flushed one changes nothing, and the flush-to-zero form needs no
// subnormal fix-up around the instruction.
__device__ __forceinline__ float ex2_ftz(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Two elements of silu(g) * u = g * rcp(1 + exp(-g)) * u.  FTZ: exp(-g) as
// 2^(-g log2 e) by ex2_ftz (measured faster for the static, per-group and
// NVFP4 paths); otherwise __expf (measured faster for the per-token paths).
template <bool FTZ>
__device__ __forceinline__ float2 silu_mul2(uint32_t gw, uint32_t uw) {
  const float2 g = bf16x2_to_f2(gw);
  float2 e;
  if constexpr (FTZ) {
    const float2 x = f2_mul(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    e = make_float2(ex2_ftz(x.x), ex2_ftz(x.y));
  } else {
    e = make_float2(__expf(-g.x), __expf(-g.y));
  }
  const float2 d = f2_add(e, make_float2(1.0f, 1.0f));
  return f2_mul(f2_mul(g, make_float2(fast_rcp(d.x), fast_rcp(d.y))), bf16x2_to_f2(uw));
}

template <bool FTZ = true>
__device__ __forceinline__ void silu_chunk(const uint4 &gv, const uint4 &uv, float (&v)[8]) {
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = silu_mul2<FTZ>(gw[i], uw[i]);
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

// The smallest k with 448 * 2^k >= max(amax, A_MIN) (exact comparisons).
__device__ __forceinline__ int pow2_exponent(double amax) {
  const double a = fmax(amax, (double)kAmaxFloor);
  int k;
  frexp(a * (1.0 / kE4M3Max), &k);
  for (int it = 0; it < 2; ++it) {
    if (ldexp((double)kE4M3Max, k) < a) ++k;
    else if (ldexp((double)kE4M3Max, k - 1) >= a) --k;
  }
  return k;
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) m = fmax3(m, fabsf(v[i]), fabsf(v[i + 1]));
  return m;
}

// The largest |silu(g) u| in fp64 over the chunk's elements whose fp32 value
// v is at least am (1 - 2^-15): with both v and am within 2^-19 of the exact
// values, no other element can hold the group's maximum.
__device__ __forceinline__ double candidates_amax_f64(uint4 gv, uint4 uv, const float (&v)[8],
                                                      float am) {
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
  const float cut = am * (1.0f - 1.0f / 32768.0f);
  double m = 0.0;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const float2 g = bf16x2_to_f2(gw[i]), u = bf16x2_to_f2(uw[i]);
    if (fabsf(v[2 * i]) >= cut) m = fmax(m, fabs((double)g.x / (1.0 + exp(-(double)g.x)) * (double)u.x));
    if (fabsf(v[2 * i + 1]) >= cut) m = fmax(m, fabs((double)g.y / (1.0 + exp(-(double)g.y)) * (double)u.y));
  }
  return m;
}

// Rewrites one per-group UE8M0 group whose fp32 amax lay within 2^-18 of a
// power-of-two boundary, with the exponent of the fp64 amax; called by the
// whole warp after its fast stores, `near` the same in all GCH lanes of a
// group (a near group is a live one: padding groups have amax 0).
template <int GCH>
__device__ __noinline__ void pow2_group_settle(const uint16_t *gate_up, uint8_t *q, float *scale,
                                               int32_t I, int32_t s_ts, int32_t s_gs, int64_t row,
                                               int c, bool near, uint64_t q_bytes,
                                               uint64_t s_bytes) {
  uint4 gv = make_uint4(0, 0, 0, 0), uv = gv;
  if (near) {
    gv = ld_stream_ro(gate_up + row * 2 * I + c * kElemsPerChunk);
    uv = ld_stream_ro(gate_up + row * 2 * I + I + c * kElemsPerChunk);
  }
  float v[8];
  silu_chunk(gv, uv, v);
  const float am = lanes_max(amax8(v), GCH);
  double m = near ? candidates_amax_f64(gv, uv, v, am) : 0.0;
  for (int o = GCH >> 1; o > 0; o >>= 1) m = fmax(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (!near) return;
  const int e = pow2_exponent(m);
  float *sp = scale + row * s_ts + (int64_t)(c / GCH) * s_gs;
  if ((c & (GCH - 1)) == 0 && VG_ACCESS_OK(g_silu_status, sp, 4, scale, s_bytes)) *sp = exp2i(e);
  scale8(v, exp2i(-e));
  uint8_t *qp = q + row * (int64_t)I + c * kElemsPerChunk;
  if (VG_ACCESS_OK(g_silu_status, qp, 8, q, q_bytes)) st_stream(qp, quant8(v));
}

// Rewrites one NVFP4 block whose fp32 value gs * amax / 6 lay near an E4M3
// midpoint, with the code the exact value rounds to; called by the whole warp
// after its fast stores (so little is live across the call), `near` the same
// in both lanes of a block.  The lane reloads its chunk c of the row; only
// candidates for the block's maximum go to fp64: an element whose fp32 |a|
// is below am (1 - 2^-15) (am the fp32 block amax; both carry under 2^-19 of
// error) cannot be it.
__device__ __noinline__ void nvfp4_silu_settle(const uint16_t *gate_up, uint8_t *q4, uint8_t *sf,
                                               int32_t I, int64_t row, int c, float gs, bool near,
                                               uint64_t q_bytes, uint64_t sf_bytes) {
  uint4 gv = make_uint4(0, 0, 0, 0), uv = gv;
  if (near) {
    gv = ld_stream_ro(gate_up + row * 2 * I + c * kElemsPerChunk);
    uv = ld_stream_ro(gate_up + row * 2 * I + I + c * kElemsPerChunk);
  }
  float v[8];
  silu_chunk(gv, uv, v);
  const float am = lanes_max(amax8(v), 2);
  double m = near ? candidates_amax_f64(gv, uv, v, am) : 0.0;
  m = fmax(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  if (!near) return;
  const double x = (double)gs * m / (double)kE2M1Max;
  const float xh = (float)x;
  const uint32_t code = e4m3_code_df(xh, (float)(x - (double)xh));
  const float sv = e4m3_value(code);
  scale8(v, sv > 0.f ? gs * fast_rcp(sv) : 0.f);
  uint8_t *fp = sf + row * (int64_t)(I / kNvfp4Block) + c / 2;
  if ((c & 1) == 0 && VG_ACCESS_OK(g_silu_status, fp, 1, sf, sf_bytes)) *fp = (uint8_t)code;
  uint8_t *qp = q4 + row * (int64_t)(I / 2) + c * 4;
  if (VG_ACCESS_OK(g_silu_status, qp, 4, q4, q_bytes))
    st_stream(qp, quant_e2m1x8(v) & (sv > 0.f ? 0xFFFFFFFFu : 0u));
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
// OPT: per-group with scale options (UE8M0 and/or column-major), an
// instance of its own so that plain per-group code stays as it is.
// DENSE: row-segment rows (static, per-group, scale options, NVFP4) of at
// most two chunks a thread in 32 registers, four CTAs per SM: more row
// segments in flight per SM (measured on GB300 from two rows per SM:
// per-group 2048 x 14336 0.94 -> 1.00, 32768 x 28672 0.93 -> 0.99; NVFP4
// 32768 x 28672 0.88 -> 0.93; UE8M0 column-major 32768 x 14336 0.92 ->
// 0.96; static, against four chunks a thread at three CTAs, 2048 x 14336
// 0.94 -> 1.01, 512 x 14336 0.68 -> 0.81, 4096 x 14336 0.99 -> 1.01,
// 32768 x 14336 1.04 -> 1.03; below two rows per SM, a single partial
// wave, three CTAs' larger register budget is faster).
template <int VPT, int MODE, int GCH, bool BIG, bool OPT = false, bool DENSE = false>
__global__ void __launch_bounds__(BIG ? 1024 : 512, BIG ? 1 : (MODE == kPerToken ? 2 : (DENSE ? 4 : 3)))
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
  // Launched with programmatic dependent launch: the next grid is scheduled
  // while this one drains, and its first CTAs ask for their segment of the
  // row into L2 before they wait for this one to finish.
  if (lr0 == 0 && live && (int)blockIdx.x < a.pf_ctas && lr < a.nch) {
    const int c1 = lr + a.ntr * VPT < a.nch ? lr + a.ntr * VPT : a.nch;
    const uint32_t bytes = 16u * (uint32_t)(c1 - lr);
    prefetch_l2(a.gate_up + in_base + lr * kElemsPerChunk, bytes);
    prefetch_l2(a.gate_up + in_base + a.I + lr * kElemsPerChunk, bytes);
  }
  pdl_wait();

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

  pdl_launch_dependents();
  if constexpr (MODE == kNvfp4) {
    // 16-column blocks = chunk pairs (2b, 2b + 1), held by lanes lr, lr ^ 1.
    // x = gs * amax / 6 in fp32 is within ~2^-19 of the exact value (the
    // activations' error); where x(1 - 2^-17) and x(1 + 2^-17) round to
    // different E4M3 codes the block is settled in fp64 after the loop, so
    // that its code is the exact value's.
    const float gs = __ldg(a.scale);
    const float gs6 = gs * (1.0f / kE2M1Max);
    uint8_t *out = a.q + (live ? row * (int64_t)(a.I / 2) : 0);
    uint32_t near_k = 0;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      float v[8];
      silu_chunk(gv[k], uv[k], v);
      const float am = lanes_max(amax8(v), 2);
      const float x = am * gs6;
      const uint32_t cc = cvt_e4m3x2(x * (1.0f - 1.0f / 131072.0f), x * (1.0f + 1.0f / 131072.0f));
      const uint32_t code = cc & 0xFFu;
      if ((cc >> 8) != code) near_k |= 1u << k;
      const float sv = e4m3_value(code);
      scale8(v, sv > 0.f ? gs * fast_rcp(sv) : 0.f);
      const uint32_t codes = quant_e2m1x8(v) & (sv > 0.f ? 0xFFFFFFFFu : 0u);  // +0 codes
      if (live && c < a.nch) {
        uint8_t *fp = a.sf8 + row * (int64_t)(a.I / kNvfp4Block) + c / 2;
        if ((c & 1) == 0 && VG_ACCESS_OK(g_silu_status, fp, 1, a.sf8, VG_ROWS(a.T) * (uint64_t)(a.I / kNvfp4Block)))
          *fp = (uint8_t)code;
        if (VG_ACCESS_OK(g_silu_status, out + c * 4, 4, a.q, q_extent(a, true))) st_stream(out + c * 4, codes);
      }
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k)
      if (__any_sync(0xFFFFFFFFu, (near_k >> k) & 1u))
        nvfp4_silu_settle(a.gate_up, a.q, a.sf8, a.I, row, lr + k * a.ntr, gs, (near_k >> k) & 1u,
                          q_extent(a, true), VG_ROWS(a.T) * (uint64_t)(a.I / kNvfp4Block));
    return;
  }
  if constexpr (OPT) {
    uint32_t near_k = 0;
    // Per-group with scale options.  UE8M0: s = 2^e, the smallest power of
    // two with 448 s >= max(amax, A_MIN).  The fp32 amax is within ~2^-19
    // of the exact one, so a group whose amax lies within 2^-18 of a
    // boundary 448 * 2^k is settled in fp64 after the loop.
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int c = lr + k * a.ntr;
      float v[8];
      silu_chunk(gv[k], uv[k], v);
      const float am = lanes_max(amax8(v), GCH);
      float s, m;
      if (a.ue8m0) {
        const float fa = fmaxf(am, kAmaxFloor);
        const int e = pow2_exponent_448(fa);
        if (near_pow2_boundary_448(fa)) near_k |= 1u << k;
        s = exp2i(e);
        m = exp2i(-e);
      } else {
        s = silu_scale(am);
        m = fast_rcp(s);
      }
      float *sp = a.scale + row * a.s_ts + (int64_t)(c / GCH) * a.s_gs;
      if (live && c < a.nch && (c & (GCH - 1)) == 0 &&
          VG_ACCESS_OK(g_silu_status, sp, 4, a.scale, scale_extent(a, MODE)))
        *sp = s;
      scale8(v, m);
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_silu_status, a.q + out_base + c * kElemsPerChunk, 8, a.q, q_extent(a, false)))
        st_stream(a.q + out_base + c * kElemsPerChunk, quant8(v));
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k)
      if (__any_sync(0xFFFFFFFFu, (near_k >> k) & 1u))
        pow2_group_settle<GCH>(a.gate_up, a.q, a.scale, a.I, a.s_ts, a.s_gs, row, lr + k * a.ntr,
                               (near_k >> k) & 1u, q_extent(a, false), scale_extent(a, MODE));
    return;
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
        if (live && c < a.nch && (c & (GCH - 1)) == 0 &&
            VG_ACCESS_OK(g_silu_status, a.scale + row * a.ngroups + c / GCH, 4, a.scale, scale_extent(a, MODE)))
          a.scale[row * a.ngroups + c / GCH] = s;
        m = fast_rcp(s);
      }
      scale8(v, m);
      if (live && c < a.nch &&
          VG_ACCESS_OK(g_silu_status, a.q + out_base + c * kElemsPerChunk, 8, a.q, q_extent(a, false)))
        st_stream(a.q + out_base + c * kElemsPerChunk, quant8(v));
    }
    return;
  }

  // Per-token: activations stay in registers until the row amax is known.
  float act[VPT][8];
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    silu_chunk<false>(gv[k], uv[k], act[k]);
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
  if (live && lr == 0 && VG_ACCESS_OK(g_silu_status, a.scale + row, 4, a.scale, scale_extent(a, MODE)))
    a.scale[row] = s;
  const float m = fast_rcp(s);
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int c = lr + k * a.ntr;
    scale8(act[k], m);
    if (live && c < a.nch &&
        VG_ACCESS_OK(g_silu_status, a.q + out_base + c * kElemsPerChunk, 8, a.q, q_extent(a, false)))
      st_stream(a.q + out_base + c * kElemsPerChunk, quant8(act[k]));
  }
}

// ------------------------------------------------ TMA per-token kernel
//
// Persistent CTAs, one row at a time, for per-token rows at large T.  A row
// is NSEG column segments; segment s of the current row sits in stage s of
// shared memory (its gate part, then its up part), copied by two bulk TMA
// copies.  As soon as every thread has pulled segment s's activations into
// registers, the stage is refilled with segment s of the next row, so the
// copies overlap the rest of pass 1, the amax reduction, the quantisation
// and the stores.  NSEG = 2 keeps a 112 KB row (I = 28672) within one SM's
// shared memory while still overlapping its copy with compute.  Dynamic
// shared memory: NSEG stages, then NSEG full mbarriers.

template <int VPT, bool BIG, int NSEG>
__global__ void __launch_bounds__(BIG ? 1024 : 512, BIG ? 1 : 2)
    silu_fp8_tma_token_kernel(const SiluArgs a) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ float red[2][32];
  constexpr int KS = VPT / NSEG;                      // chunks per thread per segment
  const int seg_ch = a.nch / NSEG;                     // chunks per segment
  const uint32_t seg_bytes = 16u * (uint32_t)seg_ch;   // one half (gate or up) of a stage
  uint64_t *full = reinterpret_cast<uint64_t *>(dsm + (size_t)NSEG * 2 * seg_bytes);
  const int tid = threadIdx.x;
  const int64_t first = blockIdx.x, stride = gridDim.x;

  auto issue = [&](int sg, int64_t row) {
    unsigned char *st = dsm + (size_t)sg * 2 * seg_bytes;
    const uint16_t *src = a.gate_up + row * 2 * a.I + (int64_t)sg * seg_ch * kElemsPerChunk;
    // (debug builds: a copy whose source is out of range is replaced by a
    // plain arrival, so that the stage's wait still completes)
    [[maybe_unused]] const uint64_t in_bytes = VG_ROWS(a.T) * 4ull * (uint64_t)a.I;
    if (!VG_ACCESS_OK(g_silu_status, src, seg_bytes, a.gate_up, in_bytes) ||
        !VG_ACCESS_OK(g_silu_status, src + a.I, seg_bytes, a.gate_up, in_bytes)) {
      mbar_arrive(&full[sg]);
      return;
    }
    mbar_arrive_expect_tx(&full[sg], 2 * seg_bytes);
    tma_load_bulk(st, src, seg_bytes, &full[sg]);
    tma_load_bulk(st + seg_bytes, src + a.I, seg_bytes, &full[sg]);
  };
  VG_NEVER_BARRIER;
  if (tid == 0) {
    for (int sg = 0; sg < NSEG; ++sg) mbar_init(&full[sg], 1);
    VG_NEVER_BARRIER_INIT();
    fence_mbar_init();
  }
  __syncthreads();
  // Programmatic dependent launch, as the persistent norm kernel: nothing in
  // global memory before the previous grid has finished (its first row is
  // only asked into L2); the next grid's CTAs take the slots of this one's
  // as they exit.
  if (tid == 0 && first < a.T && a.pf_ctas > 0)
    prefetch_l2(a.gate_up + first * 2 * a.I, 4u * (uint32_t)a.I);
  pdl_wait();
  if (tid == 0 && first < a.T)
    for (int sg = 0; sg < NSEG; ++sg) issue(sg, first);
  pdl_launch_dependents();

  bool failed = false;
  int fail_sg = 0;      // the segment whose wait gave up
  bool ahead = false;   // stages before fail_sg already hold the next row's copies
  int64_t i = 0;
  for (int64_t row = first; row < a.T && !failed; row += stride, ++i) {
    float act[VPT][8];
    float am = 0.f;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg) {
      const unsigned char *st = dsm + (size_t)sg * 2 * seg_bytes;
      const bool ok = mbar_wait_bounded(&full[sg], (uint32_t)(i & 1)) && !VG_FORCED_TIMEOUT(i == 0 && sg == 0);
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        const int c = tid + k * a.ntr;  // chunk within the segment
        const uint4 gv = (ok && c < seg_ch) ? lds128(st + c * 16) : make_uint4(0, 0, 0, 0);
        const uint4 uv = (ok && c < seg_ch) ? lds128(st + seg_bytes + c * 16) : make_uint4(0, 0, 0, 0);
        silu_chunk<false>(gv, uv, act[sg * KS + k]);
        am = fmaxf(am, amax8(act[sg * KS + k]));
      }
      // every thread has read segment sg: refill its stage with the next row
      if (__syncthreads_or(!ok)) {
        failed = true;
        fail_sg = sg;
        ahead = row + stride < a.T;
        break;
      }
      if (tid == 0 && row + stride < a.T) {
        fence_proxy_async_smem();
        issue(sg, row + stride);
      }
    }
    if (failed) break;
    am = warp_max(am);
    float *r = red[i & 1];
    if ((tid & 31) == 0) r[tid >> 5] = am;
    __syncthreads();
    am = 0.f;
    for (int w = 0; w < (a.ntr >> 5); ++w) am = fmaxf(am, r[w]);
    const float s = silu_scale(am);
    if (tid == 0 && VG_ACCESS_OK(g_silu_status, a.scale + row, 4, a.scale, scale_extent(a, kPerToken)))
      a.scale[row] = s;
    const float m = fast_rcp(s);
    const int64_t out_base = row * a.I;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        const int c = tid + k * a.ntr;
        scale8(act[sg * KS + k], m);
        if (c < seg_ch &&
            VG_ACCESS_OK(g_silu_status, a.q + out_base + ((int64_t)sg * seg_ch + c) * kElemsPerChunk, 8, a.q,
                         q_extent(a, false)))
          st_stream(a.q + out_base + ((int64_t)sg * seg_ch + c) * kElemsPerChunk,
                    quant8(act[sg * KS + k]));
      }
  }
  if (failed && tid == 0) {
    atomicOr(&g_silu_status, kErrWaitTimeout);
    // the copies this CTA may still have in flight: one per stage, of the
    // next row for stages already refilled, else of the current row
    for (int sg = 0; sg < NSEG; ++sg)
      mbar_wait_bounded(&full[sg], (uint32_t)((i + (sg < fail_sg && ahead ? 1 : 0)) & 1));
  }
}

template <int VPT, bool BIG, int NSEG>
cudaError_t launch_tma_token(const SiluArgs &a, const SiluTmaPlan &p, cudaStream_t s) {
  auto kern = silu_fp8_tma_token_kernel<VPT, BIG, NSEG>;
  static std::atomic<uint64_t> opted_in{0};  // once per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(opted_in.load(std::memory_order_acquire) & bit)) {
    e = opt_in_dynamic_smem(reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    opted_in.fetch_or(bit, std::memory_order_release);
  }
  const size_t need = silu_tma_token_smem_bytes(a.I, NSEG);
  return launch_pdl(kern, dim3((unsigned)p.grid), dim3((unsigned)p.block),
                    p.smem > need ? p.smem : need, s, a);
}

template <int VPT>
cudaError_t launch_mode(const SiluArgs &a, int mode, const RowPlan &p, cudaStream_t s) {
  const dim3 g((unsigned)p.grid, (unsigned)p.segs), b((unsigned)p.block());
  switch (mode) {
    case kStatic:
      if constexpr (VPT <= 2)
        if (p.dense) return launch_pdl(silu_fp8_kernel<VPT, kStatic, 1, false, false, true>, g, b, 0, s, a);
      return launch_pdl(silu_fp8_kernel<VPT, kStatic, 1, false>, g, b, 0, s, a);
    case kNvfp4:  // the per-group plan: at most two chunks a thread
      if constexpr (VPT <= 2)
        return p.dense ? launch_pdl(silu_fp8_kernel<VPT, kNvfp4, 2, false, false, true>, g, b, 0, s, a)
                       : launch_pdl(silu_fp8_kernel<VPT, kNvfp4, 2, false>, g, b, 0, s, a);
      else
        return cudaErrorInvalidConfiguration;
    case kPerToken:
      return p.block() > 512 ? launch_pdl(silu_fp8_kernel<VPT, kPerToken, 1, true>, g, b, 0, s, a)
                             : launch_pdl(silu_fp8_kernel<VPT, kPerToken, 1, false>, g, b, 0, s, a);
    default:
      if (a.ue8m0 || a.s_gs != 1) {
        if constexpr (VPT <= 2)
          if (p.dense)
            return a.gch == 8 ? launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 8, false, true, true>, g, b, 0, s, a)
                              : launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 16, false, true, true>, g, b, 0, s, a);
        return a.gch == 8 ? launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 8, false, true>, g, b, 0, s, a)
                          : launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 16, false, true>, g, b, 0, s, a);
      }
      if constexpr (VPT <= 2)
        if (p.dense)
          return a.gch == 8
                     ? launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 8, false, false, true>, g, b, 0, s, a)
                     : launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 16, false, false, true>, g, b, 0, s, a);
      return a.gch == 8 ? launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 8, false>, g, b, 0, s, a)
                        : launch_pdl(silu_fp8_kernel<VPT, kPerGroup, 16, false>, g, b, 0, s, a);
  }
  return cudaGetLastError();
}

}  // namespace

size_t silu_tma_token_smem_bytes(int I, int nseg) { return (size_t)4 * I + 8 * (size_t)nseg; }

cudaError_t launch_silu_fp8_tma_token(SiluArgs a, const SiluTmaPlan &p, cudaStream_t s) {
  a.ntr = p.block;
  a.rpc = 1;
  if (p.nseg == 2)  // four chunks a thread, two per segment
    return p.block > 512 ? launch_tma_token<4, true, 2>(a, p, s) : launch_tma_token<4, false, 2>(a, p, s);
  switch (p.vpt) {
    case 1: return p.block > 512 ? launch_tma_token<1, true, 1>(a, p, s) : launch_tma_token<1, false, 1>(a, p, s);
    case 2: return p.block > 512 ? launch_tma_token<2, true, 1>(a, p, s) : launch_tma_token<2, false, 1>(a, p, s);
    default: return p.block > 512 ? launch_tma_token<4, true, 1>(a, p, s) : launch_tma_token<4, false, 1>(a, p, s);
  }
}

uint32_t read_silu_status(bool reset) {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_silu_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_silu_status, &zero, sizeof(zero)) != cudaSuccess) return 0xFFFFFFFFu;
  }
  return v;
}

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
