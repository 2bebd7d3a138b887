// common.cuh -- device helpers shared by the fused norm / SiLU -> FP8 kernels.
//
// bf16 pairs travel packed in 32-bit words (element 0 in the low half), fp8
// codes packed four to a word (element 0 in the lowest byte), so every global
// access is a 16-byte (inputs) or 8-byte (fp8 outputs) vector.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "launch.h"

namespace vg {

constexpr float kE4M3Max = 448.0f;   // largest finite OCP E4M3FN value
constexpr float kAmaxFloor = 1e-10f; // floor on a dynamic amax (no 0/0 on zero rows)
constexpr int kElemsPerChunk = 8;    // bf16 elements per 16-byte vector

// max(a, b, c) by PTX's three-operand max (sm_100 and later); a NaN operand
// is ignored, so the result is NaN only when all three are.  Amaxes over
// pairs take one of these instead of two two-operand maxes.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------------ bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two fp32 values to bf16 (RNE) and pack them, `lo` in the low half.
// cvt...bf16x2.f32 d, a, b puts a in the upper half and b in the lower half.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// bf16(a + b) for two bf16 pairs: the exact sum rounded once to nearest
// even (IEEE addition in the bf16 format, subnormals kept), one instruction.
__device__ __forceinline__ uint32_t add_bf16x2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------ fp8

// Two fp32 -> two E4M3 codes, RNE with saturation to +-448 (NaN -> 0x7F),
// `lo` in the low byte.  Same operand order rule as the bf16x2 form.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Eight fp32 -> eight E4M3 codes packed into 8 bytes, element 0 first.
__device__ __forceinline__ uint2 quant8(const float (&v)[8]) {
  uint2 o;
  o.x = cvt_e4m3x2(v[0], v[1]) | (cvt_e4m3x2(v[2], v[3]) << 16);
  o.y = cvt_e4m3x2(v[4], v[5]) | (cvt_e4m3x2(v[6], v[7]) << 16);
  return o;
}


// Programmatic dependent launch: the grid may be scheduled while the
// previous kernel in the stream finishes; its kernel waits
// (griddepcontrol.wait) for that kernel's completion before reading memory,
// so stream order is kept.
template <class... P, class... A>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 g, dim3 b, size_t smem, cudaStream_t s,
                              A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A &&>(args)...);
}

// The two halves of it inside a kernel: wait for the previous grid, and let
// the next one be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asks for [p, p + bytes) to be brought into L2: bulk prefetches of at most
// 16 KB each, with no destination and nothing to wait for.  p must be
// 16-byte aligned and bytes a multiple of 16.  A CTA issues this for its
// first rows before pdl_wait(), so that their DRAM round trip overlaps the
// previous grid's drain.  It cannot make the CTA read stale data: the
// prefetch only fills L2, the device's point of coherence, which also takes
// every write of the previous grid, and the CTA's own loads come after the
// wait.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  const char *c = static_cast<const char *>(p);
  for (uint32_t off = 0; off < bytes; off += 16384u) {
    const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(n) : "memory");
  }
}

// -------------------------------------------------------- debug checks
//
// Debug builds (-DVG_DEBUG_CHECKS, a test-only copy of the library): every
// global store, and the source of every bulk copy, is first checked against
// the extent of the tensor it touches.  An access outside it is skipped and
// sets kErrBounds in the translation unit's status word, so an indexing
// mistake shows up as a status flag, not as a fault or as overwritten
// memory.  Product builds compile each check to `true`.
// VG_DEBUG_SHRINK_EXTENT (tests only) reports every tensor one row short,
// so that the checks of a row's last accesses fire.
constexpr uint32_t kErrBounds = 4u;
#ifdef VG_DEBUG_SHRINK_EXTENT
#define VG_ROWS(T) ((uint64_t)(T) - 1u)
#else
#define VG_ROWS(T) ((uint64_t)(T))
#endif
#ifdef VG_DEBUG_CHECKS
__device__ __forceinline__ bool access_ok(uint32_t *status, const void *p, uint32_t n,
                                          const void *base, uint64_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(p), b = reinterpret_cast<uint64_t>(base);
  if (base != nullptr && a >= b && a + n <= b + bytes) return true;
  atomicOr(status, kErrBounds);
  return false;
}
#define VG_ACCESS_OK(status, p, n, base, bytes) \
  ::vg::access_ok(&(status), (const void *)(p), (uint32_t)(n), (const void *)(base), (uint64_t)(bytes))
#else
#define VG_ACCESS_OK(status, p, n, base, bytes) true
#endif

// -------------------------------------------------------------- memory ops

// Read-only data streamed once: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_ro(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Data streamed once that this kernel may also overwrite (the residual when
// updated in place): coherent load, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only data shared by every row (the RMSNorm weight): keep it cached.
__device__ __forceinline__ uint4 ld_keep(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::evict_last.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Outputs written once: streaming stores (evict-first in L2).
__device__ __forceinline__ void st_stream(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream(void *p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream(void *p, uint32_t v) {
  asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// --------------------------------------------------------------- reductions

// Butterfly reductions: every participating lane ends with the bit-identical
// result (each level combines the same two operands on both partners).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Max over aligned sets of `width` lanes (width a power of two <= 32).
__device__ __forceinline__ float lanes_max(float v, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Dequantisation scale of a dynamic row or group: fp32(max(amax, floor)/448).
__device__ __forceinline__ float dynamic_scale(float amax) {
  return fmaxf(amax, kAmaxFloor) / kE4M3Max;
}

// ------------------------------------------------ double-float arithmetic
//
// The dynamic-scale path needs the row's 1/sqrt(mean(r^2) + eps) to ~2^-44
// (fp64 is far too slow on this part), so it is carried as an unevaluated
// sum hi + lo of two fp32 numbers.

// hi + lo += x with the rounding error of the addition kept exactly in lo
// (Knuth's TwoSum; no multiply, so no contraction can change it).
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
  const float s = hi + x;
  const float bp = s - hi;
  const float e = (hi - (s - bp)) + (x - bp);
  hi = s;
  lo += e;
}

// Butterfly sum of (hi, lo) pairs over aligned sets of `width` lanes.
// TwoSum's error term is exact, so both partners of every exchange get
// bit-identical results.
__device__ __forceinline__ void lanes_sum2(float &hi, float &lo, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
    const float s = hi + oh;
    const float bp = s - hi;
    const float e = (hi - (s - bp)) + (oh - bp);
    hi = s;
    lo = (lo + ol) + e;
  }
}

// y + dy ~= 1/sqrt(S/n + eps) for S = s_hi + s_lo, to ~2^-44 relative, with
// |dy| <= half an ulp of y:
// m = S/n + eps in double-float (the FMA remainder of the division is exact
// because it spans few bits), y0 = rsqrt(m) to ~2^-22, then one Newton step
// y = y0 (1 + rho/2 + 3 rho^2/8) with rho = 1 - m y0^2 from exact products.
__device__ __forceinline__ void rsqrt_df(float s_hi, float s_lo, float n, float inv_n, float eps,
                                         float &y, float &dy) {
  const float q = s_hi * inv_n;
  const float ql = (fmaf(-q, n, s_hi) + s_lo) * inv_n;
  const float m = q + eps;
  const float bp = m - q;
  const float ml = ((q - (m - bp)) + (eps - bp)) + ql;
  const float y0 = rsqrtf(m);
  const float p = y0 * y0, pl = fmaf(y0, y0, -p);  // y0^2 = p + pl exactly
  const float t = m * p, tl = fmaf(m, p, -t);      // m p = t + tl exactly
  const float rho = (1.0f - t) - (tl + fmaf(m, pl, ml * p));
  const float c = y0 * rho * fmaf(0.375f, rho, 0.5f);
  y = y0 + c;               // renormalise: |c| << y0, so Fast2Sum is exact
  dy = (y0 - y) + c;
  // An infinite sum of squares (an infinite element) gives 1/sqrt(inf) = 0,
  // which the refinement above would turn into inf * 0 = NaN.  A NaN sum
  // stays NaN.
  if (s_hi == __int_as_float(0x7F800000)) y = dy = 0.f;
}

// --------------------------------------------------------- packed fp32 x2
//
// sm_100+ issues two fp32 operations per instruction; each lane is rounded
// exactly like the scalar instruction.

__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// A bf16 pair (element 0 in the low half) as two fp32 values.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

}  // namespace vg
