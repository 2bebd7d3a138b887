// tma.cuh -- bulk (non-tensor) TMA copies global -> shared, completed on an
// mbarrier, plus the bounded waits the pipelined kernels use.
//
// cp.async.bulk needs 16-byte aligned source and destination and a size that
// is a multiple of 16 bytes; every row copied here is n bf16 with n % 8 == 0
// starting at a 16-byte aligned row of a 16-byte aligned tensor.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vg {

// A wait gives up after this many failed try_wait polls (each poll may
// suspend the thread for a while): seconds, far beyond any healthy copy.
// (A test build lowers it.)
#ifndef VG_WAIT_LIMIT
#define VG_WAIT_LIMIT (1u << 22)
#endif
constexpr uint32_t kWaitLimit = VG_WAIT_LIMIT;

// Error bits a kernel leaves in its translation unit's status word.
constexpr uint32_t kErrWaitTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async proxy (the TMA unit).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared memory accesses before
// later async-proxy (TMA) accesses to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Plain arrival (no transaction bytes), e.g. a consumer releasing a stage.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the barrier's phase with the given parity; false after
// kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bulk copy of `bytes` from global to shared memory, counted on `bar`.
__device__ __forceinline__ void tma_load_bulk(void *dst_smem, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Test-only builds (VG_TEST_FORCE_WAIT_TIMEOUT): a barrier that nothing
// arrives on.  A pipelined kernel waits on it after its first stage wait, so
// that wait runs out and the CTA takes its failure path while its other
// copies are in flight.  Product builds compile all of this away.
#ifdef VG_TEST_FORCE_WAIT_TIMEOUT
#define VG_NEVER_BARRIER __shared__ uint64_t vg_never_bar
#define VG_NEVER_BARRIER_INIT() mbar_init(&vg_never_bar, 1)
#define VG_FORCED_TIMEOUT(first) ((first) && !mbar_wait_bounded(&vg_never_bar, 0))
#else
#define VG_NEVER_BARRIER
#define VG_NEVER_BARRIER_INIT()
#define VG_FORCED_TIMEOUT(first) false
#endif

__device__ __forceinline__ uint4 lds128(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

}  // namespace vg
