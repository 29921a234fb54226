// Inline-PTX helpers for sm_103a shared by the GEMM and the data-movement
// kernels: mbarriers with bounded waits (per thread and per converged warp),
// warp leader election, and the untiled bulk (TMA) copy from global to
// shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dt {

// Bound of every mbarrier wait unless the caller passes its own.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Gives up (and
// returns false) when another role has raised the CTA's abort flag or after
// WAIT_LIMIT_NS; the caller then records DT_DEV_ERR_TIMEOUT and unwinds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// One thread of a converged warp: the leader issues what one thread must
// issue (copies, MMAs, commits) while the whole warp walks the loop, so the
// loop's values stay warp-uniform.  Taken once per warp and kept: every
// commit must come from the thread that issued the MMAs it tracks.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// mbar_wait for a whole converged warp: every lane tests the barrier and the
// warp leaves together (a phase, once seen complete, stays complete until
// the warp itself lets the barrier move on).  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer();
  uint32_t spins = 0;
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if ((++spins & 255u) == 0) {
      const int give_up = (*abort_flag != 0) || (globaltimer() - t0 > limit_ns);
      if (__any_sync(0xffffffffu, give_up)) return false;
    }
  }
}

// Untiled bulk copy global -> this CTA's shared memory, completion counted
// on `bar` (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  uint64_t g;
  asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(g) : "l"(gsrc));
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(g), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

}  // namespace dt
