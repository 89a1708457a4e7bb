// common.cuh -- sm_103a device helpers shared by the libgqa kernels:
// mbarrier rings with bounded waits, bulk (TMA) copies, a device error word.
//
// Every wait in this library is bounded: after kWaitNs (2 s) of polling, the
// waiting thread records an error code in the kernel's error word and gives
// up, so a lost arrival degrades into a reported error instead of a hung GPU.
// No code path traps.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"  // kDefaultWaitNs

namespace gqa {

constexpr int kHq = 32;        // query heads
constexpr int kHkv = 8;        // KV heads
constexpr int kGroup = 4;      // query heads per KV head
constexpr int kD = 128;        // head dim
constexpr int kPage = 64;      // tokens per NVFP4 page

// Error codes written into a kernel's error word (bitwise OR).
constexpr uint32_t kErrWaitTimeout = 1u;
constexpr uint32_t kErrBadIndex = 2u;     // an out-of-range page index was skipped
constexpr uint32_t kErrBadIndptr = 4u;    // qo_indptr is not non-decreasing from 0 to total_q
constexpr uint32_t kErrSelfCheck = 8u;    // a debug export's internal cross-check failed

constexpr uint64_t kWaitNs = kDefaultWaitNs;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}


// try_wait that may suspend the thread (instead of returning at once) until
// the phase completes or about `hint_ns` nanoseconds pass, so waiting warps
// do not take issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// records kErrWaitTimeout in *err) if it has not completed within kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
    if (global_timer_ns() - t0 > kWaitNs) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}


// 1-D bulk copy global -> shared through the TMA unit, with an L2 eviction-
// priority hint (policy from createpolicy); completion is counted on `bar` as
// transaction bytes.  src, dst and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace gqa
