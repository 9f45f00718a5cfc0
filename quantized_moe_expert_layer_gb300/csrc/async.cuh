// Asynchronous-copy and mbarrier helpers (sm_103a): shared-memory mbarriers
// with bounded waits (the tensor-core kernels' TMA and MMA hand-offs) and
// cp.async (16 or 4 bytes, per thread).
#pragma once

#include <stdint.h>

namespace moe {
namespace {

// Default budget of one bounded wait (clock64 cycles, about 1 s).  The
// waits of a forward take the layer's budget (moe_set_wait_budget); the drains
// before a CTA exits always take this one, so that no CTA leaves with a copy or
// an MMA in flight.
constexpr long long kWaitBudget = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// arrive and add `bytes` to the transaction count the current phase waits for
__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
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
// Bounded wait for the phase of the given parity to complete.  Returns false
// (after setting *abort) when `budget` cycles pass, or at once if another
// thread aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          long long budget) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > budget) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
// The same with a suspend-time hint: a waiting thread sleeps in the barrier
// (woken when the phase completes) instead of spinning, so it leaves its
// sub-partition's issue slots to the other warps.
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                long long budget) {
  const long long t0 = clock64();
  while (!mbar_test_sleep(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > budget) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
// The same, first testing the phase without blocking (for waits whose phase
// has usually completed long before: no clock read, no suspend on the fast path).
__device__ __forceinline__ bool mbar_done(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               long long budget) {
  return mbar_done(bar, parity) || mbar_wait(bar, parity, abort, budget);
}
// Bounded wait that ignores the abort flag (draining copies before exit).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity) && clock64() - t0 < kWaitBudget) {
  }
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async (per thread)
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
// 4 bytes (both addresses 4-byte aligned)
__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace
}  // namespace moe
