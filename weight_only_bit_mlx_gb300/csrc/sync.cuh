// sync.cuh - shared-memory barrier helpers with bounded waits (sm_103a).
//
// Every wait in the library's kernels goes through mbar_wait_bounded(): it sleeps in
// mbarrier.try_wait with a suspend-time hint (the thread wakes when the phase
// completes) and gives up once `budget_ns` of %globaltimer time has passed, or when
// another warp of the CTA has already given up (shared abort flag).  A kernel
// whose wait gives up records QL_ERR_TIMEOUT in the status word and returns; no
// wait in this library can spin forever.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace qlk {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// orders this thread's generic-proxy shared-memory accesses before later async-proxy
// (bulk copy, tensor core) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Suspends the thread until the phase completes or about kSuspendNs have passed.
constexpr uint32_t kSuspendNs = 100000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Wait until the barrier's phase with parity `parity` has completed.  Returns false
// (without having waited for it) if the budget ran out or *abort became nonzero.
// A completed phase costs one non-blocking test; otherwise the thread sleeps in
// mbarrier.try_wait (woken when the phase completes) instead of spinning, so waiting
// warps take no issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t budget_ns,
                                                  const volatile int *abort) {
  const uint32_t addr = smem_addr(bar);
  if (mbar_test_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(addr, parity)) return true;
    if (abort != nullptr && *abort != 0) return false;
    if (globaltimer_ns() - t0 > budget_ns) return false;
  }
}

// Named hardware barrier over `nthreads` threads (warps wait without issuing).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void record_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

}  // namespace qlk
