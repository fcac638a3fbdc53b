// il_ptx.cuh -- inline-PTX wrappers shared by the kernels that move data with
// the asynchronous copy engine: mbarriers (with bounded waits), bulk and tensor
// copies global -> shared, and the proxy fence between ordinary shared-memory
// accesses and those copies.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace il {

// A bounded wait gives up after about one second at 2 GHz.
constexpr unsigned long long kWaitLimitCycles = 2ull << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred P1;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n"
      "selp.b32 %0, 1, 0, P1;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete may sleep up to
// `ns` nanoseconds (woken early when the phase completes) instead of returning
// at once: waiting warps then take no issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred P1;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2, %3;\n"
      "selp.b32 %0, 1, 0, P1;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait that sleeps between tests (see mbar_try_wait_sleep); otherwise as
// mbar_wait below.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned* status, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 2000)) {
    if (*abort_flag) return mbar_try_wait(bar, parity);
    if ((unsigned long long)(clock64() - start) > kWaitLimitCycles) {
      *abort_flag = 1;
      atomicOr(status, code);
      return false;
    }
  }
  return true;
}

// Bounded wait for the phase with the given parity.  Returns false -- after
// raising the CTA's abort flag and or-ing `code` into the device status word --
// when the wait runs out, or when another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* status,
                                         unsigned code) {
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    // a phase that completed stays completed: re-check so that roles waiting on
    // the same phase agree even when the abort flag rises meanwhile
    if (*abort_flag) return mbar_try_wait(bar, parity);
    if ((unsigned long long)(clock64() - start) > kWaitLimitCycles) {
      *abort_flag = 1;
      atomicOr(status, code);
      return false;
    }
  }
  return true;
}

// Bounded wait with an explicit limit and no side effects (drain after an abort).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned long long limit) {
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity))
    if ((unsigned long long)(clock64() - start) > limit) return false;
  return true;
}

// One contiguous global -> shared copy of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority policy (weights streamed once).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                           uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Orders this thread's earlier ordinary shared-memory accesses before its later
// asynchronous-proxy operations (a bulk copy into the same bytes), and the reverse.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace il
