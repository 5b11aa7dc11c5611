// Bounded mbarrier waits shared by the tensor-core kernels (internal header).
//
// Every wait on an mbarrier phase in this library is bounded: a role that waits
// longer than the limit sets the CTA's abort flag, ORs MTPSD_STATUS_WAIT_TIMEOUT
// into the caller's status word and returns false, and the other roles of the
// CTA, seeing the abort flag at their next check, give up too.  The kernel then
// drains its own copies in flight (with waits bounded the same way), frees its
// TMEM and returns: no wait can hang the GPU, and no failure traps.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mtpsd {
namespace mbar {

// 2 s: far beyond any phase of a healthy launch (the longest are microseconds).
constexpr unsigned long long DEFAULT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One non-blocking-return probe of the phase with the given parity.  CLUSTER: acquire at cluster scope,
// for barriers whose bytes or arrivals come from the other CTA of a cluster.
template <bool CLUSTER>
__device__ __forceinline__ bool try_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  uint32_t ok;
  if constexpr (CLUSTER) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
        "p;\n}\n"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  }
  return ok != 0;
}

// The same probe, but a thread whose phase is not complete sleeps until it completes or hint_ns pass
// (the suspend-time hint), instead of returning at once: a waiting warp then takes no issue slots from
// the warps that work.
template <bool CLUSTER>
__device__ __forceinline__ bool try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  uint32_t ok;
  if constexpr (CLUSTER) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, "
        "0, p;\n}\n"
        : "=r"(ok) : "r"(a), "r"(parity), "r"(hint_ns) : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(a), "r"(parity), "r"(hint_ns) : "memory");
  }
  return ok != 0;
}

// Longest sleep of one probe: short against the time limit, so the abort flag and the limit are still
// checked often, and long against any phase of a healthy launch.
constexpr uint32_t SLEEP_HINT_NS = 20000;

// Waits for the phase; false when it gave up: the limit passed (this thread then sets *abort_flag and
// flags the status word) or another role of the CTA set *abort_flag first.  Both are checked after
// every sleeping probe.
template <bool CLUSTER>
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                     unsigned long long limit_ns) {
  if (try_wait<CLUSTER>(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (try_wait_sleep<CLUSTER>(bar, parity, SLEEP_HINT_NS)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      flag_status(status, MTPSD_STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
}

// A non-blocking probe of the phase with the given parity (CTA scope).
__device__ __forceinline__ bool test_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  return ok != 0;
}

}  // namespace mbar
}  // namespace mtpsd
