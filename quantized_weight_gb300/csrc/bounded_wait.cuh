// bounded_wait.cuh -- mbarrier waits that cannot hang a GPU.
//
// Every wait on an mbarrier in the qmm kernels gives up after kWaitLimitNs of
// wall time (the %globaltimer register).  A wait that gives up raises a
// CTA-wide abort flag in shared memory, which the other roles of the CTA poll
// while they wait, and records QMM_ERR_DEVICE_TIMEOUT in a device status word
// that the host reads back through qmm_check().  Each translation unit owns
// its own status word (kernels are compiled without relocatable device code).
#pragma once
#include <cstdint>

#include "sm100_ptx.cuh"

namespace qmm {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: every legitimate wait is far shorter
constexpr int kTimeoutStatus = -6;                 // QMM_ERR_DEVICE_TIMEOUT
constexpr uint32_t kSleepNs = 200000;              // longest sleep inside one try_wait

struct WaitCtl {
  volatile int *abort;   // shared memory, CTA-wide
  int *status;           // global memory, this translation unit's status word
};

// True once the phase with `parity` completed; false if this CTA aborted or
// the wait ran out of time (which then aborts the CTA and records the status).
// A waiting thread sleeps inside try_wait (woken when the phase completes), so
// waiting warps take no issue slots from the warps doing work.
// `limit_ns` shorter than kWaitLimitNs serves only the test hook that makes a
// wait run out on purpose.  With `stop_on_abort` false the wait ignores the
// CTA's abort flag (it still gives up at the limit): for the thread that
// issued the copies being waited for, which must not exit before they land.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                             uint64_t limit_ns = kWaitLimitNs, bool stop_on_abort = true) {
  if (sm100::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm100::globaltimer_ns();
  for (;;) {
    if (sm100::mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if (stop_on_abort && *c.abort) return false;
    if (sm100::globaltimer_ns() - t0 > limit_ns) {
      *c.abort = 1;
      atomicExch(c.status, kTimeoutStatus);
      return false;
    }
  }
}

// Used only while draining after an abort: bounded, records nothing.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = sm100::globaltimer_ns();
  while (!sm100::mbar_try_wait_sleep(bar, parity, kSleepNs))
    if (sm100::globaltimer_ns() - t0 > kWaitLimitNs) break;
}

}  // namespace qmm
