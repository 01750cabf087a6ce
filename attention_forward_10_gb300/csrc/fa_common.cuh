// fa_common.cuh -- pieces shared by the attention forward kernels: bounded
// mbarrier waits with a CTA-wide abort flag.
#pragma once

#include <cstdint>

#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

constexpr int kStatusTimeout = 5;  // == FA_ERR_DEVICE_TIMEOUT

struct Ctl {
  volatile int* abort_flag;  // shared memory, CTA-wide
  int* status;               // global status word
  unsigned long long timeout_ns;
};

static __device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl& c,
                                       int site) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*c.abort_flag) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      *c.abort_flag = 1;
      atomicCAS(c.status, 0, kStatusTimeout | (site << 8));
      return false;
    }
  }
}

// Bounded wait for the phase of `bar` with the given parity.  False means the
// wait ran out (or another role gave up): the caller must stop its work.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                         int site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c, site);
}

// Bounded wait that ignores the abort flag (used while draining on exit).
static __device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                        unsigned long long limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

}  // namespace fa
