// fa_common.cuh -- pieces shared by the attention kernels: bounded mbarrier
// waits with a CTA-wide abort flag, and the coalesced row store of an
// epilogue.
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

// Store of 32 columns (16 packed words w) of the rows of one warp,
// one row per lane: a 4x4 transpose of 16-byte chunks within each group of
// four lanes (two shfl_xor stages) leaves lane 4g + i with chunk i of the
// rows of lanes 4g .. 4g + 3, so that each of the four stores writes 8 rows'
// 64 contiguous bytes (whole 32-byte sectors) instead of 32 rows' 16 bytes.
// row_ptr(r): where lane r's 32 columns go (nullptr: that row is not stored).
template <typename RowPtr>
__device__ __forceinline__ void store_rows_x32(uint32_t (&w)[16], int lane, RowPtr row_ptr) {
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j & m) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // the low lane of the pair keeps chunk j and sends chunk j|m, the
        // high lane keeps j|m and sends j
        const uint32_t send = hi ? w[4 * j + e] : w[4 * (j | m) + e];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        if (hi)
          w[4 * j + e] = recv;
        else
          w[4 * (j | m) + e] = recv;
      }
    }
  }
  const int g = lane >> 2, i = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint16_t* dst = row_ptr(4 * g + k);
    if (dst != nullptr)
      *reinterpret_cast<uint4*>(dst + 8 * i) =
          make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}

}  // namespace fa
