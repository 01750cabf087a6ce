// fa_launch.h -- internal interface between the C-ABI layer (fa_api.cu) and
// the per-head-dim kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "fa_params.h"

namespace fa {

// Dynamic shared memory one CTA of the forward kernel needs for head dim d.
int fwd_smem_bytes(int d);

// Enqueue the forward kernel for head dim 64 / 128 with `grid` persistent CTAs.
cudaError_t launch_fwd_d64(const FaParams& p, bool causal, bool bf16, int grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(const FaParams& p, bool causal, bool bf16, int grid,
                            cudaStream_t stream);

// Enqueue the watchdog self-test kernel (one CTA).
cudaError_t launch_watchdog_selftest(int* status, unsigned long long timeout_ns,
                                     cudaStream_t stream);

}  // namespace fa
