// fa_launch.h -- internal interface between the C-ABI layer (fa_api.cu) and
// the per-head-dim kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <utility>

#include "fa_params.h"

namespace fa {

unsigned long long current_context_id();

// Raise the dynamic shared-memory limit of `Kernel` to `bytes`, once per
// device and context (the attribute belongs to the function in one context;
// setting it before every launch would cost a driver call each time).
template <auto Kernel>
cudaError_t smem_attribute_once(int bytes) {
  constexpr int kDevices = 64;
  static std::atomic<unsigned long long> done[kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = current_context_id();
  const bool cacheable = ctx != 0 && dev >= 0 && dev < kDevices;
  if (cacheable && done[dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cacheable) done[dev].store(ctx, std::memory_order_release);
  return e;
}

// Launch `kernel` on `stream` with programmatic stream serialisation: the
// grid may start launching while the stream's previous kernel finishes (its
// CTAs wait in griddep_wait before touching global memory), so that the
// set-up of back-to-back launches overlaps the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


// Enqueue the forward kernel for head dim 64 / 128 with `grid` persistent CTAs
// (two 128-row query tiles per work unit, 128-key K/V tiles).
cudaError_t launch_fwd_d64(const FaParams& p, bool causal, bool bf16, int grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(const FaParams& p, bool causal, bool bf16, int grid,
                            cudaStream_t stream);
// Head dim 256: one 128-row query tile per work unit, 64-key K/V tiles.
cudaError_t launch_fwd_d256(const FaParams& p, bool causal, bool bf16, int grid,
                            cudaStream_t stream);
// The same for packed variable-length batches (p.cu_seqlens set); the
// launchers above forward to these.
cudaError_t launch_fwd_d64_packed(const FaParams& p, bool causal, bool bf16, int grid,
                                  cudaStream_t stream);
cudaError_t launch_fwd_d128_packed(const FaParams& p, bool causal, bool bf16, int grid,
                                   cudaStream_t stream);
cudaError_t launch_fwd_d256_packed(const FaParams& p, bool causal, bool bf16, int grid,
                                   cudaStream_t stream);

// Backward: the pre-pass (LSE * log2 e and rowsum(dO * O) into the padded
// workspace), then the dK/dV and dQ kernels, all on `stream`.
// p_kv / p_q: the parameters of the dK/dV and dQ kernels (their unit counts
// differ); grid_kv / grid_q their persistent grids.
cudaError_t launch_bwd_d64(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                           const void* dout, const float* lse, float* lse2, float* dsum,
                           bool causal, bool bf16, int grid_kv, int grid_q, int num_sms,
                           cudaStream_t stream);
cudaError_t launch_bwd_d128(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                            const void* dout, const float* lse, float* lse2, float* dsum,
                            bool causal, bool bf16, int grid_kv, int grid_q, int num_sms,
                            cudaStream_t stream);
// The same for packed variable-length batches (p.cu_seqlens set); the two
// launchers above forward to these.
cudaError_t launch_bwd_d64_packed(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                                  const void* dout, const float* lse, float* lse2, float* dsum,
                                  bool causal, bool bf16, int grid_kv, int grid_q, int num_sms,
                                  cudaStream_t stream);
cudaError_t launch_bwd_d128_packed(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                                   const void* dout, const float* lse, float* lse2,
                                   float* dsum, bool causal, bool bf16, int grid_kv, int grid_q,
                                   int num_sms, cudaStream_t stream);

// FP8 forward: V^T ([heads][d][n_pad] bytes, zero past N) from V
// ([heads][N][d] bytes), then the d=128 E4M3 kernel (p.tm_v maps V^T).
cudaError_t launch_transpose_v_e4m3(const void* v, void* vt, int num_heads, int N, int n_pad,
                                    int d, int num_sms, cudaStream_t stream);
cudaError_t launch_fwd_d128_fp8(const FaParams& p, bool causal, int grid, cudaStream_t stream);

// Shape of a split-KV merge: num_bh heads of N rows of d columns; split s
// holds keys [s * split_keys, (s + 1) * split_keys); query i may see keys
// i - win_left .. i + win_right (both already clamped to [0, N]).
struct CombineArgs {
  int num_bh, N, d;
  int num_splits, split_keys;
  int win_left, win_right;
};

// Enqueue the merge of split-KV partials (o_part [S][num_bh][N][d] 16-bit,
// lse_part [S][num_bh][N] fp32) into o and lse (lse may be null).
cudaError_t launch_splitkv_combine(const void* o_part, const float* lse_part, void* o,
                                   float* lse, const CombineArgs& a, bool bf16, int num_sms,
                                   cudaStream_t stream);

// Unique id of the calling thread's current CUDA context (cuCtxGetId), 0 if
// there is none or it cannot be read.  Ids are never reused within a process.
unsigned long long current_context_id();

// Device address of the fixed split-KV scratch of the current device `dev`
// (FA_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned), looked up on the first
// call per device and context; nullptr with the CUDA error in *rc if that
// fails (the runtime's last error is cleared).
void* noalloc_scratch(int dev, cudaError_t* rc);

// Enqueue the watchdog self-test kernel (one CTA).
cudaError_t launch_watchdog_selftest(int* status, unsigned long long timeout_ns,
                                     cudaStream_t stream);

}  // namespace fa
