// fa_fwd_d128_packed.cu -- instantiations and launcher of the forward kernel, head dim 128 (packed variable-length batches).
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

template <bool CAUSAL, bool BF16, bool TABLE = false>
cudaError_t launch_one(const FaParams& p, int grid, cudaStream_t stream) {
  constexpr int kSmem = Layout<128>::kSmemBytes;
  constexpr auto kernel = fa_fwd_kernel<128, CAUSAL, BF16, true, false, TABLE>;
  cudaError_t e = smem_attribute_once<kernel>(kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(grid), dim3(kNumThreads), kSmem, stream, p);
}

}  // namespace

cudaError_t launch_fwd_d128_packed(const FaParams& p, bool causal, bool bf16, int grid,
                                   cudaStream_t stream) {
  if (causal && p.unit_table)  // units from the per-CTA unit table
    return bf16 ? launch_one<true, true, true>(p, grid, stream)
                : launch_one<true, false, true>(p, grid, stream);
  if (causal) return bf16 ? launch_one<true, true>(p, grid, stream)
                          : launch_one<true, false>(p, grid, stream);
  return bf16 ? launch_one<false, true>(p, grid, stream)
              : launch_one<false, false>(p, grid, stream);
}

}  // namespace fa
