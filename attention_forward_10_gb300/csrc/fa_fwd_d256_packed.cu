// fa_fwd_d256_packed.cu -- instantiations and launcher of the head-dim-256 kernel (packed variable-length batches).
#include "fa_fwd_d256_kernel.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

template <bool CAUSAL, bool BF16>
cudaError_t launch_one(const FaParams& p, int grid, cudaStream_t stream) {
  constexpr int kSmem = d256::kSmemBytes;
  constexpr auto kernel = fa_fwd_d256_kernel<CAUSAL, BF16, true>;
  cudaError_t e = smem_attribute_once<kernel>(kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(grid), dim3(d256::kThreads), kSmem, stream, p);
}

}  // namespace

cudaError_t launch_fwd_d256_packed(const FaParams& p, bool causal, bool bf16, int grid,
                                   cudaStream_t stream) {
  if (causal) return bf16 ? launch_one<true, true>(p, grid, stream)
                          : launch_one<true, false>(p, grid, stream);
  return bf16 ? launch_one<false, true>(p, grid, stream)
              : launch_one<false, false>(p, grid, stream);
}

}  // namespace fa
