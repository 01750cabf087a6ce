// fa_bwd_d128_packed.cu -- instantiations and launcher of the backward kernels,
// head dim 128 (packed variable-length batches).
#include "fa_bwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

template <bool CAUSAL, bool BF16, bool TABLE = false>
cudaError_t launch_all(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                       const void* dout, const float* lse, float* lse2, float* dsum,
                       int grid_kv, int grid_q, int num_sms, cudaStream_t stream) {
  // pre-pass: D/16 threads per padded row, grid-stride over num_sms * 8 blocks
  const long long threads = static_cast<long long>(p_q.num_bh) * p_q.n_pad * (128 / 16);
  long long blocks = (threads + 255) / 256;
  if (blocks > static_cast<long long>(num_sms) * 8) blocks = static_cast<long long>(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  cudaError_t e = launch_pdl(bwd::fa_bwd_prepass_kernel<128, BF16, true>,
                             dim3(static_cast<int>(blocks)), dim3(256), 0, stream,
                             static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                             lse, lse2, dsum, p_q.num_bh, p_q.N, p_q.n_pad, p_q);
  if (e != cudaSuccess) return e;
  constexpr int kSmem = bwd::Layout<128>::kSmemBytes;
  constexpr auto kv = bwd::fa_bwd_dkdv_kernel<128, CAUSAL, BF16, true, TABLE>;
  constexpr auto dq = bwd::fa_bwd_dq_kernel<128, CAUSAL, BF16, true, TABLE>;
  e = smem_attribute_once<kv>(kSmem);
  if (e != cudaSuccess) return e;
  e = smem_attribute_once<dq>(kSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kv, dim3(grid_kv), dim3(bwd::kThreads), kSmem, stream, p_kv);
  if (e != cudaSuccess) return e;
  return launch_pdl(dq, dim3(grid_q), dim3(bwd::kThreads), kSmem, stream, p_q);
}

}  // namespace

cudaError_t launch_bwd_d128_packed(const BwdParams& p_kv, const BwdParams& p_q, const void* o,
                                   const void* dout, const float* lse, float* lse2, float* dsum,
                                   bool causal, bool bf16, int grid_kv, int grid_q, int num_sms,
                                   cudaStream_t stream) {
  if (causal && p_kv.unit_table)  // units from the per-CTA unit tables
    return bf16 ? launch_all<true, true, true>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv,
                                               grid_q, num_sms, stream)
                : launch_all<true, false, true>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv,
                                                grid_q, num_sms, stream);
  if (causal)
    return bf16 ? launch_all<true, true>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv, grid_q,
                                         num_sms, stream)
                : launch_all<true, false>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv, grid_q,
                                          num_sms, stream);
  return bf16 ? launch_all<false, true>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv, grid_q,
                                        num_sms, stream)
              : launch_all<false, false>(p_kv, p_q, o, dout, lse, lse2, dsum, grid_kv, grid_q,
                                         num_sms, stream);
}

}  // namespace fa
