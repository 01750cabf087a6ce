// fa_combine.cu -- merge of split-KV partial results.
//
// With the keys of a query row cut into splits, split s yields a partial
// output O_s (normalised by its own row sum) and its log-sum-exp L_s over the
// split's keys.  The full row is then
//     L = ln sum_s exp(L_s),      O = sum_s exp(L_s - L) O_s
// (the softmax over all keys is the L_s-weighted mixture of the per-split
// softmaxes) -- the same merge of log-normalisers the online softmax of
// LeetCUDA "flash_attn_mma_tiling_qk.cu" applies tile by tile, applied once
// across splits.  A split that holds none of the row's admissible keys is
// skipped (its partial was never written).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ float to_float(uint32_t half_bits) {
  if constexpr (BF16) {
    return __uint_as_float(half_bits << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(half_bits)));
  }
}

// One thread per 8 output elements (16 bytes) of a row; d/8 threads per row.
// The partials of up to four splits are loaded before any is accumulated, so
// that several 16-byte reads per thread are in flight.
template <bool BF16>
__global__ void __launch_bounds__(256)
    fa_splitkv_combine_kernel(const uint16_t* __restrict__ o_part,
                              const float* __restrict__ lse_part, uint16_t* __restrict__ o,
                              float* __restrict__ lse, CombineArgs a) {
  griddep_wait();  // (programmatic dependent launch: see fa_launch.h)
  griddep_launch_dependents();
  const int tpr = a.d / 8;
  const long long rows = static_cast<long long>(a.num_bh) * a.N;
  const long long total = rows * tpr;
  const long long part_stride = rows;  // rows per split
  for (long long gid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       gid < total; gid += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row_id = gid / tpr;  // bh * N + i
    const int part = static_cast<int>(gid % tpr);
    const int i = static_cast<int>(row_id % a.N);
    // keys query i may see: [lo, hi); split s holds [s*split_keys, +split_keys)
    const long long lo = static_cast<long long>(i) - a.win_left;
    const long long hi = static_cast<long long>(i) + a.win_right + 1;
    const int s_first = static_cast<int>((lo > 0 ? lo : 0) / a.split_keys);
    const long long last_key = (hi < a.N ? hi : a.N) - 1;
    const int s_last = static_cast<int>(last_key / a.split_keys);  // splits [s_first, s_last]
    float m = -INFINITY;
    for (int s = s_first; s <= s_last; ++s) m = fmaxf(m, lse_part[s * part_stride + row_id]);
    uint32_t packed[4] = {0, 0, 0, 0};
    float row_lse = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = s_first; s <= s_last; ++s) sum += expf(lse_part[s * part_stride + row_id] - m);
      row_lse = m + logf(sum);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const uint16_t* src = o_part + row_id * a.d + part * 8;
      const long long split_elems = part_stride * a.d;
      for (int s0 = s_first; s0 <= s_last; s0 += 4) {
        uint4 v[4];
        float wgt[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int s = s0 + k;
          if (s <= s_last) {
            v[k] = *reinterpret_cast<const uint4*>(src + s * split_elems);
            wgt[k] = expf(lse_part[s * part_stride + row_id] - row_lse);
          } else {
            v[k] = make_uint4(0, 0, 0, 0);
            wgt[k] = 0.f;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t words[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] += wgt[k] * to_float<BF16>(words[e] & 0xffffu);
            acc[2 * e + 1] += wgt[k] * to_float<BF16>(words[e] >> 16);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) packed[e] = pack2<BF16>(acc[2 * e], acc[2 * e + 1]);
    }
    *reinterpret_cast<uint4*>(o + row_id * a.d + part * 8) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (part == 0 && lse != nullptr) lse[row_id] = row_lse;
  }
}

}  // namespace

cudaError_t launch_splitkv_combine(const void* o_part, const float* lse_part, void* o,
                                   float* lse, const CombineArgs& a, bool bf16, int num_sms,
                                   cudaStream_t stream) {
  const long long threads = static_cast<long long>(a.num_bh) * a.N * (a.d / 8);
  long long blocks = (threads + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const auto* op = static_cast<const uint16_t*>(o_part);
  auto* out = static_cast<uint16_t*>(o);
  const dim3 g(static_cast<int>(blocks)), b(256);
  return bf16 ? launch_pdl(fa_splitkv_combine_kernel<true>, g, b, 0, stream, op, lse_part, out,
                           lse, a)
              : launch_pdl(fa_splitkv_combine_kernel<false>, g, b, 0, stream, op, lse_part,
                           out, lse, a);
}

}  // namespace fa
