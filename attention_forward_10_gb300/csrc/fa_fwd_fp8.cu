// fa_fwd_fp8.cu -- the FP8 (E4M3) forward: V transpose and the d=128 kernel
// instantiations.
//
// The P V product takes V as its B operand with the keys (its K dimension)
// contiguous, so the launcher first writes V^T, [heads][d][n_pad] bytes with
// zero keys past N, into the caller's workspace; the forward kernel then
// reads K-major tiles of Q, K and V^T (one byte per element, 128-byte rows).
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

// vt[h][c][n] = v[h][n][c] for n < N, 0 for N <= n < n_pad.  Two 64-key x
// 64-column byte tiles per iteration (256 threads, 16 bytes each way per
// tile; both tiles' loads are issued before the first barrier, so that each
// block keeps 8 KB in flight).
__global__ void __launch_bounds__(256)
    fa_transpose_v_e4m3_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                               int num_heads, int N, int n_pad, int d) {
  griddep_wait();  // (programmatic dependent launch: see fa_launch.h)
  griddep_launch_dependents();
  __shared__ uint8_t tile[2][64][64 + 16];
  const int t = threadIdx.x;
  const int kt = n_pad / 64, ct = d / 64;
  const long long tiles = static_cast<long long>(num_heads) * kt * ct;
  const long long stride = 2ll * gridDim.x;
  for (long long x0 = blockIdx.x; x0 < tiles; x0 += stride) {
    int h[2], n0[2], c0[2];
    bool live[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const long long x = x0 + k * static_cast<long long>(gridDim.x);
      live[k] = x < tiles;
      const long long xx = live[k] ? x : x0;
      h[k] = static_cast<int>(xx / (kt * ct));
      const int rem = static_cast<int>(xx % (kt * ct));
      n0[k] = (rem / ct) * 64;
      c0[k] = (rem % ct) * 64;
    }
    {
      const int r = t / 4, q = t % 4;  // key row r, 16-byte column chunk q
      uint4 val[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        val[k] = make_uint4(0, 0, 0, 0);
        if (live[k] && n0[k] + r < N)
          val[k] = *reinterpret_cast<const uint4*>(
              v + (static_cast<long long>(h[k]) * N + n0[k] + r) * d + c0[k] + q * 16);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) *reinterpret_cast<uint4*>(&tile[k][r][q * 16]) = val[k];
    }
    __syncthreads();
    {
      const int c = t / 4, q = t % 4;  // output row c (a column of V), keys q*16..
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!live[k]) continue;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = static_cast<uint32_t>(tile[k][q * 16 + 4 * e][c]) |
                 (static_cast<uint32_t>(tile[k][q * 16 + 4 * e + 1][c]) << 8) |
                 (static_cast<uint32_t>(tile[k][q * 16 + 4 * e + 2][c]) << 16) |
                 (static_cast<uint32_t>(tile[k][q * 16 + 4 * e + 3][c]) << 24);
        *reinterpret_cast<uint4*>(vt + (static_cast<long long>(h[k]) * d + c0[k] + c) * n_pad +
                                  n0[k] + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    __syncthreads();
  }
}

template <bool CAUSAL>
cudaError_t launch_one(const FaParams& p, int grid, cudaStream_t stream) {
  constexpr int kSmem = Layout<128, true>::kSmemBytes;
  constexpr auto kernel = fa_fwd_kernel<128, CAUSAL, true, false, true>;
  cudaError_t e = smem_attribute_once<kernel>(kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(grid), dim3(kNumThreads), kSmem, stream, p);
}

}  // namespace

cudaError_t launch_transpose_v_e4m3(const void* v, void* vt, int num_heads, int N, int n_pad,
                                    int d, int num_sms, cudaStream_t stream) {
  const long long tiles = static_cast<long long>(num_heads) * (n_pad / 64) * (d / 64);
  const long long pairs = (tiles + 1) / 2;  // two tiles per block iteration
  long long blocks = pairs < static_cast<long long>(num_sms) * 8 ? pairs
                                                               : static_cast<long long>(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  return launch_pdl(fa_transpose_v_e4m3_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0,
                    stream, static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt),
                    num_heads, N, n_pad, d);
}

cudaError_t launch_fwd_d128_fp8(const FaParams& p, bool causal, int grid, cudaStream_t stream) {
  return causal ? launch_one<true>(p, grid, stream) : launch_one<false>(p, grid, stream);
}

}  // namespace fa
