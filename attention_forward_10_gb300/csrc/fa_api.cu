// fa_api.cu -- the C ABI of libfa_gb300.so: argument validation, TMA tensor
// maps, persistent-grid sizing and the launch.  Declarations and the full
// contract are in include/fa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

// Device status word: the kernels' bounded waits record a timeout here.
__device__ int g_status_word;

// One CTA waits on a barrier nobody arrives on; the bounded wait must give
// up, record the timeout and return.
__global__ void fa_watchdog_selftest_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_storage;
  const uint32_t b = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_storage = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Ctl ctl{reinterpret_cast<volatile int*>(&abort_storage), status, timeout_ns};
    wait_bar(b, 0, ctl, kSiteSelftest);
  }
  __syncthreads();
}

cudaError_t launch_watchdog_selftest(int* status, unsigned long long timeout_ns,
                                     cudaStream_t stream) {
  fa_watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

namespace {

constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_max_ctas{0};

struct DeviceInfo {
  std::once_flag once;
  int ok = 0;           // 1: usable sm_103 device
  int num_sms = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

// Per-device set-up with that device current: capability check, SM count and
// the device address of the status word.
DeviceInfo* device_info(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& info = g_dev[dev];
  std::call_once(info.once, [&] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return;
    info.num_sms = sms;
    info.status = static_cast<int*>(addr);
    info.ok = (major == 10 && minor == 3) ? 1 : 0;
  });
  return &info;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 4-D view of a contiguous [BH][N][d] 16-bit tensor for 128-byte-swizzled
// tiles: dim0 = 64 elements (128 B, innermost), dim1 = N rows (stride d*2 B),
// dim2 = d/64 column blocks (stride 128 B), dim3 = BH heads (stride N*d*2 B).
// A box {64, rows, blocks, 1} lands in shared memory as [blocks][rows][64],
// the K-major layout the MMA descriptors expect; rows past N read as zero and
// are not written by stores.
bool encode_qkvo_map(CUtensorMap* map, const void* base, int N, int d, int bh, bool bf16,
                     int box_rows, int box_blocks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(d / 64),
                        static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, 128,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(box_blocks), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
}

}  // namespace
}  // namespace fa

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_set_wait_timeout_us(long long timeout_us) {
  if (timeout_us < 1) return FA_ERR_INVALID_ARG;
  fa::g_timeout_ns.store(static_cast<unsigned long long>(timeout_us) * 1000ull);
  return FA_OK;
}

int fa_set_max_ctas(int max_ctas) {
  if (max_ctas < 0) return FA_ERR_INVALID_ARG;
  fa::g_max_ctas.store(max_ctas);
  return FA_OK;
}

int fa_num_sms(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  fa::DeviceInfo* info = fa::device_info(dev);
  return (info != nullptr && info->num_sms > 0) ? info->num_sms : -1;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, float scale, int causal, int dtype, void* stream) {
  return fa_fwd_ext(q, k, v, o, lse, B, H, H, N, d, scale, causal, -1, -1, dtype, stream);
}

int fa_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse, int B,
               int H, int H_kv, int N, int d, float scale, int causal, int window_left,
               int window_right, int dtype, void* stream) {
  using namespace fa;
  if (B < 0 || H < 0 || N < 0 || H_kv < 0) return FA_ERR_INVALID_ARG;
  if (H > 0 && (H_kv == 0 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return FA_ERR_MISALIGNED;
  if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(B) * H;
  // work units per (b,h): pairs of 128-row query tiles (d <= 128) or single
  // 128-row tiles (d = 256)
  const int rows_per_unit = (d == 256) ? kBlockM : kRowsPerUnit;
  const long long pairs = (static_cast<long long>(N) + rows_per_unit - 1) / rows_per_unit;
  // (headroom: the last-wave split below may add up to one wave of units)
  if (bh >= (1ll << 31) || bh * pairs + 4096 >= (1ll << 31)) return FA_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo* info = device_info(dev);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  if (!info->ok) return FA_ERR_UNSUPPORTED;

  const bool bf16 = dtype == FA_DTYPE_BF16;
  FaParams p;
  const int ibh = static_cast<int>(bh);
  const int ibh_kv = static_cast<int>(static_cast<long long>(B) * H_kv);
  // d = 256 streams 64-key K/V tiles and stores O in two 128-column halves
  const int kv_rows = (d == 256) ? 64 : kBlockN;
  const int o_blocks = (d == 256) ? 2 : d / 64;
  if (!encode_qkvo_map(&p.tm_q, q, N, d, ibh, bf16, kBlockM, d / 64) ||
      !encode_qkvo_map(&p.tm_k, k, N, d, ibh_kv, bf16, kv_rows, d / 64) ||
      !encode_qkvo_map(&p.tm_v, v, N, d, ibh_kv, bf16, kv_rows, d / 64) ||
      !encode_qkvo_map(&p.tm_o, o, N, d, ibh, bf16, kBlockM, o_blocks))
    return FA_ERR_CUDA;
  p.lse = lse;
  p.status = info->status;
  p.timeout_ns = g_timeout_ns.load();
  p.N = N;
  p.num_bh = static_cast<int>(bh);
  p.num_pairs = static_cast<int>(pairs);
  p.num_units = static_cast<int>(bh * pairs);
  p.n_ktiles = (N + kv_rows - 1) / kv_rows;
  p.H = H;
  p.group = H / H_kv;
  // window bounds: negative or beyond N means unbounded (= N); causal caps
  // the right bound at 0
  p.win_left = (window_left < 0 || window_left > N) ? N : window_left;
  p.win_right = (window_right < 0 || window_right > N) ? N : window_right;
  if (causal) p.win_right = 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);

  int grid = info->num_sms;
  const int cap = g_max_ctas.load();
  if (cap > 0 && cap < grid) grid = cap;
  p.num_pair_units = p.num_units;
  if (d != 256) {
    // Balance the last wave: its L pair units become 2L single-tile units
    // when those fit in one wave.
    const long long pair_units = bh * pairs;
    const long long partial = pair_units % grid;
    if (pair_units > grid && partial > 0 && 2 * partial <= grid) {
      p.num_pair_units = static_cast<int>(pair_units - partial);
      p.num_units = static_cast<int>(pair_units + partial);
    }
  }
  if (p.num_units < grid) grid = p.num_units;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = (d == 64)    ? launch_fwd_d64(p, causal != 0, bf16, grid, s)
                  : (d == 128) ? launch_fwd_d128(p, causal != 0, bf16, grid, s)
                               : launch_fwd_d256(p, causal != 0, bf16, grid, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_get_device_status(void* stream, int* site) {
  using namespace fa;
  if (site != nullptr) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo* info = device_info(dev);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, info->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word == 0) return FA_OK;
  const int zero = 0;
  if (cudaMemcpy(info->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_CUDA;
  if (site != nullptr) *site = word >> 8;
  return word & 0xff;
}

int fa_selftest_watchdog(long long timeout_us, void* stream) {
  using namespace fa;
  if (timeout_us < 1) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DeviceInfo* info = device_info(dev);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  if (!info->ok) return FA_ERR_UNSUPPORTED;
  cudaError_t e = launch_watchdog_selftest(
      info->status, static_cast<unsigned long long>(timeout_us) * 1000ull,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
