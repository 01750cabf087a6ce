// fa_api.cu -- the C ABI of libfa_gb300.so: argument validation, TMA tensor
// maps, persistent-grid sizing and the launch.  Declarations and the full
// contract are in include/fa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
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
PFN_cuCtxGetCurrent_v4000 ctx_current_fn();
PFN_cuCtxGetId_v12000 ctx_id_fn();
}  // namespace

unsigned long long current_context_id() {
  auto get = ctx_current_fn();
  auto get_id = ctx_id_fn();
  if (get == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_max_ctas{0};
std::atomic<int> g_gqa_pack{1};

struct DeviceInfo {
  std::once_flag once;
  int ok = 0;           // 1: usable sm_103 device
  int num_sms = 0;
  int* status = nullptr;  // status word of the context `status_ctx`
  unsigned long long status_ctx = 0;
  std::mutex mu;
};
DeviceInfo g_dev[kMaxDevices];

// Per-device set-up with that device current: capability check, SM count and
// the device address of the status word.  The address belongs to the
// device's current context: it is looked up again whenever the calling
// thread's context differs from the one it was taken in (after
// cudaDeviceReset, or under another driver context), so no kernel is handed
// the address of a destroyed context.
// What a call needs of its device, copied under the device's lock.
struct DevState {
  int ok = 0;
  int num_sms = 0;
  int* status = nullptr;
};

DevState* device_info(int dev, DevState* out) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& info = g_dev[dev];
  std::call_once(info.once, [&] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return;
    info.num_sms = sms;
    info.ok = (major == 10 && minor == 3) ? 1 : 0;
  });
  std::lock_guard<std::mutex> lock(info.mu);
  const unsigned long long ctx = current_context_id();
  if (info.status == nullptr || ctx == 0 || ctx != info.status_ctx) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
      cudaGetLastError();  // leave no stale error for the caller's next check
      info.status = nullptr;
      info.status_ctx = 0;
    } else {
      info.status = static_cast<int*>(addr);
      // (read after the look-up, which makes the primary context current)
      info.status_ctx = current_context_id();
    }
  }
  out->ok = info.ok;
  out->num_sms = info.num_sms;
  out->status = info.status;
  return out;
}

PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  }();
  return fn;
}

PFN_cuCtxGetId_v12000 ctx_id_fn() {
  static PFN_cuCtxGetId_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  }();
  return fn;
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

// 4-D view of a packed [rows][heads][d] 16-bit tensor (variable-length
// batches): dim0 = 64 elements, dim1 = rows (stride heads*d*2 B), dim2 = d/64
// column blocks (stride 128 B), dim3 = heads (stride d*2 B).  The same box
// {64, rows, blocks, 1} lands in shared memory in the same [blocks][rows][64]
// order as the [B][H][N][d] view above.
bool encode_packed_map(CUtensorMap* map, const void* base, int rows, int heads, int d,
                       bool bf16, int box_rows, int box_blocks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(d / 64),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2,
                           128, static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(box_blocks), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D view of a packed [rows][H][d] 16-bit tensor whose query heads come in
// groups of `g` (grouped-query packing): dim0 = 64 elements, dim1 = the g
// heads of a group (stride d*2 B), dim2 = rows (stride H*d*2 B), dim3 = d/64
// column blocks (stride 128 B), dim4 = groups (stride g*d*2 B).  The box {64,
// g, 128/g, d/64, 1} lands in shared memory as [d/64][128/g rows][g][64]:
// the [blocks][tile rows][64] order of the 4-D views, tile row = row * g +
// head.
bool encode_packed_gqa_map(CUtensorMap* map, const void* base, int rows, int H, int g, int d,
                           bool bf16) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t hd = static_cast<cuuint64_t>(d) * 2;
  cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(d / 64), static_cast<cuuint64_t>(H / g)};
  cuuint64_t strides[4] = {hd, static_cast<cuuint64_t>(H) * hd, 128,
                           static_cast<cuuint64_t>(g) * hd};
  cuuint32_t box[5] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(kBlockM / g),
                       static_cast<cuuint32_t>(d / 64), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  5, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D byte view for the FP8 kernel's 128-byte-row tiles: dim0 = 128 bytes
// (innermost), dim1 = rows (stride row_stride), dim2 = 128-byte blocks
// (stride 128), dim3 = heads (stride head_stride); box {128, box_rows, 1, 1}.
bool encode_e4m3_map(CUtensorMap* map, const void* base, int rows, int row_bytes,
                     unsigned long long row_stride, unsigned long long head_stride, int heads,
                     int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(row_bytes / 128), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {row_stride, 128, head_stride};
  cuuint32_t box[4] = {128, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
    case FA_ERR_SCRATCH_LIMIT: return "FA_ERR_SCRATCH_LIMIT";
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

int fa_set_gqa_pack(int enable) {
  if (enable != 0 && enable != 1) return FA_ERR_INVALID_ARG;
  fa::g_gqa_pack.store(enable);
  return FA_OK;
}

int fa_num_sms(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  fa::DevState dev_state;
  fa::DevState* info = fa::device_info(dev, &dev_state);
  return (info != nullptr && info->num_sms > 0) ? info->num_sms : -1;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, float scale, int causal, int dtype, void* stream) {
  return fa_fwd_ext(q, k, v, o, lse, B, H, H, N, d, scale, causal, -1, -1, dtype, stream);
}

}  // extern "C"

namespace fa {
namespace {

// Everything fa_fwd_ext and fa_fwd_splitkv share: validation, tensor maps,
// grid sizing, launch.  With num_splits > 1 the outputs are the split
// partials: o_out / lse_out hold num_splits * B * H heads.
struct ForwardCall {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, H_kv, N, d;
  float scale;
  int causal, window_left, window_right, dtype;
  void* stream;
  // variable-length batches: B sequences packed along the rows, N = the
  // longest query sequence; nullptr / 0 for the [B][H][N][d] layout.  Keys
  // have their own offsets, total and longest length (the query ones for
  // self-attention) and both sides optional used lengths.
  const int* cu_seqlens = nullptr;
  int total = 0;
  const int* cu_seqlens_k = nullptr;
  int total_k = 0;
  int N_k = 0;
  const int* seqused_q = nullptr;
  const int* seqused_k = nullptr;
  // FP8 (E4M3) inputs: descale factors and the V^T workspace
  bool fp8 = false;
  float descale_q = 1.f, descale_k = 1.f, descale_v = 1.f;
  void* vt = nullptr;
  int n_pad = 0;
};

int validate(const ForwardCall& c) {
  if (c.B < 0 || c.H < 0 || c.N < 0 || c.H_kv < 0) return FA_ERR_INVALID_ARG;
  if (c.H > 0 && (c.H_kv == 0 || c.H % c.H_kv != 0)) return FA_ERR_INVALID_ARG;
  if (c.dtype != FA_DTYPE_F16 && c.dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (c.causal != 0 && c.causal != 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(c.scale) && c.scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (c.d != 64 && c.d != 128 && c.d != 256) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

bool empty_problem(const ForwardCall& c) { return c.B == 0 || c.H == 0 || c.N == 0; }

int check_pointers(const ForwardCall& c) {
  if (c.q == nullptr || c.k == nullptr || c.v == nullptr || c.o == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(c.q, 16) || !aligned(c.k, 16) || !aligned(c.v, 16) || !aligned(c.o, 16))
    return FA_ERR_MISALIGNED;
  if (c.lse != nullptr && !aligned(c.lse, 4)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

// K/V tile length of the kernel that serves head dim d.
int kv_tile_rows(int d) { return d == 256 ? 64 : kBlockN; }

// Work units per (b,h): pairs of 128-row query tiles (d <= 128) or single
// 128-row tiles (d = 256).
long long units_per_head(int N, int d) {
  const int rows = (d == 256) ? kBlockM : kRowsPerUnit;
  return (static_cast<long long>(N) + rows - 1) / rows;
}

// log2 of the query heads packed per tile row group for this call (0: no
// grouped-query packing).  Packed batches with d <= 128 whose query heads
// share K/V heads in groups of 2..16 (a power of two) pack a group's heads
// into each tile, so a group streams its K/V once and short query
// sequences (decoding) still fill the 128 tile rows.
int gqa_pack_log2(const ForwardCall& c) {
  if (c.cu_seqlens == nullptr || c.fp8 || c.d > 128 || g_gqa_pack.load() == 0) return 0;
  const int g = c.H / c.H_kv;
  if (g < 2 || g > 16 || (g & (g - 1)) != 0) return 0;
  int lg = 0;
  while ((1 << lg) < g) ++lg;
  return lg;
}

int launch_forward(const ForwardCall& c, void* o_out, float* lse_out, int num_splits,
                   int split_tiles) {
  using namespace fa;
  const int gqa_log2 = gqa_pack_log2(c);
  // (grouped-query packing: problems are (sequence, K/V head) pairs whose
  // rows are positions x heads of the group)
  const long long bh = static_cast<long long>(c.B) * (c.H >> gqa_log2);
  const long long pairs = units_per_head(static_cast<int>(std::min<long long>(
                                             static_cast<long long>(c.N) << gqa_log2,
                                             (1ll << 31) - 1)),
                                         c.d);
  // (headroom: the last-wave split below may add up to one wave of units)
  if (bh >= (1ll << 31) || bh * pairs * num_splits + 4096 >= (1ll << 31))
    return FA_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DevState dev_state;
  DevState* info = device_info(dev, &dev_state);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  if (!info->ok) return FA_ERR_UNSUPPORTED;

  const int N = c.N, d = c.d;
  const bool bf16 = c.dtype == FA_DTYPE_BF16;
  FaParams p;
  const int ibh = static_cast<int>(bh);
  const int ibh_kv = static_cast<int>(static_cast<long long>(c.B) * c.H_kv);
  // d = 256 streams 64-key K/V tiles and stores O in two 128-column halves
  const int kv_rows = kv_tile_rows(d);
  const int o_blocks = (d == 256) ? 2 : d / 64;
  const bool packed = c.cu_seqlens != nullptr;
  if (c.fp8) {
    // Q, K: [heads][N][128] bytes; V^T: [H_kv heads][128][n_pad] bytes; O bf16
    const unsigned long long nd = static_cast<unsigned long long>(N) * d;
    if (!encode_e4m3_map(&p.tm_q, c.q, N, d, d, nd, ibh, kBlockM) ||
        !encode_e4m3_map(&p.tm_k, c.k, N, d, d, nd, ibh_kv, kBlockN) ||
        !encode_e4m3_map(&p.tm_v, c.vt, d, c.n_pad, c.n_pad,
                         static_cast<unsigned long long>(d) * c.n_pad, ibh_kv, d) ||
        !encode_qkvo_map(&p.tm_o, o_out, N, d, ibh, true, kBlockM, o_blocks))
      return FA_ERR_CUDA;
  } else if (packed) {
    // no key rows at all: every query row is fully masked, and the K/V maps
    // (read, then masked out) view the query buffer instead
    const bool no_keys = c.total_k == 0;
    const void* kb = no_keys ? c.q : c.k;
    const void* vb = no_keys ? c.q : c.v;
    const int k_rows = no_keys ? c.total : c.total_k;
    const bool q_ok =
        gqa_log2 ? encode_packed_gqa_map(&p.tm_q, c.q, c.total, c.H, 1 << gqa_log2, d, bf16) &&
                       encode_packed_gqa_map(&p.tm_o, o_out, c.total, c.H, 1 << gqa_log2, d,
                                             bf16)
                 : encode_packed_map(&p.tm_q, c.q, c.total, c.H, d, bf16, kBlockM, d / 64) &&
                       encode_packed_map(&p.tm_o, o_out, c.total, c.H, d, bf16, kBlockM,
                                         o_blocks);
    if (!q_ok ||
        !encode_packed_map(&p.tm_k, kb, k_rows, c.H_kv, d, bf16, kv_rows, d / 64) ||
        !encode_packed_map(&p.tm_v, vb, k_rows, c.H_kv, d, bf16, kv_rows, d / 64))
      return FA_ERR_CUDA;
  } else if (!encode_qkvo_map(&p.tm_q, c.q, N, d, ibh, bf16, kBlockM, d / 64) ||
             !encode_qkvo_map(&p.tm_k, c.k, N, d, ibh_kv, bf16, kv_rows, d / 64) ||
             !encode_qkvo_map(&p.tm_v, c.v, N, d, ibh_kv, bf16, kv_rows, d / 64) ||
             !encode_qkvo_map(&p.tm_o, o_out, N, d, ibh * num_splits, bf16, kBlockM, o_blocks)) {
    return FA_ERR_CUDA;
  }
  p.cu_seqlens = c.cu_seqlens;
  p.cu_seqlens_k = packed ? (c.cu_seqlens_k != nullptr ? c.cu_seqlens_k : c.cu_seqlens) : nullptr;
  p.seqused_q = packed ? c.seqused_q : nullptr;
  p.seqused_k = packed ? c.seqused_k : nullptr;
  p.total_rows = packed ? c.total : 0;
  p.total_rows_k = packed ? (c.cu_seqlens_k != nullptr ? c.total_k : c.total) : 0;
  const int N_k = (packed && c.cu_seqlens_k != nullptr) ? c.N_k : N;
  p.N_k = N_k;
  p.gqa_log2 = gqa_log2;
  // (one pair per problem: the table's order is the plain one, and building
  // it would only delay the start)
  p.unit_table = (packed && c.causal && d != 256 && num_splits == 1 && c.B <= kTableSeqs &&
                  pairs > 1 && pairs <= kTablePairs)
                     ? 1
                     : 0;
  p.o_ptr = static_cast<uint16_t*>(o_out);
  p.lse = lse_out;
  p.status = info->status;
  p.timeout_ns = g_timeout_ns.load();
  p.N = N;
  p.num_bh = ibh;
  p.num_pairs = static_cast<int>(pairs);
  p.num_units = static_cast<int>(bh * pairs * num_splits);
  p.n_ktiles = (N + kv_rows - 1) / kv_rows;
  p.H = c.H;
  p.group = c.H / c.H_kv;
  // window bounds: negative or beyond N + N_k means unbounded (= N + N_k,
  // wider than any query's distance to any key); causal caps the right
  // bound at 0
  const int unbounded = N + N_k;
  p.win_left = (c.window_left < 0 || c.window_left > unbounded) ? unbounded : c.window_left;
  p.win_right = (c.window_right < 0 || c.window_right > unbounded) ? unbounded : c.window_right;
  if (c.causal) p.win_right = 0;
  p.num_splits = num_splits;
  p.split_tiles = split_tiles;
  p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634);
  p.descale_v = 1.f;
  if (c.fp8) {
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * c.descale_q * c.descale_k *
                                      1.4426950408889634);
    p.descale_v = c.descale_v;
  }

  int grid = info->num_sms;
  const int cap = g_max_ctas.load();
  if (cap > 0 && cap < grid) grid = cap;
  p.num_pair_units = p.num_units;
  if (d != 256 && num_splits == 1 && !packed) {
    // Balance the last wave: its L pair units become 2L single-tile units
    // when those fit in one wave.  With fewer pair units than CTAs, as many
    // pairs as there are idle CTAs become two single-tile units each (a
    // small launch then ends sooner; packed launches, whose decode units
    // are bound by HBM, measured no faster).
    const long long pair_units = bh * pairs;
    long long split = 0;
    if (pair_units > grid) {
      const long long partial = pair_units % grid;
      if (partial > 0 && 2 * partial <= grid) split = partial;
    } else {
      split = std::min(pair_units, grid - pair_units);
    }
    if (split > 0) {
      p.num_pair_units = static_cast<int>(pair_units - split);
      p.num_units = static_cast<int>(pair_units + split);
    }
  }
  if (p.num_units < grid) grid = p.num_units;

  cudaStream_t s = static_cast<cudaStream_t>(c.stream);
  if (c.fp8) {
    cudaError_t e = launch_transpose_v_e4m3(c.v, c.vt, ibh_kv, N, c.n_pad, d, info->num_sms, s);
    if (e == cudaSuccess) e = launch_fwd_d128_fp8(p, c.causal != 0, grid, s);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  cudaError_t e = (d == 64)    ? launch_fwd_d64(p, c.causal != 0, bf16, grid, s)
                  : (d == 128) ? launch_fwd_d128(p, c.causal != 0, bf16, grid, s)
                               : launch_fwd_d256(p, c.causal != 0, bf16, grid, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Longest CTA of a persistent launch with `splits` key splits of
// `split_tiles` K/V tiles each, in K/V tile steps: work item i (base unit
// i / splits, split i % splits, in the kernels' unit order) runs on CTA
// i % grid (causal: wave_order(i) % grid, the slot that runs it), and an item
// costs its tiles of each query tile plus one step of set-up and epilogue.
long long estimate_makespan(const ForwardCall& c, int win_left, int win_right, int splits,
                            int split_tiles, int grid) {
  const int rows = (c.d == 256) ? kBlockM : kRowsPerUnit;
  const int tiles_per_unit = rows / kBlockM;
  const int kv = kv_tile_rows(c.d);
  const int num_bh = c.B * c.H;
  const int per_head = static_cast<int>(units_per_head(c.N, c.d));
  const long long base_units = static_cast<long long>(num_bh) * per_head;
  long long cta_cost[1024] = {};
  long long worst = 0;
  for (long long u = 0; u < base_units; ++u) {
    // causal launches take the last query rows of every head first
    const int pair = c.causal ? per_head - 1 - static_cast<int>(u / num_bh)
                              : static_cast<int>(u % per_head);
    for (int sp = 0; sp < splits; ++sp) {
      long long cost = 0;
      for (int g = 0; g < tiles_per_unit; ++g) {
        const int r0 = pair * rows + g * kBlockM;
        if (r0 >= c.N) continue;
        int n0 = 0, n1 = 0;
        key_tile_range(r0, std::min(c.N, r0 + kBlockM), c.N, win_left, win_right, kv, &n0,
                       &n1);
        if (splits > 1) clip_to_split(sp, split_tiles, &n0, &n1);
        cost += n1 - n0;
      }
      // d = 256 tiles hold 64 keys: count in 128-key steps
      if (kv != kBlockN) cost = (cost + 1) / 2;
      if (cost == 0) continue;
      const long long item = u * splits + sp;
      const long long slot =
          c.causal ? wave_order(static_cast<int>(item), static_cast<int>(base_units * splits), grid)
                   : item;
      long long& t = cta_cost[slot % grid];
      t += cost + 1;
      worst = std::max(worst, t);
    }
  }
  return worst;
}

// The automatic split count of recent shapes: choosing one walks the whole
// persistent schedule for every candidate count, far longer than a launch.
struct PlanKey {
  int B, H, N, d, causal, win_left, win_right, num_sms;
  bool operator==(const PlanKey& o) const {
    return B == o.B && H == o.H && N == o.N && d == o.d && causal == o.causal &&
           win_left == o.win_left && win_right == o.win_right && num_sms == o.num_sms;
  }
};
struct PlanEntry {
  PlanKey key;
  int want;
  bool used;
};
constexpr int kPlanCacheSize = 64;
std::mutex g_plan_mutex;
PlanEntry g_plan_cache[kPlanCacheSize];
int g_plan_next = 0;

int automatic_split_count(const ForwardCall& c, int num_sms, int n_ktiles);

// Split count actually used for a requested one, and the K/V tiles per
// split.  0 asks for a count that fills the SMs: when the query units alone
// leave SMs idle (or unevenly loaded, as causal units are), the count with
// the shortest estimated makespan plus merge time.
void plan_splits(const ForwardCall& c, int requested, int num_sms, int* splits,
                 int* split_tiles) {
  const int n_ktiles = (c.N + kv_tile_rows(c.d) - 1) / kv_tile_rows(c.d);
  int want = requested;
  if (want <= 0) {
    const PlanKey key{c.B, c.H, c.N, c.d, c.causal, c.window_left < 0 ? -1 : c.window_left,
                      c.window_right < 0 ? -1 : c.window_right, num_sms};
    bool hit = false;
    {
      std::lock_guard<std::mutex> lock(g_plan_mutex);
      for (const PlanEntry& e : g_plan_cache)
        if (e.used && e.key == key) {
          want = e.want;
          hit = true;
          break;
        }
    }
    if (!hit) {
      want = automatic_split_count(c, num_sms, n_ktiles);
      std::lock_guard<std::mutex> lock(g_plan_mutex);
      g_plan_cache[g_plan_next] = PlanEntry{key, want, true};
      g_plan_next = (g_plan_next + 1) % kPlanCacheSize;
    }
  }
  if (want > n_ktiles) want = n_ktiles;
  if (want < 1) want = 1;
  const int tiles = (n_ktiles + want - 1) / want;
  *split_tiles = tiles;
  *splits = (n_ktiles + tiles - 1) / tiles;
}

int automatic_split_count(const ForwardCall& c, int num_sms, int n_ktiles) {
  int want = 1;
  {
    const long long units = static_cast<long long>(c.B) * c.H * units_per_head(c.N, c.d);
    const int grid = std::min(num_sms, 1024);
    if (units < grid && n_ktiles > 1) {
      const int win_left = (c.window_left < 0 || c.window_left > c.N) ? c.N : c.window_left;
      const int win_right =
          c.causal ? 0 : ((c.window_right < 0 || c.window_right > c.N) ? c.N : c.window_right);
      // Cost in 128-key tile steps of one query tile (about 1.1 us x d/128
      // on a GB300 SM).  The split partials are written by the forward and
      // read back by the merge (at about 5 TB/s), and the merge is one more
      // launch (about 3 us).
      const double step_us = 1.1 * c.d / 128.0;
      const double row_bytes = static_cast<double>(c.B) * c.H * c.N * (2.0 * c.d + 4.0);
      double best = static_cast<double>(estimate_makespan(c, win_left, win_right, 1, n_ktiles,
                                                          grid));
      for (int s = 2; s <= std::min(n_ktiles, 32); ++s) {
        const int tiles = (n_ktiles + s - 1) / s;
        const int used = (n_ktiles + tiles - 1) / tiles;
        if (used != s) continue;  // same split as a smaller count
        const double merge_us = (2.0 * s + 1.0) * row_bytes / 5.0e6 + 3.0;
        const double t =
            static_cast<double>(estimate_makespan(c, win_left, win_right, s, tiles, grid)) +
            merge_us / step_us;
        if (t < best) {
          best = t;
          want = s;
        }
      }
    }
  }
  return want;
}

// Workspace layout: partial O [S][B*H][N][d] (16-bit), then partial LSE
// [S][B*H][N] (fp32) at the next 256-byte boundary.
unsigned long long workspace_o_bytes(const ForwardCall& c, int splits) {
  return static_cast<unsigned long long>(splits) * c.B * c.H * c.N * c.d * 2ull;
}
unsigned long long workspace_bytes(const ForwardCall& c, int splits) {
  const unsigned long long o_bytes = (workspace_o_bytes(c, splits) + 255ull) & ~255ull;
  return o_bytes + static_cast<unsigned long long>(splits) * c.B * c.H * c.N * 4ull;
}

int splitkv_forward(const ForwardCall& c, int num_splits, void* workspace,
                    unsigned long long ws_bytes) {
  using namespace fa;
  int st = validate(c);
  if (st != FA_OK) return st;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  if (empty_problem(c)) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  // the SM count is needed only to choose the split count
  int num_sms = 0;
  if (num_splits == 0) {
    num_sms = fa_num_sms();
    if (num_sms <= 0) return FA_ERR_CUDA;
  }
  int splits = 1, split_tiles = 0;
  plan_splits(c, num_splits, num_sms, &splits, &split_tiles);
  if (splits == 1) return launch_forward(c, c.o, c.lse, 1, 0);
  if (workspace == nullptr || ws_bytes < workspace_bytes(c, splits)) return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* lse_part = reinterpret_cast<float*>(ws + ((workspace_o_bytes(c, splits) + 255ull) & ~255ull));
  st = launch_forward(c, ws, lse_part, splits, split_tiles);
  if (st != FA_OK) return st;
  CombineArgs a;
  a.num_bh = c.B * c.H;
  a.N = c.N;
  a.d = c.d;
  a.num_splits = splits;
  a.split_keys = split_tiles * kv_tile_rows(c.d);
  a.win_left = (c.window_left < 0 || c.window_left > c.N) ? c.N : c.window_left;
  a.win_right = (c.window_right < 0 || c.window_right > c.N) ? c.N : c.window_right;
  if (c.causal) a.win_right = 0;
  cudaError_t e = launch_splitkv_combine(ws, lse_part, c.o, c.lse, a, c.dtype == FA_DTYPE_BF16,
                                         fa_num_sms(), static_cast<cudaStream_t>(c.stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse, int B,
               int H, int H_kv, int N, int d, float scale, int causal, int window_left,
               int window_right, int dtype, void* stream) {
  using namespace fa;
  const ForwardCall c{q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left,
                      window_right, dtype, stream};
  int st = validate(c);
  if (st != FA_OK) return st;
  if (empty_problem(c)) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  return launch_forward(c, o, lse, 1, 0);
}

int fa_splitkv_workspace_bytes(int B, int H, int N, int d, int causal, int window_left,
                               int window_right, int num_splits, unsigned long long* bytes) {
  using namespace fa;
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  const ForwardCall c{nullptr, nullptr, nullptr, nullptr, nullptr, B, H, H > 0 ? H : 1, N,
                      d, 1.f, causal, window_left, window_right, FA_DTYPE_BF16, nullptr};
  int st = validate(c);
  if (st != FA_OK) return st;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  if (empty_problem(c)) return FA_OK;
  int num_sms = 0;
  if (num_splits == 0) {
    num_sms = fa_num_sms();
    if (num_sms <= 0) return FA_ERR_CUDA;
  }
  int splits = 1, split_tiles = 0;
  plan_splits(c, num_splits, num_sms, &splits, &split_tiles);
  *bytes = splits > 1 ? workspace_bytes(c, splits) : 0;
  return FA_OK;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                   int window_right, int dtype, int num_splits, void* workspace,
                   unsigned long long workspace_bytes, void* stream) {
  using namespace fa;
  const ForwardCall c{q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left,
                      window_right, dtype, stream};
  return splitkv_forward(c, num_splits, workspace, workspace_bytes);
}

// Split-KV into the library's fixed per-device scratch (declared with its
// limits and hazards in fa.h; the array and its look-up are in fa_noalloc.cu).
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int N, int d, float scale, int causal,
                           int window_left, int window_right, int dtype, int num_splits,
                           void* stream) {
  using namespace fa;
  const ForwardCall c{q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left,
                      window_right, dtype, stream};
  int st = validate(c);
  if (st != FA_OK) return st;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  if (empty_problem(c)) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  int num_sms = 0;
  if (num_splits == 0) {
    num_sms = fa_num_sms();
    if (num_sms <= 0) return FA_ERR_CUDA;
  }
  const unsigned long long limit = FA_NOALLOC_SCRATCH_BYTES;
  int splits = 1, split_tiles = 0;
  plan_splits(c, num_splits, num_sms, &splits, &split_tiles);
  if (num_splits == 0) {
    // automatic count: the largest count at or below the planned one that fits
    while (splits > 1 && workspace_bytes(c, splits) > limit)
      plan_splits(c, splits - 1, num_sms, &splits, &split_tiles);
  } else if (splits > 1 && workspace_bytes(c, splits) > limit) {
    return FA_ERR_SCRATCH_LIMIT;
  }
  if (splits == 1) return splitkv_forward(c, 1, nullptr, 0);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaError_t rc = cudaSuccess;
  void* scratch = noalloc_scratch(dev, &rc);
  if (scratch == nullptr || rc != cudaSuccess) return FA_ERR_CUDA;
  // the count is passed explicitly, so it resolves to `splits` again
  return splitkv_forward(c, splits, scratch, limit);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int batch, int max_seqlen, int total, int H, int H_kv,
                  int d, float scale, int causal, int window_left, int window_right, int dtype,
                  void* stream) {
  // self-attention within each sequence: the keys share the query offsets
  return fa_fwd_varlen_qk(q, k, v, o, lse, cu_seqlens, cu_seqlens, nullptr, nullptr, batch,
                          max_seqlen, max_seqlen, total, total, H, H_kv, d, scale, causal,
                          window_left, window_right, dtype, stream);
}

int fa_fwd_varlen_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens_q, const int* cu_seqlens_k, const int* seqused_q,
                     const int* seqused_k, int batch, int max_seqlen_q, int max_seqlen_k,
                     int total_q, int total_k, int H, int H_kv, int d, float scale, int causal,
                     int window_left, int window_right, int dtype, void* stream) {
  using namespace fa;
  // B = batch and N = max_seqlen_q in the shared checks
  ForwardCall c{q, k, v, o, lse, batch, H, H_kv, max_seqlen_q, d, scale, causal,
                window_left, window_right, dtype, stream, cu_seqlens_q, total_q};
  c.cu_seqlens_k = cu_seqlens_k;
  c.total_k = total_k;
  c.N_k = max_seqlen_k;
  c.seqused_q = seqused_q;
  c.seqused_k = seqused_k;
  if (total_q < 0 || total_k < 0 || max_seqlen_k < 0) return FA_ERR_INVALID_ARG;
  // positions and window bounds stay far from int overflow
  if (max_seqlen_q >= (1 << 30) || max_seqlen_k >= (1 << 30)) return FA_ERR_INVALID_ARG;
  int st = validate(c);
  if (st != FA_OK) return st;
  if (empty_problem(c) || total_q == 0) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || !aligned(seqused_q, 4) ||
      !aligned(seqused_k, 4))
    return FA_ERR_MISALIGNED;
  return launch_forward(c, o, lse, 1, 0);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Forward on host buffers: chunks of whole K/V-head groups are copied in,
// computed and copied out through a ring of device staging slots, with the
// copies in each direction on a helper stream of their own.
// ------------------------------------------------------------------------
namespace fa {
namespace {

constexpr int kHostSlots = 3;   // ring depth: copy-in, compute, copy-out in flight
constexpr int kHostChunks = 8;  // chunks a problem is cut into by default
constexpr unsigned long long kHostMinChunkBytes = 4ull << 20;  // input bytes per chunk

struct HostPlan {
  long long groups;     // B * H_kv: a K/V head with the query heads that read it
  long long per_chunk;  // groups per chunk
  long long chunks;
  int slots;
  unsigned long long q_bytes, kv_bytes, lse_bytes, slot_bytes;  // per slot
};

unsigned long long align256(unsigned long long x) { return (x + 255ull) & ~255ull; }

// Sub-buffers of one slot: Q and O (per_chunk * group query heads), K, V
// (per_chunk K/V heads), LSE; each starts on a 256-byte boundary.
void host_slot_layout(const ForwardCall& c, long long per_chunk, bool with_lse, HostPlan* pl) {
  const unsigned long long grp = static_cast<unsigned long long>(c.H / c.H_kv);
  const unsigned long long nd = static_cast<unsigned long long>(c.N) * c.d;
  const unsigned long long pc = static_cast<unsigned long long>(per_chunk);
  pl->per_chunk = per_chunk;
  pl->chunks = (pl->groups + per_chunk - 1) / per_chunk;
  pl->slots = static_cast<int>(std::min<long long>(kHostSlots, pl->chunks));
  pl->q_bytes = align256(pc * grp * nd * 2);
  pl->kv_bytes = align256(pc * nd * 2);
  pl->lse_bytes = with_lse ? align256(pc * grp * c.N * 4) : 0;
  pl->slot_bytes = 2 * pl->q_bytes + 2 * pl->kv_bytes + pl->lse_bytes;
}

// About kHostChunks chunks, each with at least kHostMinChunkBytes of input
// (small problems run as fewer, larger chunks).
void host_default_plan(const ForwardCall& c, bool with_lse, HostPlan* pl) {
  pl->groups = static_cast<long long>(c.B) * c.H_kv;
  const unsigned long long grp = static_cast<unsigned long long>(c.H / c.H_kv);
  const unsigned long long in_per_group = (grp + 2) * static_cast<unsigned long long>(c.N) * c.d * 2;
  long long per = (pl->groups + kHostChunks - 1) / kHostChunks;
  const long long min_per =
      static_cast<long long>((kHostMinChunkBytes + in_per_group - 1) / in_per_group);
  per = std::min(std::max(per, min_per), pl->groups);
  host_slot_layout(c, per, with_lse, pl);
}

// The default plan, shrunk (fewer groups per chunk, then fewer slots) until
// its slots fit in `ws_bytes`.  False when not even one group fits.
bool host_plan_for(const ForwardCall& c, bool with_lse, unsigned long long ws_bytes,
                   HostPlan* pl) {
  host_default_plan(c, with_lse, pl);
  const long long per0 = pl->per_chunk;
  for (int slots = pl->slots; slots >= 1; --slots) {
    long long lo = 1, hi = per0, best = 0;  // the largest fitting count
    while (lo <= hi) {
      const long long mid = lo + (hi - lo) / 2;
      host_slot_layout(c, mid, with_lse, pl);
      if (pl->slot_bytes * std::min(pl->slots, slots) <= ws_bytes) {
        best = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    if (best > 0) {
      host_slot_layout(c, best, with_lse, pl);
      pl->slots = std::min(pl->slots, slots);
      return true;
    }
  }
  return false;
}

// Helper streams and events of one device, made on first use and kept for
// the life of the process; the mutex serialises the enqueue of concurrent
// calls (which then share the streams in order).
struct HostPipe {
  std::once_flag once;
  cudaError_t init_rc = cudaSuccess;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t fork = nullptr, join_in = nullptr, join_out = nullptr;
  cudaEvent_t in[kHostSlots] = {}, done[kHostSlots] = {}, out[kHostSlots] = {};
  std::mutex mu;
};
HostPipe g_host_pipes[kMaxDevices];

HostPipe* host_pipe(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  HostPipe* hp = &g_host_pipes[dev];
  std::call_once(hp->once, [hp] {
    cudaError_t e = cudaStreamCreateWithFlags(&hp->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->s_out, cudaStreamNonBlocking);
    cudaEvent_t* evs[3 + 3 * kHostSlots] = {&hp->fork, &hp->join_in, &hp->join_out};
    for (int i = 0; i < kHostSlots; ++i) {
      evs[3 + i] = &hp->in[i];
      evs[3 + kHostSlots + i] = &hp->done[i];
      evs[3 + 2 * kHostSlots + i] = &hp->out[i];
    }
    for (cudaEvent_t* ev : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    hp->init_rc = e;
  });
  return hp->init_rc == cudaSuccess ? hp : nullptr;
}

int host_forward(const ForwardCall& c, const HostPlan& pl, const char* q_h, const char* k_h,
                 const char* v_h, char* o_h, float* lse_h, char* ws) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  HostPipe* hp = host_pipe(dev);
  if (hp == nullptr) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(hp->mu);
  cudaStream_t s = static_cast<cudaStream_t>(c.stream);
  const unsigned long long grp = static_cast<unsigned long long>(c.H / c.H_kv);
  const unsigned long long nd = static_cast<unsigned long long>(c.N) * c.d;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

  // fork: the helper streams start behind everything already on `s`
  // (earlier users of the workspace included)
  cudaError_t e = cudaEventRecord(hp->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->s_in, hp->fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->s_out, hp->fork, 0);
  int st = FA_OK;
  for (long long i = 0; i < pl.chunks && e == cudaSuccess; ++i) {
    const int slot = static_cast<int>(i % pl.slots);
    const long long g0 = i * pl.per_chunk;
    const unsigned long long ng =
        static_cast<unsigned long long>(std::min(pl.groups, g0 + pl.per_chunk) - g0);
    const unsigned long long q_off = static_cast<unsigned long long>(g0) * grp * nd * 2;
    const unsigned long long kv_off = static_cast<unsigned long long>(g0) * nd * 2;
    const unsigned long long qb = ng * grp * nd * 2, kvb = ng * nd * 2;
    char* const dq = ws + static_cast<unsigned long long>(slot) * pl.slot_bytes;
    char* const dout = dq + pl.q_bytes;
    char* const dk = dout + pl.q_bytes;
    char* const dv = dk + pl.kv_bytes;
    float* const dl = lse_h != nullptr ? reinterpret_cast<float*>(dv + pl.kv_bytes) : nullptr;

    // copy in, once the slot's previous chunk has been copied out
    if (i >= pl.slots) e = cudaStreamWaitEvent(hp->s_in, hp->out[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq, q_h + q_off, qb, h2d, hp->s_in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k_h + kv_off, kvb, h2d, hp->s_in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v_h + kv_off, kvb, h2d, hp->s_in);
    if (e == cudaSuccess) e = cudaEventRecord(hp->in[slot], hp->s_in);
    // compute on the caller's stream: the chunk's groups as ng heads of
    // K/V with grp query heads each
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->in[slot], 0);
    if (e != cudaSuccess) break;
    ForwardCall cc = c;
    cc.q = dq;
    cc.k = dk;
    cc.v = dv;
    cc.o = dout;
    cc.lse = dl;
    cc.B = static_cast<int>(ng);
    cc.H = static_cast<int>(grp);
    cc.H_kv = 1;
    st = launch_forward(cc, dout, dl, 1, 0);
    if (st != FA_OK) break;
    // copy out
    e = cudaEventRecord(hp->done[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->s_out, hp->done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o_h + q_off, dout, qb, d2h, hp->s_out);
    if (e == cudaSuccess && dl != nullptr)
      e = cudaMemcpyAsync(lse_h + static_cast<unsigned long long>(g0) * grp * c.N, dl,
                          ng * grp * c.N * 4, d2h, hp->s_out);
    if (e == cudaSuccess) e = cudaEventRecord(hp->out[slot], hp->s_out);
  }
  // join both helper streams back into `s` (after a failure too)
  cudaError_t j = cudaEventRecord(hp->join_in, hp->s_in);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s, hp->join_in, 0);
  if (j == cudaSuccess) j = cudaEventRecord(hp->join_out, hp->s_out);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s, hp->join_out, 0);
  if (st != FA_OK) return st;
  return (e == cudaSuccess && j == cudaSuccess) ? FA_OK : FA_ERR_CUDA;
}

int host_validate(const ForwardCall& c) {
  const int st = validate(c);
  if (st != FA_OK) return st;
  if (c.window_left < -1 || c.window_right < -1) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_fwd_host_workspace_bytes(int B, int H, int H_kv, int N, int d, int with_lse,
                                unsigned long long* bytes) {
  using namespace fa;
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  if (with_lse != 0 && with_lse != 1) return FA_ERR_INVALID_ARG;
  const ForwardCall c{nullptr, nullptr, nullptr, nullptr, nullptr, B, H, H_kv, N, d, 1.f, 0, -1,
                      -1, FA_DTYPE_BF16, nullptr};
  const int st = host_validate(c);
  if (st != FA_OK) return st;
  if (empty_problem(c)) return FA_OK;
  HostPlan pl;
  host_default_plan(c, with_lse != 0, &pl);
  *bytes = pl.slot_bytes * pl.slots;
  return FA_OK;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                int window_right, int dtype, void* workspace,
                unsigned long long workspace_bytes, void* stream) {
  using namespace fa;
  const ForwardCall c{q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left,
                      window_right, dtype, stream};
  int st = host_validate(c);
  if (st != FA_OK) return st;
  if (empty_problem(c)) return FA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || workspace == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  HostPlan pl;
  if (!host_plan_for(c, lse != nullptr, workspace_bytes, &pl)) return FA_ERR_INVALID_ARG;
  return host_forward(c, pl, static_cast<const char*>(q), static_cast<const char*>(k),
                      static_cast<const char*>(v), static_cast<char*>(o), lse,
                      static_cast<char*>(workspace));
}

int fa_bwd_workspace_bytes(int B, int H, int N, unsigned long long* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  const unsigned long long n_pad = (static_cast<unsigned long long>(N) + 127ull) / 128ull * 128ull;
  *bytes = 2ull * static_cast<unsigned long long>(B) * static_cast<unsigned long long>(H) * n_pad * 4ull;
  return FA_OK;
}

}  // extern "C"

namespace fa {
namespace {

// The packed-batch arguments of a backward launch (all nullptr / 0 for the
// [B][H][N][d] layout): query offsets and rows, key offsets and rows (the
// query ones for self-attention), used lengths, the longest key length.
struct BwdPacked {
  const int* cu_q = nullptr;
  const int* cu_k = nullptr;
  const int* used_q = nullptr;
  const int* used_k = nullptr;
  int total_q = 0, total_k = 0, N_k = 0;
};

// fa_bwd and fa_bwd_varlen(_qk): B sequences of N rows ([B][H][N][d]), or,
// with cu_q, B packed sequences of at most N query and N_k key rows.
int bwd_launch(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, void* workspace,
               unsigned long long workspace_bytes, int B, int H, int H_kv, int N, int d,
               float scale, int causal, int window_left, int window_right, int dtype,
               void* stream, const BwdPacked& pk) {
  const int* cu_seqlens = pk.cu_q;
  const int total = pk.total_q;
  const ForwardCall c{q, k, v, dq, nullptr, B, H, H_kv, N, d, scale, causal, window_left,
                      window_right, dtype, stream};
  int st = validate(c);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const bool packed = cu_seqlens != nullptr;
  if (packed && (total < 0 || pk.total_k < 0 || pk.N_k < 0 || pk.cu_k == nullptr))
    return FA_ERR_INVALID_ARG;
  if (empty_problem(c) || (packed && total == 0)) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  if (packed && (!aligned(pk.cu_k, 4) || !aligned(pk.used_q, 4) || !aligned(pk.used_k, 4)))
    return FA_ERR_MISALIGNED;
  const int N_k = packed ? pk.N_k : N;
  const int total_k = packed ? pk.total_k : 0;
  if (o == nullptr || lse == nullptr || dout == nullptr || dk == nullptr || dv == nullptr ||
      workspace == nullptr)
    return FA_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256) || (packed && !aligned(cu_seqlens, 4)))
    return FA_ERR_MISALIGNED;
  unsigned long long need = 0;
  fa_bwd_workspace_bytes(B, H, N, &need);
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_tiles = (static_cast<long long>(N) + 127) / 128;
  const long long n_tiles_k = (static_cast<long long>(N_k) + 127) / 128;
  if (bh * n_tiles >= (1ll << 31) || static_cast<long long>(B) * H_kv * n_tiles_k >= (1ll << 31))
    return FA_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DevState dev_state;
  DevState* info = device_info(dev, &dev_state);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  if (!info->ok) return FA_ERR_UNSUPPORTED;
  const bool bf16 = dtype == FA_DTYPE_BF16;
  const int ibh = static_cast<int>(bh), ibkv = B * H_kv;
  BwdParams p;
  if (packed) {
    // (no key rows at all: the K/V maps view the query memory; every key
    // tile is then empty and nothing reads through them)
    const void* kb = total_k > 0 ? k : q;
    const void* vb = total_k > 0 ? v : q;
    const int k_rows = total_k > 0 ? total_k : total;
    const int kv_heads = total_k > 0 ? H_kv : H;
    if (!encode_packed_map(&p.tm_q, q, total, H, d, bf16, 128, d / 64) ||
        !encode_packed_map(&p.tm_k, kb, k_rows, kv_heads, d, bf16, 128, d / 64) ||
        !encode_packed_map(&p.tm_v, vb, k_rows, kv_heads, d, bf16, 128, d / 64) ||
        !encode_packed_map(&p.tm_do, dout, total, H, d, bf16, 128, d / 64))
      return FA_ERR_CUDA;
  } else if (!encode_qkvo_map(&p.tm_q, q, N, d, ibh, bf16, 128, d / 64) ||
             !encode_qkvo_map(&p.tm_k, k, N, d, ibkv, bf16, 128, d / 64) ||
             !encode_qkvo_map(&p.tm_v, v, N, d, ibkv, bf16, 128, d / 64) ||
             !encode_qkvo_map(&p.tm_do, dout, N, d, ibh, bf16, 128, d / 64)) {
    return FA_ERR_CUDA;
  }
  const int n_pad = static_cast<int>(n_tiles * 128);
  float* lse2 = static_cast<float*>(workspace);
  float* dsum = lse2 + static_cast<long long>(ibh) * n_pad;
  p.lse2 = lse2;
  p.dsum = dsum;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.status = info->status;
  p.timeout_ns = g_timeout_ns.load();
  p.N = N;
  p.n_pad = n_pad;
  p.n_tiles = static_cast<int>(n_tiles);
  p.num_bh = ibh;
  p.num_bkv = ibkv;
  p.H = H;
  p.H_kv = H_kv;
  p.group = H / H_kv;
  // (an unbounded window reaches every key: N + N_k covers any shift)
  const int unbounded = N + N_k;
  p.win_left = (window_left < 0 || window_left > unbounded) ? unbounded : window_left;
  p.win_right = (window_right < 0 || window_right > unbounded) ? unbounded : window_right;
  if (causal) p.win_right = 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.cu_seqlens = cu_seqlens;
  p.cu_seqlens_k = packed ? pk.cu_k : nullptr;
  p.seqused_q = packed ? pk.used_q : nullptr;
  p.seqused_k = packed ? pk.used_k : nullptr;
  p.total_rows = packed ? total : 0;
  p.total_rows_k = total_k;
  p.N_k = N_k;
  p.n_tiles_k = static_cast<int>(n_tiles_k);
  BwdParams p_kv = p, p_q = p;
  p_kv.num_units = static_cast<int>(static_cast<long long>(ibkv) * n_tiles_k);
  p_q.num_units = static_cast<int>(bh * n_tiles);
  // packed causal launches order their units from a per-CTA table (both
  // kernels, or neither)
  const long long max_tiles = n_tiles > n_tiles_k ? n_tiles : n_tiles_k;
  const int table = (packed && causal && B <= kTableSeqs && max_tiles > 1 &&
                     max_tiles <= kBwdTableTiles)
                        ? 1
                        : 0;
  p_kv.unit_table = table;
  p_q.unit_table = table;
  int grid = info->num_sms;
  const int cap = g_max_ctas.load();
  if (cap > 0 && cap < grid) grid = cap;
  const int grid_kv = p_kv.num_units < grid ? p_kv.num_units : grid;
  const int grid_q = p_q.num_units < grid ? p_q.num_units : grid;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      (d == 64) ? launch_bwd_d64(p_kv, p_q, o, dout, lse, lse2, dsum, causal != 0, bf16, grid_kv,
                                 grid_q, info->num_sms, s)
                : launch_bwd_d128(p_kv, p_q, o, dout, lse, lse2, dsum, causal != 0, bf16,
                                  grid_kv, grid_q, info->num_sms, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, void* workspace,
           unsigned long long workspace_bytes, int B, int H, int H_kv, int N, int d,
           float scale, int causal, int window_left, int window_right, int dtype,
           void* stream) {
  return fa::bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H,
                        H_kv, N, d, scale, causal, window_left, window_right, dtype, stream,
                        fa::BwdPacked{});
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens,
                  int batch, int max_seqlen, int total, int H, int H_kv, int d, float scale,
                  int causal, int window_left, int window_right, int dtype, void* workspace,
                  unsigned long long workspace_bytes, void* stream) {
  if (batch > 0 && H > 0 && max_seqlen > 0 && total > 0 && cu_seqlens == nullptr)
    return FA_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr) {
    // nothing to do only if the problem is empty; the checks are shared
    if (batch < 0 || H < 0 || max_seqlen < 0 || total < 0) return FA_ERR_INVALID_ARG;
    return FA_OK;
  }
  fa::BwdPacked pk;
  pk.cu_q = cu_seqlens;
  pk.cu_k = cu_seqlens;
  pk.total_q = total;
  pk.total_k = total;
  pk.N_k = max_seqlen;
  return fa::bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, batch,
                        H, H_kv, max_seqlen, d, scale, causal, window_left, window_right, dtype,
                        stream, pk);
}

int fa_bwd_varlen_qk(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     const int* cu_seqlens_q, const int* cu_seqlens_k, const int* seqused_q,
                     const int* seqused_k, int batch, int max_seqlen_q, int max_seqlen_k,
                     int total_q, int total_k, int H, int H_kv, int d, float scale, int causal,
                     int window_left, int window_right, int dtype, void* workspace,
                     unsigned long long workspace_bytes, void* stream) {
  if (batch < 0 || H < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0)
    return FA_ERR_INVALID_ARG;
  // positions and window bounds stay far from int overflow
  if (max_seqlen_q >= (1 << 30) || max_seqlen_k >= (1 << 30)) return FA_ERR_INVALID_ARG;
  if (batch == 0 || H == 0 || max_seqlen_q == 0 || total_q == 0) {
    // nothing to do; the shared checks of the other arguments still apply
    return fa::bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, batch,
                          H, H_kv, max_seqlen_q, d, scale, causal, window_left, window_right,
                          dtype, stream, fa::BwdPacked{});
  }
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
  fa::BwdPacked pk;
  pk.cu_q = cu_seqlens_q;
  pk.cu_k = cu_seqlens_k;
  pk.used_q = seqused_q;
  pk.used_k = seqused_k;
  pk.total_q = total_q;
  pk.total_k = total_k;
  pk.N_k = max_seqlen_k;
  return fa::bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, batch,
                        H, H_kv, max_seqlen_q, d, scale, causal, window_left, window_right,
                        dtype, stream, pk);
}

int fa_fwd_fp8_workspace_bytes(int B, int H_kv, int N, int d, unsigned long long* bytes) {
  if (bytes == nullptr) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || H_kv < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const unsigned long long n_pad = (static_cast<unsigned long long>(N) + 127ull) / 128ull * 128ull;
  *bytes = static_cast<unsigned long long>(B) * static_cast<unsigned long long>(H_kv) * d * n_pad;
  return FA_OK;
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int H_kv, int N, int d, float scale, float descale_q, float descale_k,
               float descale_v, int causal, int window_left, int window_right, void* workspace,
               unsigned long long workspace_bytes, void* stream) {
  using namespace fa;
  ForwardCall c{q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left,
                window_right, FA_DTYPE_BF16, stream};
  int st = validate(c);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  for (float x : {descale_q, descale_k, descale_v})
    if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_INVALID_ARG;
  if (empty_problem(c)) return FA_OK;
  st = check_pointers(c);
  if (st != FA_OK) return st;
  unsigned long long need = 0;
  fa_fwd_fp8_workspace_bytes(B, H_kv, N, d, &need);
  if (workspace == nullptr || workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  c.fp8 = true;
  c.descale_q = descale_q;
  c.descale_k = descale_k;
  c.descale_v = descale_v;
  c.vt = workspace;
  c.n_pad = static_cast<int>((static_cast<long long>(N) + 127) / 128 * 128);
  return launch_forward(c, o, lse, 1, 0);
}

int fa_get_device_status(void* stream, int* site) {
  using namespace fa;
  if (site != nullptr) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  DevState dev_state;
  DevState* info = device_info(dev, &dev_state);
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
  DevState dev_state;
  DevState* info = device_info(dev, &dev_state);
  if (info == nullptr || info->status == nullptr) return FA_ERR_CUDA;
  if (!info->ok) return FA_ERR_UNSUPPORTED;
  cudaError_t e = launch_watchdog_selftest(
      info->status, static_cast<unsigned long long>(timeout_us) * 1000ull,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
