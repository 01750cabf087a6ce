// fa_noalloc.cu -- the fixed device scratch of fa_fwd_splitkv_noalloc.
//
// Some callers of the split-KV forward cannot hand it a workspace:
//   * code that must not call cudaMalloc / cudaFree on its hot path, because
//     both can synchronise the device and stall every stream (cudaFree always
//     does), which a latency-bound serving loop cannot afford;
//   * engines that reserve their device memory once at start-up and have no
//     allocator left to hand out a scratch buffer per call;
//   * plain C callers with no caching allocator, which would otherwise have to
//     keep a workspace alive across asynchronous calls themselves.
// For them the library keeps one scratch array per device in static device
// memory (FA_NOALLOC_SCRATCH_BYTES bytes), so the call allocates nothing.
//
// The array sits in its own translation unit: with lazily loaded CUDA
// modules its memory is taken only once a process first asks for its address,
// not by every user of the library.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_launch.h"

// File-scope scratch.  Nothing in it needs to start at zero: every byte the
// merge kernel reads was written earlier in the same call by the split
// forward.  All calls on one device share it (see fa_fwd_splitkv_noalloc).
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace fa {
namespace {

constexpr int kScratchDevices = 64;

// The scratch address of each device, with the id of the context it was
// looked up in.
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx = 0;
};
ScratchAddr g_scratch[kScratchDevices];
std::mutex g_scratch_mutex;

}  // namespace

void* noalloc_scratch(int dev, cudaError_t* rc) {
  *rc = cudaSuccess;
  if (dev < 0 || dev >= kScratchDevices) {
    *rc = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& a = g_scratch[dev];
  // The address is a device address of one context: a call made under
  // another one (a new primary context after cudaDeviceReset, or a driver
  // context of the caller's own) looks it up again instead of handing the
  // kernels an address of a context that may be gone.
  const unsigned long long ctx = current_context_id();
  if (a.ptr != nullptr && ctx != 0 && ctx == a.ctx) return a.ptr;
  // First call on this device and context (which is current): look the
  // array up.  A failure is not cached, so a later call tries again, and the
  // runtime's error state is cleared so that it is not reported against an
  // unrelated later call.
  void* p = nullptr;
  *rc = cudaGetSymbolAddress(&p, g_fa_noalloc_scratch);
  if (*rc != cudaSuccess) {
    cudaGetLastError();
    a.ptr = nullptr;
    a.ctx = 0;
    return nullptr;
  }
  a.ptr = p;
  a.ctx = current_context_id();
  return p;
}

}  // namespace fa
