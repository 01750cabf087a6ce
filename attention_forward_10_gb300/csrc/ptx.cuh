// ptx.cuh -- hand-written inline-PTX wrappers for sm_103a: mbarriers, TMA
// tensor copies, tcgen05 tensor-memory allocation / MMA / loads / stores.
//
// Every wrapper is a thin shell around one PTX instruction (or a fixed pair
// of them); there is no CUTLASS or CuTe underneath.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --------------------------------------------------------------------------
// mbarrier
// --------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same test, but a thread whose phase is not complete may sleep up to
// `hint_ns` nanoseconds (it wakes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Named barrier over `count` threads (ids 1..15; id 0 is __syncthreads).
// Programmatic dependent launch.  griddep_wait: block until the grid this
// one depends on (the previous kernel of the stream, when this one was
// launched with programmatic stream serialisation) has completed and its
// memory is visible; a no-op otherwise.  griddep_launch_dependents: let the
// next such kernel of the stream start launching once every CTA of this
// grid has issued it (or exited).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and bulk-group bookkeeping
// --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// 4-D tiled load global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// 5-D tiled load global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(bar)
      : "memory");
}

// 5-D tiled store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_5d(const void* map, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// 4-D tiled store shared -> global (bulk-group completion).
// 1-D bulk copy global -> shared, completing `bytes` on mbarrier `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :
      : "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const void* map, uint32_t src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store has finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tcgen05) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b,
                                             uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// --------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, fences
// --------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns, base address written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   start address, leading / stride byte offsets (all in bytes; encoded >>4),
//   descriptor version 1 (bits 46-47), swizzle mode "128B" (value 2, bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo,
                                                    uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16,
//   1 = bf16), bit 15 A major (0 = K), bit 16 B major (1 = MN),
//   bits 17-22 N>>3, bits 24-28 M>>4.
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N, bool bf16,
                                                      bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Warpgroup-wide register budget changes (all 4 warps of a warpgroup).
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// --------------------------------------------------------------------------
// MMA bursts
// --------------------------------------------------------------------------
// 8 back-to-back K=16 MMAs D (+)= A*B^T, both operands K-major
// 128B-swizzled tiles in shared memory: step k adds a fixed offset (in 16-byte
// units) to both descriptors; the first step overwrites D when `accumulate` is
// 0, later steps accumulate.  Issued as one burst so the tensor pipe is fed
// without gaps.
__device__ __forceinline__ void mma_ss_kmajor_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ak, bk;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 ak, %1, 2;\n\t"
      "add.s64 bk, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 4;\n\t"
      "add.s64 bk, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 6;\n\t"
      "add.s64 bk, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1024;\n\t"
      "add.s64 bk, %2, 1024;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1026;\n\t"
      "add.s64 bk, %2, 1026;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1028;\n\t"
      "add.s64 bk, %2, 1028;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1030;\n\t"
      "add.s64 bk, %2, 1030;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 back-to-back K=16 MMAs D (+)= A*B^T, both operands K-major
// 128B-swizzled tiles in shared memory: step k adds a fixed offset (in 16-byte
// units) to both descriptors; the first step overwrites D when `accumulate` is
// 0, later steps accumulate.  Issued as one burst so the tensor pipe is fed
// without gaps.
__device__ __forceinline__ void mma_ss_kmajor_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ak, bk;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 ak, %1, 2;\n\t"
      "add.s64 bk, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 4;\n\t"
      "add.s64 bk, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 6;\n\t"
      "add.s64 bk, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 back-to-back K=16 MMAs D (+)= A*B^T over a 256-wide reduction: A a K-major
// 128B-swizzled 128-row tile (64-element column blocks 16 KB apart), B a
// K-major 64-row tile (column blocks 8 KB apart).  First step overwrites D
// unless `accumulate`.
__device__ __forceinline__ void mma_ss_kmajor_x16_q128_k64(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ak, bk;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 ak, %1, 2;\n\t"
      "add.s64 bk, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 4;\n\t"
      "add.s64 bk, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 6;\n\t"
      "add.s64 bk, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1024;\n\t"
      "add.s64 bk, %2, 512;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1026;\n\t"
      "add.s64 bk, %2, 514;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1028;\n\t"
      "add.s64 bk, %2, 516;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 1030;\n\t"
      "add.s64 bk, %2, 518;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 2048;\n\t"
      "add.s64 bk, %2, 1024;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 2050;\n\t"
      "add.s64 bk, %2, 1026;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 2052;\n\t"
      "add.s64 bk, %2, 1028;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 2054;\n\t"
      "add.s64 bk, %2, 1030;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 3072;\n\t"
      "add.s64 bk, %2, 1536;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 3074;\n\t"
      "add.s64 bk, %2, 1538;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 3076;\n\t"
      "add.s64 bk, %2, 1540;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 3078;\n\t"
      "add.s64 bk, %2, 1542;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ak, bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 back-to-back K=16 MMAs D (+)= A*B, A in tensor memory (step k reads
// columns a_tmem + 8k), B an MN-major 128B-swizzled tile with 16-row steps
// 2048 bytes apart.  First step overwrites D unless `accumulate`.
__device__ __forceinline__ void mma_ts_mnmajor_x4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 bk;\n\t.reg .b32 ak;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "add.u32 ak, %1, 8;\n\t"
      "add.s64 bk, %2, 128;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ak], bk, %3, pt;\n\t"
      "add.u32 ak, %1, 16;\n\t"
      "add.s64 bk, %2, 256;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ak], bk, %3, pt;\n\t"
      "add.u32 ak, %1, 24;\n\t"
      "add.s64 bk, %2, 384;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [ak], bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// --------------------------------------------------------------------------
// Arithmetic helpers
// --------------------------------------------------------------------------
// Packed pair arithmetic (two fp32 lanes per instruction).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// (a.lo*b.lo + c.lo, a.hi*b.hi + c.hi), round to nearest
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats (round to nearest even) into one 32-bit word: `lo` in the
// low half, `hi` in the high half.
// 4 back-to-back K=32 MMAs of kind::f8f6f4 (FP8 E4M3 x E4M3 -> fp32), both
// operands K-major 128B-swizzled tiles in shared memory with 128-byte rows:
// step k reads bytes [32k, 32k + 32) of every row (descriptor + 2k).  The
// first step overwrites D unless `accumulate`.
__device__ __forceinline__ void mma_f8_ss_kmajor_x4(uint32_t d_tmem, uint64_t a_desc,
                                                    uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 ak, bk;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 ak, %1, 2;\n\t"
      "add.s64 bk, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 4;\n\t"
      "add.s64 bk, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ak, bk, %3, pt;\n\t"
      "add.s64 ak, %1, 6;\n\t"
      "add.s64 bk, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ak, bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 back-to-back K=32 MMAs of kind::f8f6f4 with A in tensor memory (four
// E4M3 elements per 32-bit column, so step k reads columns a_tmem + 8k) and
// B a K-major 128B-swizzled tile with 128-byte rows (descriptor + 2k).
__device__ __forceinline__ void mma_f8_ts_kmajor_x4(uint32_t d_tmem, uint32_t a_tmem,
                                                    uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b64 bk;\n\t.reg .b32 ak;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\t"
      "setp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, pf;\n\t"
      "add.u32 ak, %1, 8;\n\t"
      "add.s64 bk, %2, 2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ak], bk, %3, pt;\n\t"
      "add.u32 ak, %1, 16;\n\t"
      "add.s64 bk, %2, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ak], bk, %3, pt;\n\t"
      "add.u32 ak, %1, 24;\n\t"
      "add.s64 bk, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [ak], bk, %3, pt;\n\t"
      "}"
      :
      : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four fp32 values rounded to nearest FP8 E4M3 (saturating to +-448), packed
// into one 32-bit word, element k in byte k.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// The low / high 16-bit element of a packed pair, widened to fp32 (exact).
template <bool BF16>
__device__ __forceinline__ float unpack_lo(uint32_t w) {
  if constexpr (BF16) return __uint_as_float(w << 16);
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f) : "r"(w));
  return f;
}
template <bool BF16>
__device__ __forceinline__ float unpack_hi(uint32_t w) {
  if constexpr (BF16) return __uint_as_float(w & 0xffff0000u);
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}"
      : "=f"(f) : "r"(w));
  return f;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// --------------------------------------------------------------------------
// TMEM loads (load + wait fused so the outputs are never read early) and
// stores, 32x32b shape: thread i of the warp addresses TMEM lane
// (lane_base + i), consecutive 32-bit columns.
// --------------------------------------------------------------------------
// Load 32 consecutive 32-bit TMEM columns of this thread's lane (32x32b
// shape) and wait for the load to land before the registers are used.
__device__ __forceinline__ void tmem_ld_x32_sync(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Store 16 consecutive 32-bit TMEM columns of this thread's lane (32x32b).
// 32 consecutive columns at `ta` into ra and 32 at `tb` into rb (this warp's
// 32 lanes), with a single wait for both loads.
__device__ __forceinline__ void tmem_ld_2x32_sync(uint32_t ta, uint32_t* ra, uint32_t tb,
                                                  uint32_t* rb) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7]), "=r"(ra[8]), "=r"(ra[9]), "=r"(ra[10]), "=r"(ra[11]), "=r"(ra[12]), "=r"(ra[13]), "=r"(ra[14]), "=r"(ra[15]), "=r"(ra[16]), "=r"(ra[17]), "=r"(ra[18]), "=r"(ra[19]), "=r"(ra[20]), "=r"(ra[21]), "=r"(ra[22]), "=r"(ra[23]), "=r"(ra[24]), "=r"(ra[25]), "=r"(ra[26]), "=r"(ra[27]), "=r"(ra[28]), "=r"(ra[29]), "=r"(ra[30]), "=r"(ra[31]), "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7]), "=r"(rb[8]), "=r"(rb[9]), "=r"(rb[10]), "=r"(rb[11]), "=r"(rb[12]), "=r"(rb[13]), "=r"(rb[14]), "=r"(rb[15]), "=r"(rb[16]), "=r"(rb[17]), "=r"(rb[18]), "=r"(rb[19]), "=r"(rb[20]), "=r"(rb[21]), "=r"(rb[22]), "=r"(rb[23]), "=r"(rb[24]), "=r"(rb[25]), "=r"(rb[26]), "=r"(rb[27]), "=r"(rb[28]), "=r"(rb[29]), "=r"(rb[30]), "=r"(rb[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :
      : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Store 32 consecutive 32-bit TMEM columns of this thread's lane (32x32b).
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :
      : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Load 128 consecutive columns as four 32-column loads (four independent
// 32-register destination blocks), then wait once.
__device__ __forceinline__ void tmem_ld_x32x4_sync(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
}

// tmem_ld_x32x4_sync that also returns, in m[j], the maximum of the 32
// values that load j brought into this thread (tcgen05.ld.red, a form of
// the tensor-memory load that sm_103a adds: the reduction runs in the load
// path, so the row maximum of a score tile costs no FMNMX instructions).
// NaN inputs are not propagated (no .NaN qualifier); -inf and signed zeros
// reduce as fmaxf does.
__device__ __forceinline__ void tmem_ld_max_x32x4_sync(uint32_t taddr, uint32_t* r, float* m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %128, [%132];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %129, [%133];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, %130, [%134];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, %131, [%135];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), "=f"(m[0]), "=f"(m[1]), "=f"(m[2]), "=f"(m[3])
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
}

// Two 32-column reducing loads (columns [0, 64) at taddr), one wait; m[j] is
// the maximum of block j.  See tmem_ld_max_x32x4_sync.
__device__ __forceinline__ void tmem_ld_max_x32x2_sync(uint32_t taddr, uint32_t* r, float* m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %64, [%66];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %65, [%67];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=f"(m[0]), "=f"(m[1])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
}

}  // namespace fa
