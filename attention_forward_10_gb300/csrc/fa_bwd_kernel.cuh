// fa_bwd_kernel.cuh -- attention backward (dQ, dK, dV) for sm_103a, d <= 128.
//
// What is computed (flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp",
// CollectiveMainloopBwd::mma, with its LSE in natural-log units here):
//   P_ij  = exp(s_ij - LSE_i)         (s = scale Q K^T, masked entries 0)
//   dP_ij = dO_i . v_j,   D_i = rowsum(dO_i * O_i)  (the page's dPsum)
//   dS_ij = P_ij (dP_ij - D_i)
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K
//
// Two kernels and no atomics, so every gradient is deterministic:
//   * dK/dV kernel: a work unit is one 128-key tile of one K/V head; it loops
//     over the query tiles (and, for grouped heads, the query heads) that
//     can see those keys, computing S^T = K Q^T and dP^T = V dO^T with one
//     key per tensor-memory lane, so that P^T and dS^T are the A operands of
//     dV += P^T dO and dK += dS^T Q straight from tensor memory.
//   * dQ kernel: a work unit is one 128-row query tile; it loops over the
//     key tiles that row tile sees, computing S = Q K^T and dP = dO V^T (one
//     query per lane) and dQ += dS K.
// A pre-pass writes -LSE_i * log2(e) and -D_i into a workspace padded to
// whole 128-row tiles (padding: -inf and 0, so padded query rows get P = 0).
//
// Warp roles (352 threads): warps 0-7 compute P and dS, one tensor-memory
// lane (row) per thread, warps 0-3 for the first 64 columns of a tile and
// warps 4-7 for the last 64, and split the epilogue the same way; warp 8
// issues TMA copies; warp 9 issues the S and dP products, warp 10 the
// gradient products.  Tensor memory, columns:
// [0,128) S, [128,256) dP, then the fp32 accumulators: dV and dK (dK/dV
// kernel) or dQ (dQ kernel), D columns each, and in the dQ kernel dS at
// [384,480).
//
// Each step's elementwise work runs in two phases, P from S (phase A) and dS
// from dP and P (phase B), each overlapping a product on the tensor pipe:
//   * dK/dV kernel, per step: S^T, dP^T, dV += P^T dO, dK += dS^T Q.  Phase A
//     starts when S^T has completed and runs while dP^T is computed; it
//     stores P^T (16-bit) over the first 32 of each half's 64 S^T columns,
//     and the dV product starts; phase B runs meanwhile and stores dS^T the
//     same way over dP^T's columns for the dK product.
//   * dQ kernel: the issuer runs one step ahead.  After step j's S has been
//     read by every thread (phase A), S of step j+1 is issued; phase B of
//     step j writes dS to its own columns, then dQ += dS K of step j and dP
//     of step j+1 are issued.  The next dS store waits for that dP's commit,
//     which also covers the dQ product that read the previous dS.
// A product that overwrites tensor-memory columns an earlier product read
// (S^T over P^T, dP^T over dS^T) is issued only after that product's commit
// has arrived: the PTX ISA orders two tcgen05.mma of one thread only when
// they share the accumulator and shape.  Every mbarrier wait is bounded.
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_params.h"
#include "ptx.cuh"

namespace fa {
namespace bwd {

// Entry check failure of the backward kernels (not a wait): the status word
// gets FA_ERR_MISALIGNED with this site code.
constexpr int kStatusMisaligned = 3;  // == FA_ERR_MISALIGNED
constexpr int kSiteSmemBase = 13;

constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // issues the S (S^T) and dP (dP^T) products
constexpr int kGradWarp = 10;  // issues the gradient products (dV and dK, or dQ)
constexpr int kEwThreads = 256;  // warps 0-7
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256;
constexpr uint32_t kColDS = 384;  // dQ kernel: dS (96 columns)
// dK/dV kernel: S^T and dP^T alternate between the regions at 0 and 128
// from step to step (step j: S^T at region(j), dP^T at region(j + 1)).
__device__ __forceinline__ uint32_t region(uint32_t step) { return (step & 1u) * 128u; }

// Shared memory layout of both kernels (tiles 1024-byte aligned for the
// 128-byte swizzle): two 128-row tiles that stay for the whole unit (K, V or
// Q, dO); ring A, three stages of the streamed tile needed first in a step
// (Q in the dK/dV kernel, K in the dQ kernel); ring B, two stages of the
// other one (dO, with the stage's 128 LSE2 and 128 D values, or V); then
// the barriers.  The dynamic shared memory base must be 1024-byte aligned:
// no slack is reserved (the kernels check and give up with
// FA_ERR_MISALIGNED otherwise).
template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr uint32_t kTile = 128 * D * 2;
  static constexpr int kStagesA = 3, kStagesB = 2;
  static constexpr uint32_t kFixOff = 0;                                 // 2 tiles
  static constexpr uint32_t kRingAOff = 2 * kTile;                       // stage s: 1 tile
  static constexpr uint32_t kRingBOff = kRingAOff + kStagesA * kTile;    // stage s: 1 tile
  static constexpr uint32_t kVecOff = kRingBOff + kStagesB * kTile;      // stage s: 1 KB
  static constexpr uint32_t kBarOff = kVecOff + kStagesB * 1024;
  // barriers
  static constexpr int kFixFull = 0, kFixEmpty = 1;
  static constexpr int kAFull = 2;    // + stage
  static constexpr int kAEmpty = 5;   // + stage
  static constexpr int kBFull = 8;    // + stage
  static constexpr int kBEmpty = 10;  // + stage
  static constexpr int kSDone = 12;     // the S (S^T) product has completed
  static constexpr int kDPDone = 13;    // the dP (dP^T) product has completed
  static constexpr int kPStored = 14;   // dK/dV: P^T is in tensor memory (256 arrivals)
  static constexpr int kDSStored = 15;  // dS (dS^T) is in tensor memory (256 arrivals)
  static constexpr int kSRead = 16;     // dQ: S has been read by every thread (256 arrivals)
  static constexpr int kDPRead = 17;    // dP (dP^T) has been read by every thread (256)
  static constexpr int kVDone = 18;     // dK/dV: the dV product has completed
  static constexpr int kAccDone = 19, kAccFree = 20;
  static constexpr int kDrain = 21;     // both issuing threads' last products (2 arrivals)
  static constexpr int kNumBars = 22;
  static constexpr uint32_t kCtlOff = kBarOff + kNumBars * 8;
  // unit table of packed causal launches: sequence ids (bytes), then the
  // cumulative unit counts of the tile groups (ints)
  static constexpr uint32_t kTableIdsOff = kCtlOff + 16;
  static constexpr uint32_t kTableCumOff = kTableIdsOff + kTableSeqs;
  static constexpr uint32_t kSmemBytes = kTableCumOff + 4 * (kBwdTableTiles + 1);
  static_assert(kSmemBytes <= 232448, "exceeds the shared memory of one CTA");
};

// Unit table of a packed causal launch (shared memory, built once per CTA).
// Sequence b has cnt(b) units per head, unit x of it costing more as x
// grows (dQ: query tile x sees key tiles 0 .. x; dK/dV: key tile
// cnt(b) - 1 - x is seen by x + 1 query tiles).  Units are taken in groups
// of equal x, highest first: group k (x = P - 1 - k) holds unit x of every
// sequence that has one (ids[0 .. q_k), the sequences sorted by cnt,
// largest first) for every head; cum[k] units precede group k, cum[P] exist
// in all, and slots past cum[P] are empty units.
struct BwdTable {
  const uint8_t* ids;
  const int* cum;
};

// Builds the table (one warp; every lane calls it) for `batch` sequences
// (at most kTableSeqs) and P groups (at most kBwdTableTiles).
template <typename Cnt>
__device__ __forceinline__ void build_bwd_table(int batch, int P, int heads, Cnt cnt,
                                                uint8_t* ids, int* cum, int lane) {
  int np[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int b = lane + 32 * i;
    np[i] = b < batch ? cnt(b) : -1;
  }
  int rank[2] = {0, 0};
  for (int b2 = 0; b2 < batch; ++b2) {
    const int v0 = __shfl_sync(0xffffffffu, np[0], b2 & 31);
    const int v1 = __shfl_sync(0xffffffffu, np[1], b2 & 31);
    const int n2 = b2 < 32 ? v0 : v1;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int b = lane + 32 * i;
      rank[i] += (n2 > np[i] || (n2 == np[i] && b2 < b)) ? 1 : 0;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
    if (lane + 32 * i < batch) ids[rank[i]] = static_cast<uint8_t>(lane + 32 * i);
  int running = 0;
  if (lane == 0) cum[0] = 0;
  for (int k = 0; k < P; ++k) {
    const int x = P - 1 - k;
    const int c = __popc(__ballot_sync(0xffffffffu, np[0] > x)) +
                  __popc(__ballot_sync(0xffffffffu, np[1] > x));
    running += c * heads;
    if (lane == 0) cum[k + 1] = running;
  }
}

// Slot u (< num_units) of a table launch: -1 for an empty unit, else the
// sequence (*b), head (*h) and the unit's x.
__device__ __forceinline__ int bwd_table_unit(int u, int P, int heads, const BwdTable& tab,
                                              int* b, int* h) {
  if (u >= tab.cum[P]) return -1;
  int lo = 0, hi = P - 1;  // the group k with cum[k] <= u < cum[k+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab.cum[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int r = u - tab.cum[lo];
  *b = tab.ids[r / heads];
  *h = r % heads;
  return P - 1 - lo;
}

template <typename L, typename Bar>
__device__ __forceinline__ void init_barriers(Bar bar) {
  mbar_init(bar(L::kFixFull), 1);
  mbar_init(bar(L::kFixEmpty), 1);
  for (int s = 0; s < L::kStagesA; ++s) {
    mbar_init(bar(L::kAFull + s), 1);
    mbar_init(bar(L::kAEmpty + s), 1);
  }
  for (int s = 0; s < L::kStagesB; ++s) {
    mbar_init(bar(L::kBFull + s), 1);
    mbar_init(bar(L::kBEmpty + s), 1);
  }
  mbar_init(bar(L::kSDone), 1);
  mbar_init(bar(L::kDPDone), 1);
  mbar_init(bar(L::kPStored), kEwThreads);
  mbar_init(bar(L::kDSStored), kEwThreads);
  mbar_init(bar(L::kSRead), kEwThreads);
  mbar_init(bar(L::kDPRead), kEwThreads);
  mbar_init(bar(L::kVDone), 1);
  mbar_init(bar(L::kAccDone), 1);
  mbar_init(bar(L::kAccFree), kEwThreads);
  mbar_init(bar(L::kDrain), 2);
}

// Bounded wait for two phases; the fast path tests both with back-to-back
// try_waits (one round trip instead of two when both have completed).
__device__ __forceinline__ bool wait_bar2(uint32_t a, uint32_t pa, uint32_t b, uint32_t pb,
                                          const Ctl& ctl, int site) {
  uint32_t both;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%3], %4;\n\t"
      "and.pred p, p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(both)
      : "r"(a), "r"(pa), "r"(b), "r"(pb)
      : "memory");
  if (both) return true;
  return wait_bar(a, pa, ctl, site) && wait_bar(b, pb, ctl, site);
}

// Entry check of both kernels: the layout above needs a 1024-byte aligned
// shared memory base.  False (after recording FA_ERR_MISALIGNED in the
// status word) means the CTA must return at once.
__device__ __forceinline__ bool smem_base_ok(uint32_t sbase, int* status) {
  if ((sbase & 1023u) == 0) return true;
  if (threadIdx.x == 0) atomicCAS(status, 0, kStatusMisaligned | (kSiteSmemBase << 8));
  return false;
}

// Masks of the backward: key j is admissible for query i of a sequence with
// len query rows and k_len key rows when i < len, j < k_len and
// i + shift - win_left <= j <= i + shift + win_right, shift = k_len - len
// (bottom-right alignment; causal: win_right = 0).
__device__ __forceinline__ bool admissible(int i, int j, int len, int k_len, int shift, int wl,
                                           int wr) {
  return j < k_len && i < len && j <= i + shift + wr && j >= i + shift - wl;
}

// ---------------------------------------------------------------- pre-pass
// nlse2[bh][i] = -LSE * log2(e) and ndsum[bh][i] = -sum_c dO[i][c] O[i][c]
// for i < N; -inf and 0 for the padding rows up to n_pad.  d/16 threads per
// row, each with two 16-byte loads of O and two of dO in flight (a resident
// grid holds enough bytes in flight to keep HBM busy).
// (PACKED: O and dO are [total][H][d], LSE [H][total]; row i of sequence b
// is packed row cu_seqlens[b] + i, and rows past the sequence are padding.)
template <int D, bool BF16, bool PACKED>
__global__ void __launch_bounds__(256)
    fa_bwd_prepass_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                          const float* __restrict__ lse, float* __restrict__ lse2,
                          float* __restrict__ dsum, int num_bh, int N, int n_pad,
                          const BwdParams p) {
  griddep_wait();  // (programmatic dependent launch: see fa_launch.h)
  griddep_launch_dependents();
  constexpr int kTpr = D / 16;
  const long long rows = static_cast<long long>(num_bh) * n_pad;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // every lane runs the same number of iterations (the shuffles need all)
  const long long total = (rows * kTpr + 31) / 32 * 32;
  for (long long gid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       gid < total; gid += stride) {
    const long long r = gid / kTpr;
    const int part = static_cast<int>(gid % kTpr);
    const bool live = r < rows;
    const int bh = live ? static_cast<int>(r / n_pad) : 0;
    const int i = live ? static_cast<int>(r % n_pad) : n_pad;
    int row_base = 0, len = N;
    if (PACKED && live) bwd_sequence<true>(p, bh / p.H, &row_base, &len);
    const bool valid = i < len;
    // element offset of row i of head bh, and the LSE index
    const long long off =
        PACKED ? ((static_cast<long long>(row_base) + i) * p.H + bh % p.H) * D + part * 16
               : (static_cast<long long>(bh) * N + i) * D + part * 16;
    const long long lidx = PACKED ? static_cast<long long>(bh % p.H) * p.total_rows + row_base + i
                                  : static_cast<long long>(bh) * N + i;
    float acc = 0.f;
    if (valid) {
      const uint4* po = reinterpret_cast<const uint4*>(o + off);
      const uint4* pd = reinterpret_cast<const uint4*>(dout + off);
      const uint4 a0 = po[0], a1 = po[1], b0 = pd[0], b1 = pd[1];
      const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc += unpack_lo<BF16>(wa[e]) * unpack_lo<BF16>(wb[e]);
        acc += unpack_hi<BF16>(wa[e]) * unpack_hi<BF16>(wb[e]);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && part == 0) {
      // (a row without keys has LSE = -inf: P = 0 in every column)
      const float lv = valid ? lse[lidx] : -INFINITY;
      lse2[r] = lv > -INFINITY ? lv * -1.4426950408889634f : -INFINITY;
      dsum[r] = -acc;
    }
  }
}

// The elementwise work of one 64-column half of a tile, one row per thread,
// in two phases so that each overlaps a matrix product:
//   phase A (p_half):  p  = 2^(s * scale_log2 + nlse2)  (masked columns 0)
//   phase B (ds_half): ds = p * (dp + ndsum)
// (nlse2 = -LSE log2 e, ndsum = -D per column in the dK/dV kernel, per row in
// the dQ kernel).  Phase A reads the half's 64 S columns at tS + c and, when
// WRITE_P, stores P packed to 16 bits over the first 32 of them; phase B
// takes the half's 64 dP values (loaded by the caller) and stores dS packed
// into 32 columns at `tds`.  p stays in registers between the phases.  `keep(e)` is the mask of
// column c + e (only called when MASK).
template <bool BF16, bool MASK, bool WRITE_P, bool COLUMN_VECS, typename Keep>
__device__ __forceinline__ void p_half(uint32_t tS, int c, float sl2, const float* nlse2,
                                       float nlse2_row, Keep keep, float (&p)[64]) {
  uint32_t sr[64];
  tmem_ld_2x32_sync(tS + c, sr, tS + c + 32, sr + 32);
  const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const uint64_t nl = COLUMN_VECS ? *reinterpret_cast<const uint64_t*>(nlse2 + c + e)
                                    : pack_f32x2(nlse2_row, nlse2_row);
    float x0, x1;
    unpack_f32x2(
        fma_f32x2(pack_f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, nl),
        x0, x1);
    p[e] = ex2_approx(x0);
    p[e + 1] = ex2_approx(x1);
    if (MASK) {
      if (!keep(e)) p[e] = 0.f;
      if (!keep(e + 1)) p[e + 1] = 0.f;
    }
  }
  if (WRITE_P) {
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 64; e += 2) pk[e / 2] = pack2<BF16>(p[e], p[e + 1]);
    tmem_st_x32(tS + c, pk);
  }
}

template <bool BF16, bool COLUMN_VECS>
__device__ __forceinline__ void ds_half(const uint32_t (&dpr)[64], uint32_t tds, int c,
                                        const float* ndsum, float ndsum_row,
                                        const float (&p)[64]) {
  const uint64_t zero2 = pack_f32x2(0.f, 0.f);
  uint32_t dk[32];
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const uint64_t nd = COLUMN_VECS ? *reinterpret_cast<const uint64_t*>(ndsum + c + e)
                                    : pack_f32x2(ndsum_row, ndsum_row);
    const uint64_t t =
        add_f32x2(pack_f32x2(__uint_as_float(dpr[e]), __uint_as_float(dpr[e + 1])), nd);
    float d0, d1;
    unpack_f32x2(fma_f32x2(pack_f32x2(p[e], p[e + 1]), t, zero2), d0, d1);
    dk[e / 2] = pack2<BF16>(d0, d1);
  }
  tmem_st_x32(tds, dk);
}

// ---------------------------------------------------------- dK / dV kernel
struct KvUnit {
  int bkv;        // K/V head (b * H_kv + h_kv)
  int n;          // key tile
  int m_lo, nm;   // query tiles [m_lo, m_lo + nm) per query head
  int steps;      // group * nm (0: no query sees these keys)
  int row_base;   // first query row of the sequence (packed batches; else 0)
  int len;        // query rows of the sequence (N unless packed)
  int k_row_base; // first key row of the sequence (packed batches; else 0)
  int k_len;      // key rows of the sequence (N unless packed)
  bool rows;      // the tile holds key rows of the sequence (steps 0: write zeros)
};

template <bool CAUSAL, bool PACKED, bool TABLE>
__device__ __forceinline__ KvUnit decode_kv_unit(int u, const BwdParams& p,
                                                 const BwdTable& tab) {
  static_assert(!TABLE || (CAUSAL && PACKED), "the unit table orders packed causal units");
  KvUnit w;
  // (slot u of the persistent loop; dense causal launches and table
  // launches alternate the direction of their waves)
  if (CAUSAL && (!PACKED || TABLE) && u < p.num_units) u = wave_order(u, p.num_units, gridDim.x);
  if constexpr (TABLE) {
    // key tile cnt - 1 - x of head h of sequence b, cnt its key tiles
    int b = 0, h = 0;
    const int x = u < p.num_units ? bwd_table_unit(u, p.n_tiles_k, p.H_kv, tab, &b, &h) : -1;
    w.bkv = b * p.H_kv + h;
    int kb, kl;
    bwd_keys<PACKED>(p, b, &kb, &kl);
    w.n = x < 0 ? p.n_tiles_k : (kl + 127) / 128 - 1 - x;
  } else if (CAUSAL) {
    // heaviest first: the first key tiles see the most query tiles
    w.n = u / p.num_bkv;
    w.bkv = u % p.num_bkv;
  } else {
    w.bkv = u / p.n_tiles_k;
    w.n = u % p.n_tiles_k;
  }
  bwd_sequence<PACKED>(p, w.bkv / p.H_kv, &w.row_base, &w.len);
  bwd_keys<PACKED>(p, w.bkv / p.H_kv, &w.k_row_base, &w.k_len);
  w.rows = w.n * 128 < w.k_len;
  // key j is seen by queries j - shift - win_right .. j - shift + win_left
  const long long shift = static_cast<long long>(w.k_len) - w.len;
  const long long lo = static_cast<long long>(w.n) * 128 - shift - p.win_right;
  const long long hi = static_cast<long long>(w.n) * 128 + 128 - shift + p.win_left;  // exclusive
  const int row_lo = lo < 0 ? 0 : (lo > w.len ? w.len : static_cast<int>(lo));
  const int row_hi = hi > w.len ? w.len : (hi < 0 ? 0 : static_cast<int>(hi));
  w.m_lo = row_lo / 128;
  w.nm = (row_hi > row_lo && w.rows) ? (row_hi + 127) / 128 - w.m_lo : 0;
  w.steps = p.group * w.nm;
  return w;
}

// TABLE: packed causal launches that order their units from the per-CTA
// unit table (p.unit_table set).
template <int D, bool CAUSAL, bool BF16, bool PACKED, bool TABLE = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (!smem_base_ok(sbase, p.status)) return;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kCtlOff + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  constexpr uint32_t kKOff = L::kFixOff, kVOff = L::kFixOff + L::kTile;

  if (threadIdx.x == 0) {
    init_barriers<L>(bar);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_do);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // The set-up above may overlap the stream's previous kernel (programmatic
  // dependent launch); global memory is touched only after it completed.
  griddep_wait();
  griddep_launch_dependents();
  const BwdTable tab{smem + L::kTableIdsOff,
                     reinterpret_cast<const int*>(smem + L::kTableCumOff)};
  if constexpr (TABLE) {
    if (warp == 0)
      build_bwd_table(
          p.num_bkv / p.H_kv, p.n_tiles_k, p.H_kv,
          [&](int b) {
            int kb, kl;
            bwd_keys<PACKED>(p, b, &kb, &kl);
            return (kl + 127) / 128;
          },
          smem + L::kTableIdsOff, reinterpret_cast<int*>(smem + L::kTableCumOff), lane);
    __syncthreads();
  }

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t na = 0, nb = 0, units = 0;  // ring A / ring B stages filled, units
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const KvUnit w = decode_kv_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.steps == 0) continue;  // no key rows, or keys no query sees
        const uint32_t uix = units++;
        ok = wait_bar(bar(L::kFixEmpty), (uix & 1u) ^ 1u, ctl, kSiteProducerKV);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kFixFull), 2 * L::kTile);
        const int b = w.bkv / p.H_kv, hk = w.bkv % p.H_kv;
        // (packed: rows of the sequence, heads within the row)
        const int kv_head_c = PACKED ? hk : w.bkv;
        tma_load_4d(sbase + kKOff, &p.tm_k, bar(L::kFixFull), 0, w.k_row_base + w.n * 128, 0,
                    kv_head_c);
        tma_load_4d(sbase + kVOff, &p.tm_v, bar(L::kFixFull), 0, w.k_row_base + w.n * 128, 0,
                    kv_head_c);
        for (int s = 0; s < w.steps && ok; ++s) {
          const int bh = b * p.H + hk * p.group + s / w.nm;
          const int m = w.m_lo + s % w.nm;
          const int q_head_c = PACKED ? bh % p.H : bh;
          // Q into ring A
          const uint32_t sa = na % L::kStagesA;
          ok = wait_bar(bar(L::kAEmpty + sa), ((na / L::kStagesA) & 1u) ^ 1u, ctl, kSiteProducerQ);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kAFull + sa), L::kTile);
          tma_load_4d(sbase + L::kRingAOff + sa * L::kTile, &p.tm_q, bar(L::kAFull + sa), 0,
                      w.row_base + m * 128, 0, q_head_c);
          ++na;
          // dO and the stage's LSE2, D values into ring B
          const uint32_t sb = nb % L::kStagesB;
          ok = wait_bar(bar(L::kBEmpty + sb), ((nb / L::kStagesB) & 1u) ^ 1u, ctl, kSiteProducerQ);
          if (!ok) break;
          const uint32_t vec = sbase + L::kVecOff + sb * 1024;
          mbar_arrive_expect_tx(bar(L::kBFull + sb), L::kTile + 1024);
          tma_load_4d(sbase + L::kRingBOff + sb * L::kTile, &p.tm_do, bar(L::kBFull + sb), 0,
                      w.row_base + m * 128, 0, q_head_c);
          const long long voff = static_cast<long long>(bh) * p.n_pad + m * 128;
          bulk_load_1d(vec, p.lse2 + voff, 512, bar(L::kBFull + sb));
          bulk_load_1d(vec + 512, p.dsum + voff, 512, bar(L::kBFull + sb));
          ++nb;
        }
      }
      // let the copies in flight land before the CTA may exit
      for (uint32_t j = na > (uint32_t)L::kStagesA ? na - L::kStagesA : 0u; j < na; ++j)
        wait_drain(bar(L::kAFull + j % L::kStagesA), (j / L::kStagesA) & 1u, p.timeout_ns);
      for (uint32_t j = nb > (uint32_t)L::kStagesB ? nb - L::kStagesB : 0u; j < nb; ++j)
        wait_drain(bar(L::kBFull + j % L::kStagesB), (j / L::kStagesB) & 1u, p.timeout_ns);
      if (units > 0) wait_drain(bar(L::kFixFull), (units - 1) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------- S^T and dP^T products
    // Per step j: dP^T(j), then S^T(j + 1) (S^T(j) came in step j - 1 or
    // at the unit's start).
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_f16(128, 128, BF16, false);
      const uint64_t k_desc = smem_desc_sw128(sbase + kKOff, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sbase + kVOff, 16, 1024);
      // S^T = K Q^T of `step` (keys on the lanes) into region(step)
      auto issue_s = [&](uint32_t step) {
        const uint64_t q_kdesc =
            smem_desc_sw128(sbase + L::kRingAOff + (step % L::kStagesA) * L::kTile, 16, 1024);
        if constexpr (D == 128)
          mma_ss_kmajor_x8(tmem + region(step), k_desc, q_kdesc, kIdescS, 0u);
        else
          mma_ss_kmajor_x4(tmem + region(step), k_desc, q_kdesc, kIdescS, 0u);
        tc_commit(bar(L::kSDone));
      };
      uint32_t it = 0, units = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const KvUnit w = decode_kv_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.steps == 0) continue;  // no key rows, or keys no query sees
        const uint32_t uix = units++;
        ok = wait_bar(bar(L::kFixFull), uix & 1u, ctl, kSiteMmaK);
        // region(it) held the previous step's dP^T: wait until it was read
        ok = ok && (it == 0 ? wait_bar(bar(L::kAFull), 0u, ctl, kSiteMmaQ)
                            : wait_bar2(bar(L::kAFull + it % L::kStagesA),
                                        (it / L::kStagesA) & 1u, bar(L::kDPRead),
                                        (it - 1) & 1u, ctl, kSiteMmaQ));
        if (!ok) break;
        tc_fence_after_sync();
        issue_s(it);
        for (int s = 0; s < w.steps; ++s, ++it) {
          const uint32_t sb = it % L::kStagesB;
          // dP^T goes to region(it + 1), where the previous step's P^T and
          // dS^T were read by its dV and dK products (the dK product's
          // commit to its ring-A release covers both)
          ok = it == 0 ? wait_bar(bar(L::kBFull), 0u, ctl, kSiteMmaO)
                       : wait_bar2(bar(L::kBFull + sb), (it / L::kStagesB) & 1u,
                                   bar(L::kAEmpty + (it - 1) % L::kStagesA),
                                   ((it - 1) / L::kStagesA) & 1u, ctl, kSiteMmaO);
          if (!ok) break;
          tc_fence_after_sync();
          // dP^T = V dO^T
          const uint64_t do_kdesc =
              smem_desc_sw128(sbase + L::kRingBOff + sb * L::kTile, 16, 1024);
          if constexpr (D == 128)
            mma_ss_kmajor_x8(tmem + region(it + 1), v_desc, do_kdesc, kIdescS, 0u);
          else
            mma_ss_kmajor_x4(tmem + region(it + 1), v_desc, do_kdesc, kIdescS, 0u);
          tc_commit(bar(L::kDPDone));
          if (s == w.steps - 1) {
            tc_commit(bar(L::kFixEmpty));  // K and V read for the last time
          } else {
            // the next step's S^T into region(it + 1) once dP^T was read
            ok = wait_bar2(bar(L::kAFull + (it + 1) % L::kStagesA), ((it + 1) / L::kStagesA) & 1u,
                           bar(L::kDPRead), it & 1u, ctl, kSiteMmaQ);
            if (!ok) break;
            tc_fence_after_sync();
            issue_s(it + 1);
          }
        }
      }
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kGradWarp) {
    // --------------------------------------------- dV and dK products
    if (lane == 0) {
      constexpr uint32_t kIdescAcc = make_idesc_f16(128, D, BF16, true);
      uint32_t it = 0, units = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const KvUnit w = decode_kv_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.steps == 0) continue;
        const uint32_t uix = units++;
        for (int s = 0; s < w.steps; ++s, ++it) {
          const uint32_t sa = it % L::kStagesA, sb = it % L::kStagesB;
          const uint32_t x = tmem + region(it);
          // P^T stored (and dO landed: this thread reads it)
          ok = wait_bar2(bar(L::kPStored), it & 1u, bar(L::kBFull + sb), (it / L::kStagesB) & 1u,
                         ctl, kSiteMmaP);
          if (ok && s == 0 && uix > 0) {
            // the previous unit's dK, dV must have been read out
            ok = wait_bar(bar(L::kAccFree), (uix - 1) & 1u, ctl, kSiteMmaO);
          }
          if (!ok) break;
          tc_fence_after_sync();
          // dV += P^T dO (dO as the MN-major B operand; P^T of queries 0-63 at
          // x + 0, of 64-127 at x + 64; the second half of dO is 64 rows =
          // 512 descriptor units on)
          const uint64_t do_mdesc =
              smem_desc_sw128(sbase + L::kRingBOff + sb * L::kTile, 128 * 128, 1024);
          mma_ts_mnmajor_x4(tmem + kColAcc, x, do_mdesc, kIdescAcc, s > 0 ? 1u : 0u);
          mma_ts_mnmajor_x4(tmem + kColAcc, x + 64, do_mdesc + 512, kIdescAcc, 1u);
          tc_commit(bar(L::kVDone));
          ok = wait_bar2(bar(L::kDSStored), it & 1u, bar(L::kAFull + sa), (it / L::kStagesA) & 1u,
                         ctl, kSiteMmaP);
          if (!ok) break;
          tc_fence_after_sync();
          // dK += dS^T Q (dS^T of queries 0-63 at x + 32, of 64-127 at x + 96)
          const uint64_t q_mdesc =
              smem_desc_sw128(sbase + L::kRingAOff + sa * L::kTile, 128 * 128, 1024);
          mma_ts_mnmajor_x4(tmem + kColAcc + D, x + 32, q_mdesc, kIdescAcc, s > 0 ? 1u : 0u);
          mma_ts_mnmajor_x4(tmem + kColAcc + D, x + 96, q_mdesc + 512, kIdescAcc, 1u);
          // (S^T and dP^T of this step, which also read these stages, have
          // completed: dS^T was stored after dP^T's commit)
          tc_commit(bar(L::kAEmpty + sa));
          tc_commit(bar(L::kBEmpty + sb));
        }
        if (!ok) break;
        tc_commit(bar(L::kAccDone));
      }
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < kEwThreads / 32) {
    // ------------------------------------------ P^T, dS^T and the epilogue
    const int half = warp / 4;                 // query columns [64 half, +64)
    const int t = (warp % 4) * 32 + lane;      // key row within the tile == lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const int c = half * 64;
    const float sl2 = p.scale_log2;
    uint32_t it = 0, units = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      const KvUnit w = decode_kv_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
      // dV / dK rows of key tile n of K/V head bkv ([B*H_kv][N][d], or
      // packed [total_k][H_kv][d]): 32 columns of the rows of this warp
      const int j_warp = w.n * 128 + (warp % 4) * 32;  // key of lane 0's row
      auto rows_at = [&](uint16_t* base, int c0) {
        return [&, base, c0](int rl) -> uint16_t* {
          const int jr = j_warp + rl;
          if (jr >= w.k_len) return nullptr;
          const long long row = PACKED ? (static_cast<long long>(w.k_row_base) + jr) * p.H_kv +
                                             w.bkv % p.H_kv
                                       : static_cast<long long>(w.bkv) * p.N + jr;
          return base + row * D + c0;
        };
      };
      if (w.steps == 0) {
        // keys that no query sees (separate query and key lengths with a
        // window): dV = dK = 0, written without the pipeline
        if (w.rows) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t z[16] = {};
            store_rows_x32(z, lane, rows_at(half == 0 ? p.dv : p.dk, c0));
          }
        }
        continue;
      }
      const uint32_t uix = units++;
      const int j = w.n * 128 + t;  // this thread's key
      const int shift = w.k_len - w.len;  // key position of query 0
      for (int s = 0; s < w.steps; ++s, ++it) {
        const uint32_t sb = it % L::kStagesB, ph = it & 1u;
        const uint32_t x = tmem + lane_base + region(it);
        const uint32_t y = tmem + lane_base + region(it + 1);
        const int m = w.m_lo + s % w.nm;
        ok = wait_bar(bar(L::kBFull + sb), (it / L::kStagesB) & 1u, ctl, kSiteSoftmaxS);
        ok = ok && wait_bar(bar(L::kSDone), ph, ctl, kSiteSoftmaxS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        const float* nlse2 = reinterpret_cast<const float*>(smem + L::kVecOff + sb * 1024);
        const float* ndsum = nlse2 + 128;
        const int i0 = m * 128 + c;  // query of column c
        const bool need_mask = (w.n * 128 + 127 - (i0 + shift) > p.win_right) ||
                               (w.n * 128 - (i0 + 63 + shift) < -p.win_left) ||
                               (w.n * 128 + 128 > w.k_len);
        const int len = w.len, k_len = w.k_len, wl = p.win_left, wr = p.win_right;
        auto keep = [&](int e) { return admissible(i0 + e, j, len, k_len, shift, wl, wr); };
        // phase A: P^T over the first 32 of the half's S^T columns (while
        // dP^T is computed)
        float pv[64];
        if (need_mask)
          p_half<BF16, true, true, true>(x, c, sl2, nlse2, 0.f, keep, pv);
        else
          p_half<BF16, false, true, true>(x, c, sl2, nlse2, 0.f, keep, pv);
        tmem_wait_st();
        // (the previous step's dV product has completed before this P^T is
        // announced, so the issuing thread cannot miss a phase of kPStored)
        if (it > 0) {
          ok = wait_bar(bar(L::kVDone), (it - 1) & 1u, ctl, kSiteSoftmaxS);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPStored));
        // phase B: dS^T over the last 32 (while dV += P^T dO runs)
        ok = wait_bar(bar(L::kDPDone), ph, ctl, kSiteSoftmaxS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t dpr[64];
        tmem_ld_2x32_sync(y + c, dpr, y + c + 32, dpr + 32);
        tc_fence_before_sync();
        mbar_arrive(bar(L::kDPRead));
        ds_half<BF16, true>(dpr, x + c + 32, c, ndsum, 0.f, pv);
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kDSStored));
      }
      if (!ok) break;
      // ---- epilogue: warps 0-3 write dV, warps 4-7 scale * dK (this thread's key row)
      ok = wait_bar(bar(L::kAccDone), uix & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      uint16_t* const base = half == 0 ? p.dv : p.dk;
      const float mul = half == 0 ? 1.f : p.scale;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32_sync(tmem + lane_base + kColAcc + half * D + c0, r);
        uint32_t w4[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w4[e] = pack2<BF16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
        store_rows_x32(w4, lane, rows_at(base, c0));
      }
      tc_fence_before_sync();
      mbar_arrive(bar(L::kAccFree));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- dQ kernel
struct QUnit {
  int bh;         // query head
  int bkv;        // its K/V head
  int m;          // query tile
  int n0, n1;     // key tiles [n0, n1) (empty: no product to run)
  int row_base;   // first query row of the sequence (packed batches; else 0)
  int len;        // query rows of the sequence (N unless packed)
  int k_row_base; // first key row of the sequence (packed batches; else 0)
  int k_len;      // key rows of the sequence (N unless packed)
  bool rows;      // the tile holds query rows of the sequence (no keys: dQ = 0)
};

template <bool CAUSAL, bool PACKED, bool TABLE>
__device__ __forceinline__ QUnit decode_q_unit(int u, const BwdParams& p, const BwdTable& tab) {
  static_assert(!TABLE || (CAUSAL && PACKED), "the unit table orders packed causal units");
  QUnit w;
  if (CAUSAL && (!PACKED || TABLE) && u < p.num_units) u = wave_order(u, p.num_units, gridDim.x);
  if constexpr (TABLE) {
    // query tile x of head h of sequence b
    int b = 0, h = 0;
    const int x = u < p.num_units ? bwd_table_unit(u, p.n_tiles, p.H, tab, &b, &h) : -1;
    w.bh = b * p.H + h;
    w.m = x < 0 ? p.n_tiles : x;
  } else if (CAUSAL) {
    w.m = p.n_tiles - 1 - u / p.num_bh;  // heaviest first
    w.bh = u % p.num_bh;
  } else {
    w.bh = u / p.n_tiles;
    w.m = u % p.n_tiles;
  }
  w.bkv = kv_head(w.bh, p.H, p.group);
  bwd_sequence<PACKED>(p, w.bh / p.H, &w.row_base, &w.len);
  bwd_keys<PACKED>(p, w.bh / p.H, &w.k_row_base, &w.k_len);
  if (PACKED && CAUSAL && !TABLE) {
    // count the tiles from each sequence's end (its heaviest tiles first)
    w.m = (w.len + 127) / 128 - 1 - (p.n_tiles - 1 - w.m);
    if (w.m < 0) w.m = p.n_tiles;
  }
  w.rows = w.m * 128 < w.len;
  if (!w.rows) {
    w.n0 = w.n1 = 0;
    return w;
  }
  // rows m*128 .. sit at key positions m*128 + shift .. (bottom-right)
  const int shift = w.k_len - w.len;
  key_tile_range(w.m * 128 + shift, min(w.len, w.m * 128 + 128) + shift, w.k_len, p.win_left,
                 p.win_right, 128, &w.n0, &w.n1);
  return w;
}

template <int D, bool CAUSAL, bool BF16, bool PACKED, bool TABLE = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (!smem_base_ok(sbase, p.status)) return;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kCtlOff + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  constexpr uint32_t kQOff = L::kFixOff, kDOOff = L::kFixOff + L::kTile;

  if (threadIdx.x == 0) {
    init_barriers<L>(bar);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_do);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // The set-up above may overlap the stream's previous kernel (programmatic
  // dependent launch); global memory is touched only after it completed.
  griddep_wait();
  griddep_launch_dependents();
  const BwdTable tab{smem + L::kTableIdsOff,
                     reinterpret_cast<const int*>(smem + L::kTableCumOff)};
  if constexpr (TABLE) {
    if (warp == 0)
      build_bwd_table(
          p.num_bh / p.H, p.n_tiles, p.H,
          [&](int b) {
            int rb, rl;
            bwd_sequence<PACKED>(p, b, &rb, &rl);
            return (rl + 127) / 128;
          },
          smem + L::kTableIdsOff, reinterpret_cast<int*>(smem + L::kTableCumOff), lane);
    __syncthreads();
  }

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t na = 0, nb = 0, units = 0;  // ring A / ring B stages filled, units
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const QUnit w = decode_q_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.n1 == w.n0) continue;  // no query rows, or rows without keys
        const uint32_t uix = units++;
        ok = wait_bar(bar(L::kFixEmpty), (uix & 1u) ^ 1u, ctl, kSiteProducerQ);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kFixFull), 2 * L::kTile);
        // (packed: rows of the sequence, heads within the row)
        const int q_head_c = PACKED ? w.bh % p.H : w.bh;
        const int kv_head_c = PACKED ? w.bkv % p.H_kv : w.bkv;
        tma_load_4d(sbase + kQOff, &p.tm_q, bar(L::kFixFull), 0, w.row_base + w.m * 128, 0,
                    q_head_c);
        tma_load_4d(sbase + kDOOff, &p.tm_do, bar(L::kFixFull), 0, w.row_base + w.m * 128, 0,
                    q_head_c);
        for (int n = w.n0; n < w.n1 && ok; ++n) {
          // K into ring A
          const uint32_t sa = na % L::kStagesA;
          ok = wait_bar(bar(L::kAEmpty + sa), ((na / L::kStagesA) & 1u) ^ 1u, ctl,
                        kSiteProducerKV);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kAFull + sa), L::kTile);
          tma_load_4d(sbase + L::kRingAOff + sa * L::kTile, &p.tm_k, bar(L::kAFull + sa), 0,
                      w.k_row_base + n * 128, 0, kv_head_c);
          ++na;
          // V into ring B
          const uint32_t sb = nb % L::kStagesB;
          ok = wait_bar(bar(L::kBEmpty + sb), ((nb / L::kStagesB) & 1u) ^ 1u, ctl,
                        kSiteProducerKV);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kBFull + sb), L::kTile);
          tma_load_4d(sbase + L::kRingBOff + sb * L::kTile, &p.tm_v, bar(L::kBFull + sb), 0,
                      w.k_row_base + n * 128, 0, kv_head_c);
          ++nb;
        }
      }
      for (uint32_t j = na > (uint32_t)L::kStagesA ? na - L::kStagesA : 0u; j < na; ++j)
        wait_drain(bar(L::kAFull + j % L::kStagesA), (j / L::kStagesA) & 1u, p.timeout_ns);
      for (uint32_t j = nb > (uint32_t)L::kStagesB ? nb - L::kStagesB : 0u; j < nb; ++j)
        wait_drain(bar(L::kBFull + j % L::kStagesB), (j / L::kStagesB) & 1u, p.timeout_ns);
      if (units > 0) wait_drain(bar(L::kFixFull), (units - 1) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------- S and dP products
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_f16(128, 128, BF16, false);
      const uint64_t q_desc = smem_desc_sw128(sbase + kQOff, 16, 1024);
      const uint64_t do_desc = smem_desc_sw128(sbase + kDOOff, 16, 1024);
      uint32_t it = 0, units = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const QUnit w = decode_q_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.n1 == w.n0) continue;  // no query rows, or rows without keys
        const uint32_t uix = units++;
        ok = wait_bar(bar(L::kFixFull), uix & 1u, ctl, kSiteMmaQ);
        for (int n = w.n0; n < w.n1 && ok; ++n, ++it) {
          const uint32_t sa = it % L::kStagesA, sb = it % L::kStagesB;
          // S = Q K^T (queries on the lanes) over the previous step's S,
          // once every thread has read that
          ok = it == 0 ? wait_bar(bar(L::kAFull), 0u, ctl, kSiteMmaK)
                       : wait_bar2(bar(L::kAFull + sa), (it / L::kStagesA) & 1u, bar(L::kSRead),
                                   (it - 1) & 1u, ctl, kSiteMmaK);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t k_kdesc = smem_desc_sw128(sbase + L::kRingAOff + sa * L::kTile, 16, 1024);
          if constexpr (D == 128)
            mma_ss_kmajor_x8(tmem + kColS, q_desc, k_kdesc, kIdescS, 0u);
          else
            mma_ss_kmajor_x4(tmem + kColS, q_desc, k_kdesc, kIdescS, 0u);
          tc_commit(bar(L::kSDone));
          // dP = dO V^T over the previous step's dP, once read
          ok = it == 0 ? wait_bar(bar(L::kBFull), 0u, ctl, kSiteMmaV)
                       : wait_bar2(bar(L::kBFull + sb), (it / L::kStagesB) & 1u, bar(L::kDPRead),
                                   (it - 1) & 1u, ctl, kSiteMmaV);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t v_kdesc = smem_desc_sw128(sbase + L::kRingBOff + sb * L::kTile, 16, 1024);
          if constexpr (D == 128)
            mma_ss_kmajor_x8(tmem + kColDP, do_desc, v_kdesc, kIdescS, 0u);
          else
            mma_ss_kmajor_x4(tmem + kColDP, do_desc, v_kdesc, kIdescS, 0u);
          tc_commit(bar(L::kDPDone));
          tc_commit(bar(L::kBEmpty + sb));                     // V read for the last time
          if (n == w.n1 - 1) tc_commit(bar(L::kFixEmpty));  // Q and dO too
        }
      }
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kGradWarp) {
    // ------------------------------------------------------- dQ products
    if (lane == 0) {
      constexpr uint32_t kIdescAcc = make_idesc_f16(128, D, BF16, true);
      uint32_t it = 0, units = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const QUnit w = decode_q_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.n1 == w.n0) continue;
        const uint32_t uix = units++;
        for (int n = w.n0; n < w.n1; ++n, ++it) {
          const uint32_t sa = it % L::kStagesA;
          // dS stored (and K landed: this thread reads it)
          ok = wait_bar2(bar(L::kDSStored), it & 1u, bar(L::kAFull + sa), (it / L::kStagesA) & 1u,
                         ctl, kSiteMmaP);
          if (ok && n == w.n0 && uix > 0)
            ok = wait_bar(bar(L::kAccFree), (uix - 1) & 1u, ctl, kSiteMmaO);
          if (!ok) break;
          tc_fence_after_sync();
          // dQ += dS K (dS from its own columns, K as the MN-major B operand)
          const uint64_t k_mdesc =
              smem_desc_sw128(sbase + L::kRingAOff + sa * L::kTile, 128 * 128, 1024);
          mma_ts_mnmajor_x4(tmem + kColAcc, tmem + kColDS, k_mdesc, kIdescAcc,
                            n > w.n0 ? 1u : 0u);
          mma_ts_mnmajor_x4(tmem + kColAcc, tmem + kColDS + 64, k_mdesc + 512, kIdescAcc, 1u);
          // (S of this step, which also read this stage, has completed: dS
          // was stored after dP's commit)
          tc_commit(bar(L::kAEmpty + sa));
        }
        if (!ok) break;
        tc_commit(bar(L::kAccDone));
      }
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < kEwThreads / 32) {
    // ------------------------------------------------ dS and the epilogue
    const int half = warp / 4;              // key columns [64 half, +64)
    const int t = (warp % 4) * 32 + lane;   // query row within the tile == lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tDP = tmem + lane_base + kColDP;
    const int c = half * 64;
    const float sl2 = p.scale_log2;
    uint32_t it = 0, units = 0;
    bool ok = true;
    // the first unit at or after u with query rows (num_units: none)
    auto next_unit = [&](int u, QUnit& w) -> int {
      for (; u < p.num_units; u += gridDim.x) {
        w = decode_q_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        if (w.rows) break;
      }
      return u;
    };
    // this thread's -LSE2 and -D of unit w
    auto row_values = [&](const QUnit& w, float& nl, float& nd) {
      const long long vrow = static_cast<long long>(w.bh) * p.n_pad + w.m * 128 + t;
      nl = p.lse2[vrow];
      nd = p.dsum[vrow];
    };
    QUnit w{};
    int u = next_unit(blockIdx.x, w);
    float nlse2 = 0.f, ndsum = 0.f;
    if (u < p.num_units) row_values(w, nlse2, ndsum);
    while (u < p.num_units && ok) {
      // dQ rows of query tile m of head bh ([B*H][N][d], or packed
      // [total][H][d]): 32 columns of the rows of this warp
      const int i_warp = w.m * 128 + (warp % 4) * 32;  // query of lane 0's row
      auto rows_at = [&](int c0) {
        return [&, c0](int rl) -> uint16_t* {
          const int ir = i_warp + rl;
          if (ir >= w.len) return nullptr;
          const long long qrow = PACKED
                                     ? (static_cast<long long>(w.row_base) + ir) * p.H + w.bh % p.H
                                     : static_cast<long long>(w.bh) * p.N + ir;
          return p.dq + qrow * D + half * (D / 2) + c0;
        };
      };
      if (w.n1 == w.n0) {
        // query rows that see no key (separate query and key lengths): dQ = 0
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          uint32_t z[16] = {};
          store_rows_x32(z, lane, rows_at(c0));
        }
        QUnit wn{};
        const int un = next_unit(u + static_cast<int>(gridDim.x), wn);
        if (un < p.num_units) row_values(wn, nlse2, ndsum);
        u = un;
        w = wn;
        continue;
      }
      const uint32_t uix = units++;
      const int i = w.m * 128 + t;
      const int shift = w.k_len - w.len;  // key position of query 0
      const int row_end = min(w.len, w.m * 128 + 128);
      for (int n = w.n0; n < w.n1; ++n, ++it) {
        const uint32_t ph = it & 1u;
        ok = wait_bar(bar(L::kSDone), ph, ctl, kSiteSoftmaxS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        const int kbase = n * 128 + c;  // key of column c
        const bool need_mask = (kbase + 64 > w.k_len) ||
                               (kbase + 63 > w.m * 128 + shift + p.win_right) ||
                               (kbase < row_end - 1 + shift - p.win_left);
        const int len = w.len, k_len = w.k_len, wl = p.win_left, wr = p.win_right;
        auto keep = [&](int e) { return admissible(i, kbase + e, len, k_len, shift, wl, wr); };
        // phase A: P (S may be overwritten once every thread has read it)
        float pv[64];
        if (need_mask)
          p_half<BF16, true, false, false>(tS, c, sl2, nullptr, nlse2, keep, pv);
        else
          p_half<BF16, false, false, false>(tS, c, sl2, nullptr, nlse2, keep, pv);
        tc_fence_before_sync();
        mbar_arrive(bar(L::kSRead));
        // phase B: dS into its own columns
        ok = wait_bar(bar(L::kDPDone), ph, ctl, kSiteSoftmaxS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        uint32_t dpr[64];
        tmem_ld_2x32_sync(tDP + c, dpr, tDP + c + 32, dpr + 32);
        tc_fence_before_sync();
        mbar_arrive(bar(L::kDPRead));
        // the previous step's dQ product read dS: wait for its commit (also
        // keeps this store from running ahead of the dQ issuer)
        if (it > 0) {
          ok = wait_bar(bar(L::kAEmpty + (it - 1) % L::kStagesA), ((it - 1) / L::kStagesA) & 1u,
                        ctl, kSiteSoftmaxS);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after_sync();
        }
        ds_half<BF16, false>(dpr, tmem + lane_base + kColDS + c, c, nullptr, ndsum, pv);
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kDSStored));
      }
      if (!ok) break;
      // the next unit's row values, loaded before this unit's epilogue
      QUnit wn{};
      const int un = next_unit(u + static_cast<int>(gridDim.x), wn);
      float nl_next = 0.f, nd_next = 0.f;
      if (un < p.num_units) row_values(wn, nl_next, nd_next);
      // ---- epilogue: scale * dQ, columns [D/2 half, +D/2) of this thread's row
      ok = wait_bar(bar(L::kAccDone), uix & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32_sync(tmem + lane_base + kColAcc + half * (D / 2) + c0, r);
        uint32_t w4[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w4[e] = pack2<BF16>(__uint_as_float(r[2 * e]) * p.scale,
                              __uint_as_float(r[2 * e + 1]) * p.scale);
        store_rows_x32(w4, lane, rows_at(c0));
      }
      tc_fence_before_sync();
      mbar_arrive(bar(L::kAccFree));
      u = un;
      w = wn;
      nlse2 = nl_next;
      ndsum = nd_next;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace bwd
}  // namespace fa
