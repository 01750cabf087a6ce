// fa_fwd_kernel.cuh -- persistent, warp-specialised attention forward kernel
// for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
//
// What it computes: for each (b,h) and query row i,
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j   and   LSE_i (natural log),
// with keys j > i masked when causal.  The algorithm is the FlashAttention-2
// forward of LeetCUDA "flash_attn_mma_tiling_qk.cu" (tile Q by rows, stream
// K/V tiles, online row max / row sum, rescale the running output by
// exp(m_old - m_new) -- not its inverse --, divide by the row sum at the end),
// laid out the way the Hopper pages of flash-attention
// ("hopper/flash_fwd_kernel.h": a TMA producer warp, K and V pipelines,
// persistent work-tile loop, O stored with the row LSE) arrange it, and
// re-designed for Blackwell's tensor memory:
//
//   warps 0-3  softmax warpgroup 0   (query tile 0, one row per thread)
//   warps 4-7  softmax warpgroup 1   (query tile 1)
//   warp  8    TMA producer          (Q tiles, then K_j / V_j into a ring)
//   warp  9    MMA issuer            (S_g = Q_g K_j^T, O_g += P_g V_j)
//   warp  10   O store               (TMA store of each finished O tile)
//   warp  11   spare (completes the third warpgroup, so that register
//              budgets can move between warpgroups with setmaxnreg: the
//              softmax warpgroups run with 216 registers, the third with 72)
//
// All synchronisation between roles goes through mbarriers with bounded
// waits (no bar.sync among roles), so a stalled stage can always be
// abandoned without leaving another one blocked.
//
// MMA issue order.  The MMAs are issued as alternating per-tile groups
//   [P_0(j-1) V_(j-1), Q_0 K_j^T]  [P_1(j-1) V_(j-1), Q_1 K_j^T]  ...
// over the stream of K/V tiles j (continuing across work units), so that
// each tile's softmax runs while the other tile's two MMAs execute.  P_g is
// handed over in two 64-key halves (one mbarrier each), so the first half of
// P_g V starts while the softmax still computes the second.  P_g lives
// in S_g's tensor-memory columns, so Q_g K_j^T overwrites the A operand of
// P_g(j-1) V.  The PTX ISA orders two tcgen05.mma of one thread only when
// they share the accumulator and shape (its list of implicitly pipelined
// tcgen05 instruction pairs); these two have different accumulators (O_g,
// S_g), so the issuer waits for the commit of the last P_g V (barrier
// ODone_g) before it issues Q_g K_j^T.
//
// K/V stream.  K(j) and V(j) go to ring slots 2(j % h) and 2(j % h) + 1
// (h = STAGES / 2).  One "full" barrier per step, B(j), completes when the
// two tiles step j first reads have landed, V(j-1) and K(j), so the MMA
// issuer waits once per step; one commit per step releases K(j) and V(j-1)
// for the producer (release group j % h).
//
// Row maximum.  A softmax thread loads its row of S with tcgen05.ld.red.max,
// which also returns the maximum of the loaded columns (unmasked tiles use
// it; masked tiles take the maximum over the kept columns).
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128)    S_0 (scores of tile 0); P_0 (16-bit, packed in pairs) is
//              written over its first 64 columns after the row is read
//   [128,256)  S_1 / P_1
//   [256,256+D) O_0,  [256+D, 256+2D) O_1   (running outputs)
//
// Shared memory (1024-byte aligned, 128-byte TMA swizzle everywhere):
//   Q_0, Q_1       [D/64][128 rows][64]   one tile each
//   K/V ring       STAGES slots of [D/64][128 keys][64]
//   O staging      one tile, shared by the two query tiles in turn (TMA
//                  store source; tile 1 of a causal unit and the tiles of
//                  packed batches are stored by the softmax threads instead)
//   mbarriers
//
// Online softmax in the log2 domain (scale folded into scale*log2 e, as the
// Hopper pages do with softmax_scale_log2): x = s*scale*log2e, p = 2^(x - m).
// The running maximum m is only raised when a tile's maximum exceeds it by
// more than kRescaleThreshold (2^8): until then p may exceed 1 (at most 256)
// and O and the row sum keep their old reference, so the output rescale in
// tensor memory is rare (lazy rescaling).
//
// Every mbarrier wait is bounded (globaltimer); on timeout the kernel records
// a status code, raises a CTA-wide abort flag, lets in-flight copies and MMAs
// land, frees tensor memory and returns.  Nothing traps.
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

constexpr int kNumThreads = 384;
constexpr uint32_t kSoftmaxRegs = 216;  // per thread, warpgroups 0 and 1
constexpr uint32_t kControlRegs = 72;   // per thread, warpgroup 2
// Launch budget: 384 threads x 168 registers; 2*128*216 + 128*72 fits in it.
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kNumThreads * 168,
              "register split exceeds the launch budget");
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStoreWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kFp8Threshold = 2.0f;      // log2 units (FP8 P)
constexpr float kFp8POffset = 6.0f;        // log2 units (FP8 P)

// FP8: E4M3 Q, K and V^T tiles (one byte per element, 128-byte rows), so
// twice the ring slots; the output stays 16-bit.
template <int D, bool FP8 = false>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!FP8 || D == 128, "FP8 tiles are 128-byte rows");
  static constexpr uint32_t kTileBytes = kBlockM * D * (FP8 ? 1 : 2);  // Q, K or V tile
  static constexpr uint32_t kOTileBytes = kBlockM * D * 2;             // 16-bit O tile
  static constexpr int kStages = FP8 ? 8 : (D == 64) ? 6 : 4;
  static_assert(kStages % 2 == 0, "K and V share the ring in pairs");
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kQOff + 2 * kTileBytes;
  static constexpr uint32_t kStageOff = kKVOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kStageOff + kOTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 2;
  // step barriers: B(j) = kKVFull + j % (kStages / 2) completes when the
  // two tiles K/V step j first reads have landed: V(j-1) and K(j)
  static constexpr int kKVFull = 4;
  // release groups: the commit of K/V step j frees K(j) and V(j-1) and
  // arrives on group j % (kStages / 2)
  static constexpr int kKVEmpty = kKVFull + kStages;
  static constexpr int kSFull = kKVEmpty + kStages / 2;
  // P_g ready, per 64-key half: kPFull + 2 g + half
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kODone = kPFull + 4;
  static constexpr int kDrain = kODone + 2;
  static constexpr int kStageFull = kDrain + 1;       // O tile written to staging
  static constexpr int kStageEmpty = kStageFull + 1;  // staging read by the store
  static constexpr int kNumBars = kStageEmpty + 1;
  static constexpr uint32_t kCtlOff = kBarOff + kNumBars * 8;
  // unit table of packed causal launches: sequence ids (bytes), then the
  // cumulative unit counts of the pair groups (ints)
  static constexpr uint32_t kTableIdsOff = kCtlOff + 16;
  static constexpr uint32_t kTableCumOff = kTableIdsOff + kTableSeqs;
  static constexpr uint32_t kUsedBytes = kTableCumOff + 4 * (kTablePairs + 1);
  static constexpr uint32_t kSmemBytes = kUsedBytes + 1024;  // alignment slack
  static_assert(kSmemBytes <= 232448, "exceeds the shared memory of one CTA");
  // tensor-memory columns of S_g / P_g and of O_g
  __device__ static constexpr uint32_t s_col(int g) { return g * 128u; }
  __device__ static constexpr uint32_t o_col(int g) { return 256u + g * D; }
};

// Unit table of a packed causal launch (shared memory, built once per CTA).
// A unit's cost grows with its pair index from the sequence start (its rows
// see the keys up to their own position), so units are taken in groups of
// equal pair index, highest first: group k holds pair P-1-k of every
// sequence that has it (ids[0 .. q_k), the sequences sorted by their pair
// count, longest first) and every problem head, cum[k] units precede it and
// cum[P] units exist in all; slots past cum[P] are empty units.
struct UnitTable {
  const uint8_t* ids;
  const int* cum;
};

// Builds the table (one warp; every lane calls it).  Sequences beyond the
// batch count have no pairs.
__device__ __forceinline__ void build_unit_table(const FaParams& p, uint8_t* ids, int* cum,
                                                 int lane) {
  const int heads = p.H >> p.gqa_log2;
  const int batch = p.num_bh / heads;
  const int unit_pos = kRowsPerUnit >> p.gqa_log2;
  int np[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int b = lane + 32 * i;
    np[i] = -1;
    if (b < batch) {
      int first, len;
      packed_rows(p.cu_seqlens, p.seqused_q, b, p.total_rows, p.N, &first, &len);
      np[i] = (len + unit_pos - 1) / unit_pos;
    }
  }
  // rank of each sequence: more pairs first, then lower index
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
  // group k = pair P-1-k: the sequences with more than P-1-k pairs, times
  // the heads
  int running = 0;
  if (lane == 0) cum[0] = 0;
  for (int k = 0; k < p.num_pairs; ++k) {
    const int pr = p.num_pairs - 1 - k;
    const int cnt = __popc(__ballot_sync(0xffffffffu, np[0] > pr)) +
                    __popc(__ballot_sync(0xffffffffu, np[1] > pr));
    running += cnt * heads;
    if (lane == 0) cum[k + 1] = running;
  }
}

// One work unit: 256 query rows of one (b,h) = two 128-row query tiles.
// Tile g visits K/V tiles [n0[g], n1[g]) (empty when n1 == n0); the unit
// streams K/V tiles [n_beg, n_end), the union of the two ranges.
struct Unit {
  int bh;       // query head (b*H + h)
  SeqView sv;   // its rows and tensor-map heads
  int row0[2];  // first query row of each tile (within the sequence)
  int n0[2], n1[2];
  int n_beg, n_end;
};

// Slot u of the persistent loop (CTA c takes slots c, c + grid, ...) runs
// unit u, or for dense causal launches unit wave_order(u).
// Units [0, num_pair_units) are query-tile pairs.  When the pairs do not
// fill the last wave of CTAs evenly, the pairs of that partial wave are split
// instead into single-tile units (tile 0 only), one per CTA, which halves
// the length of the last wave.
template <bool CAUSAL, bool PACKED, bool TABLE>
__device__ __forceinline__ Unit decode_unit(int u, const FaParams& p, const UnitTable& tab) {
  static_assert(!TABLE || (CAUSAL && PACKED), "the unit table orders packed causal units");
  Unit w;
  if (CAUSAL && (!PACKED || TABLE) && u < p.num_units) u = wave_order(u, p.num_units, gridDim.x);
  int split = 0;
  if (p.num_splits > 1) {
    split = u % p.num_splits;
    u /= p.num_splits;
  }
  int pu = u, single = -1;  // pair-unit index; tile of a single-tile unit
  if (u >= p.num_pair_units) {
    pu = p.num_pair_units + (u - p.num_pair_units) / 2;
    single = (u - p.num_pair_units) % 2;
  }
  int pair;
  if constexpr (TABLE) {
    // the pu-th unit of the table's order (pu < num_units)
    const int heads = p.H >> p.gqa_log2;
    if (pu >= tab.cum[p.num_pairs]) {
      w.bh = 0;
      pair = p.num_pairs;  // past the units that exist: an empty unit
    } else {
      int lo = 0, hi = p.num_pairs - 1;  // the group k with cum[k] <= pu < cum[k+1]
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab.cum[mid] <= pu)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int r = pu - tab.cum[lo];
      w.bh = tab.ids[r / heads] * heads + r % heads;
      pair = p.num_pairs - 1 - lo;
    }
  } else if (CAUSAL) {
    // heaviest first: the last query pairs of every head come first
    pair = p.num_pairs - 1 - pu / p.num_bh;
    w.bh = pu % p.num_bh;
  } else {
    // consecutive units share a head (and heads sharing K/V are adjacent),
    // so K/V stay hot in L2
    w.bh = pu / p.num_pairs;
    pair = pu % p.num_pairs;
  }
  w.sv = seq_view<PACKED>(p, w.bh, split * p.num_bh + w.bh);
  const int len = w.sv.len;
  // query positions per tile and per unit (fewer with grouped-query packing,
  // where a tile row is a (position, head) pair)
  const int pk = PACKED ? p.gqa_log2 : 0;
  const int tile_pos = kBlockM >> pk, unit_pos = kRowsPerUnit >> pk;
  if (PACKED && CAUSAL && !TABLE) {
    // sequences differ in length: count the pairs from each sequence's end,
    // so that every sequence's heaviest (last) pairs come first
    pair = (len + unit_pos - 1) / unit_pos - 1 - (p.num_pairs - 1 - pair);
    if (pair < 0) pair = p.num_pairs;  // no such pair: an empty unit
  }
  w.n_beg = 0x7fffffff;
  w.n_end = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    // a single-tile unit carries its tile in slot 0
    const int r0 = (single < 0) ? pair * unit_pos + g * tile_pos
                                : pair * unit_pos + single * tile_pos;
    w.row0[g] = r0;
    if (r0 >= len || (single >= 0 && g == 1)) {
      w.n0[g] = w.n1[g] = 0;
    } else {
      // positions r0 .. sit at key positions r0 + k_off .. (bottom-right
      // alignment)
      key_tile_range(r0 + w.sv.k_off, min(len, r0 + tile_pos) + w.sv.k_off, w.sv.k_len,
                     p.win_left, p.win_right, kBlockN, &w.n0[g], &w.n1[g]);
      if (p.num_splits > 1) {
        clip_to_split(split, p.split_tiles, &w.n0[g], &w.n1[g]);
      } else if (w.n1[g] == w.n0[g]) {
        // no row of the tile has a key (fewer keys than queries, or a
        // window past the keys): one fully masked key tile gives its rows
        // O = 0 and LSE = -inf through the ordinary path
        w.n0[g] = 0;
        w.n1[g] = 1;
      }
    }
    if (w.n1[g] > w.n0[g]) {
      w.n_beg = min(w.n_beg, w.n0[g]);
      w.n_end = max(w.n_end, w.n1[g]);
    }
  }
  if (w.n_end == 0) w.n_beg = 0;  // nothing to stream
  return w;
}

// Whether tile g of unit w goes through the staging tile and a TMA store:
// the dense layout's tiles with keys, but for tile 1 of a causal unit.
// That tile and the tiles of packed batches are stored from the softmax
// threads (a coalesced row store per warp), so that a causal unit's tile 1
// does not wait for tile 0's TMA store to free the one staging tile (both
// measured faster; for units whose two tiles end together, staging both
// measured faster).
template <bool CAUSAL, bool PACKED>
__device__ __forceinline__ bool staged_tile(const FaParams& p, const Unit& w, int g) {
  (void)p;
  if (PACKED || (CAUSAL && g == 1)) return false;
  return g ? (w.n1[1] > w.n0[1]) : (w.n1[0] > w.n0[0]);
}

// Maximum of a row of scores: four independent chains.
__device__ __forceinline__ float tile_max(const float (&s)[kBlockN]) {
  float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
  for (int c = 4; c < kBlockN; c += 4) {
    mx0 = fmaxf(mx0, s[c]);
    mx1 = fmaxf(mx1, s[c + 1]);
    mx2 = fmaxf(mx2, s[c + 2]);
    mx3 = fmaxf(mx3, s[c + 3]);
  }
  return fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
}

// p = 2^(s*scale*log2e - m) for one row of a tile: one packed FMA per pair,
// then the exponentials; P (16-bit, packed in pairs) goes to tensor memory
// at tS, over the first half of the row's scores.  Returns the row sum of p
// (kept as two packed partial sums).
// Columns [C_BEGIN, C_END) only, so that P can be handed over in halves.
template <bool BF16, int C_BEGIN = 0, int C_END = kBlockN>
__device__ __forceinline__ float exp_tile_to_tmem(const float (&s)[kBlockN], float scale_log2,
                                                  float m, uint32_t tS) {
  const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
  const uint64_t neg_m2 = pack_f32x2(-m, -m);
  uint64_t acc_a = pack_f32x2(0.f, 0.f), acc_b = acc_a;
#pragma unroll
  for (int c0 = C_BEGIN; c0 < C_END; c0 += 32) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float x0, x1;
      unpack_f32x2(fma_f32x2(pack_f32x2(s[c0 + 2 * e], s[c0 + 2 * e + 1]), scale2, neg_m2), x0,
                   x1);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      if (e & 1)
        acc_b = add_f32x2(acc_b, pack_f32x2(p0, p1));
      else
        acc_a = add_f32x2(acc_a, pack_f32x2(p0, p1));
      pk[e] = pack2<BF16>(p0, p1);
    }
    tmem_st_x16(tS + c0 / 2, pk);
  }
  float a0, a1;
  unpack_f32x2(add_f32x2(acc_a, acc_b), a0, a1);
  return a0 + a1;
}

// FP8: Q, K E4M3 and V^T E4M3 ([heads][D][keys], see the launcher) with the
// products in kind::f8f6f4; P goes to tensor memory as E4M3 scaled by
// 2^kFp8POffset; O (16-bit, BF16 must be true) is multiplied by the V
// descale in the epilogue.
// FP8 form of exp_tile_to_tmem: p = 2^(s*scale*log2e - m) (m includes the
// P offset), packed four per 32-bit column as E4M3 into tensor memory at tS
// (32 columns).  Returns the row sum of the unrounded p.
__device__ __forceinline__ float exp_tile_to_tmem_e4m3(const float (&s)[kBlockN],
                                                       float scale_log2, float m, uint32_t tS) {
  const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
  const uint64_t neg_m2 = pack_f32x2(-m, -m);
  uint64_t acc_a = pack_f32x2(0.f, 0.f), acc_b = acc_a;
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < kBlockN; c += 4) {
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      float x0, x1;
      unpack_f32x2(fma_f32x2(pack_f32x2(s[c + e], s[c + e + 1]), scale2, neg_m2), x0, x1);
      p[e] = ex2_approx(x0);
      p[e + 1] = ex2_approx(x1);
    }
    acc_a = add_f32x2(acc_a, pack_f32x2(p[0], p[1]));
    acc_b = add_f32x2(acc_b, pack_f32x2(p[2], p[3]));
    pk[c / 4] = pack4_e4m3(p[0], p[1], p[2], p[3]);
  }
  tmem_st_x32(tS, pk);
  float a0, a1;
  unpack_f32x2(add_f32x2(acc_a, acc_b), a0, a1);
  return a0 + a1;
}

// TABLE: packed causal launches that take their units from the per-CTA unit
// table (p.unit_table set).
template <int D, bool CAUSAL, bool BF16, bool PACKED, bool FP8 = false, bool TABLE = false>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FaParams p) {
  using L = Layout<D, FP8>;
  static_assert(!FP8 || (BF16 && !PACKED), "FP8 runs the [B,H,N,d] layout with a bf16 output");
  // P = 2^(x - m + offset) stays below 2^(threshold + offset) <= 256 < 448,
  // the largest E4M3 value; the offset keeps small probabilities above the
  // E4M3 subnormal floor.
  constexpr float kThreshold = FP8 ? kFp8Threshold : kRescaleThreshold;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kCtlOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kCtlOff + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar(L::kQFull + g), 1);
      mbar_init(bar(L::kQEmpty + g), 1);
      mbar_init(bar(L::kSFull + g), 1);
      mbar_init(bar(L::kPFull + 2 * g), 128);
      mbar_init(bar(L::kPFull + 2 * g + 1), 128);
      mbar_init(bar(L::kODone + g), 1);
    }
    for (int s = 0; s < L::kStages / 2; ++s) mbar_init(bar(L::kKVFull + s), 1);
    for (int s = 0; s < L::kStages / 2; ++s) mbar_init(bar(L::kKVEmpty + s), 1);
    mbar_init(bar(L::kDrain), 1);
    mbar_init(bar(L::kStageFull), 128);
    mbar_init(bar(L::kStageEmpty), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_o);
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
  const UnitTable tab{smem + L::kTableIdsOff, reinterpret_cast<const int*>(smem + L::kTableCumOff)};
  if constexpr (TABLE) {
    if (warp == 0)
      build_unit_table(p, smem + L::kTableIdsOff, reinterpret_cast<int*>(smem + L::kTableCumOff),
                       lane);
    __syncthreads();
  }

  // Each role changes its register budget inside its own branch, so that no
  // code is reachable under two different budgets.
  if (warp == kProducerWarp) {
    regs_decrease<kControlRegs>();
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t kv_it = 0, q_it[2] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
        for (int g = 0; g < 2 && ok; ++g) {
          if (w.n1[g] == w.n0[g]) continue;
          ok = wait_bar(bar(L::kQEmpty + g), (q_it[g] & 1u) ^ 1u, ctl, kSiteProducerQ);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kQFull + g), L::kTileBytes);
          if (PACKED && p.gqa_log2)  // {64, heads of the group, positions, d/64, K/V head}
            tma_load_5d(sbase + L::kQOff + g * L::kTileBytes, &p.tm_q, bar(L::kQFull + g), 0, 0,
                        w.sv.row_base + w.row0[g], 0, w.sv.kv_head);
          else
            tma_load_4d(sbase + L::kQOff + g * L::kTileBytes, &p.tm_q, bar(L::kQFull + g), 0,
                        w.sv.row_base + w.row0[g], 0, w.sv.q_head);
          ++q_it[g];
        }
        for (int n = w.n_beg; n < w.n_end && ok; ++n) {
          for (int kv = 0; kv < 2; ++kv) {
            // K(j) goes to slot 2(j % h), V(j) to slot 2(j % h) + 1
            const uint32_t slot = kv_it % L::kStages;
            {
              // The slot's previous tenant, K(j-h) or V(j-h), was released by
              // the one commit of step j-h or j-h+1 (release group step % h).
              constexpr int h = L::kStages / 2;
              const int j = static_cast<int>(kv_it / 2);
              if (j >= h) {
                const int rel = kv ? j - h + 1 : j - h;
                ok = wait_bar(bar(L::kKVEmpty + rel % h), (rel / h) & 1, ctl, kSiteProducerKV);
              }
            }
            if (!ok) break;
            // K(j) and V(j - 1) complete step barrier B(j), V(j) completes
            // B(j + 1); B(j) is armed (both tiles) as K(j) goes out, which
            // may be after V(j - 1) has landed (the transaction count then
            // runs negative until the arming).  B(0) has K(0) alone.
            // A barrier's next phase may only receive copies once its previous
            // one completed: for V(j) with j >= h and K(j) with j >= h the slot
            // release above implies it (the MMA waited B(j + 1 - h), B(j - h)
            // before that release); V(h - 1), the first to reuse B(0)'s
            // object, waits for B(0) itself.
            constexpr int h = L::kStages / 2;
            const int j = static_cast<int>(kv_it / 2);
            const uint32_t sb = bar(L::kKVFull + (j + kv) % h);
            if (kv && j == h - 1) {
              ok = wait_bar(bar(L::kKVFull), 0u, ctl, kSiteProducerKV);
              if (!ok) break;
            }
            if (!kv) mbar_arrive_expect_tx(sb, (j == 0 ? 1u : 2u) * L::kTileBytes);
            if (FP8 && kv)  // V^T: all d rows of key block n
              tma_load_4d(sbase + L::kKVOff + slot * L::kTileBytes, &p.tm_v, sb, 0, 0, n,
                          w.sv.kv_head);
            else
              tma_load_4d(sbase + L::kKVOff + slot * L::kTileBytes, kv ? &p.tm_v : &p.tm_k,
                          sb, 0, w.sv.k_row_base + n * kBlockN, 0, w.sv.kv_head);
            ++kv_it;
          }
        }
      }
      constexpr uint32_t h = L::kStages / 2;
      const uint32_t steps = kv_it / 2;  // K/V steps with both tiles issued
      if (kv_it > 0) {
        // The stream's last V(steps - 1) completes B(steps) alone: arm it
        // (an odd count means K(steps) went out, and armed it, last).  A
        // parity wait cannot tell a phase from the one two later, so B(steps)
        // may only complete once the MMA issuer has waited for the object's
        // previous phase, B(steps - h).  For steps > h the release of
        // V(steps - 1 - h)'s slot, waited for above, came after that wait.
        // For steps == h, V(h - 1) went into a fresh slot and K(h), which
        // would otherwise hold B(h) back until slot 0 is released, does not
        // exist: wait here for the release of step 0, which the issuer
        // commits after waiting for B(0).
        if (kv_it % 2 == 0) {
          bool armed_ok = true;
          if (steps == h) armed_ok = wait_bar(bar(L::kKVEmpty), 0u, ctl, kSiteProducerKV);
          if (armed_ok) mbar_arrive_expect_tx(bar(L::kKVFull + steps % h), L::kTileBytes);
        }
        // Let every copy this warp issued land before the CTA may exit:
        // those of the last h step barriers B(steps + 1 - h) .. B(steps),
        // h distinct objects (an older phase of the same object could not be
        // told apart by its parity once the newer one has completed).  Older
        // copies have landed: K(steps - h) before the slot of the last V was
        // released (the MMA waited B(steps - h)), K(0) before V(h - 1) went
        // out.
        const uint32_t first = steps + 1 > h ? steps + 1 - h : 0u;
        for (uint32_t jj = first; jj <= steps; ++jj)
          wait_drain(bar(L::kKVFull + jj % h), (jj / h) & 1u, p.timeout_ns);
      }
      for (int g = 0; g < 2; ++g)
        if (q_it[g] > 0) wait_drain(bar(L::kQFull + g), (q_it[g] - 1) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    regs_decrease<kControlRegs>();
    // ---------------------------------------------------------------- MMA
    // The issuing thread does as little as possible between MMA groups: the
    // tensor pipe holds only a couple of queued MMAs.
    if (lane == 0) {
      // (FP8: the E4M3 format code is 0, B of the P V product K-major V^T)
      constexpr uint32_t kIdescS = make_idesc_f16(kBlockM, kBlockN, FP8 ? false : BF16, false);
      constexpr uint32_t kIdescO = make_idesc_f16(kBlockM, D, FP8 ? false : BF16, !FP8);
      constexpr uint32_t kSlotStep = L::kTileBytes >> 4;  // descriptor units
      // Descriptors of slot 0 / query tile 0; other slots and tiles are fixed
      // offsets in the 14-bit start-address field (no carry: smem < 256 KB).
      const uint64_t q_desc0 = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sbase + L::kKVOff, 16, 1024);
      // V is MN-major (d contiguous): 64-wide d blocks 128 keys apart (LBO),
      // 8-key groups 1024 B apart (SBO).
      const uint64_t v_desc0 = FP8 ? smem_desc_sw128(sbase + L::kKVOff, 16, 1024)
                                   : smem_desc_sw128(sbase + L::kKVOff, kBlockN * 128, 1024);
      uint32_t slot = 0;  // next K/V ring position
      uint32_t step = 0;             // K/V stream step (for the release groups)
      uint32_t q_par[2] = {0, 0}, p_par[2] = {0, 0}, o_cnt[2] = {0, 0};
      // P_g V products issued / known complete (ODone_g phases waited for)
      uint32_t o_seen[2] = {0, 0};
      bool ok = true;
      // Step j of the K/V stream is (unit u, tile n); prev_* describe step
      // j-1, whose P V products are issued in step j.
      bool prev_valid = false;
      bool prev_active[2] = {false, false}, prev_acc[2] = {false, false};
      uint32_t prev_vslot = 0;
      int u = blockIdx.x;
      Unit w = decode_unit<CAUSAL, PACKED, TABLE>(u < p.num_units ? u : 0, p, tab);
      // units without K/V tiles (a split-off tile past N) stream nothing
      while (u < p.num_units && w.n_end == w.n_beg) {
        u += gridDim.x;
        if (u < p.num_units) w = decode_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
      }
      int n = w.n_beg;
      while (ok) {
        const bool cur_valid = u < p.num_units;
        if (!cur_valid && !prev_valid) break;
        if (cur_valid && n == w.n_beg) {
          for (int g = 0; g < 2 && ok; ++g) {
            if (w.n1[g] == w.n0[g]) continue;
            ok = wait_bar(bar(L::kQFull + g), q_par[g], ctl, kSiteMmaQ);
            q_par[g] ^= 1u;
          }
          if (!ok) break;
        }
        const uint32_t kslot = slot;
        // V(j-1) and K(j), the two tiles this step reads: one wait
        ok = wait_bar(bar(L::kKVFull + step % (L::kStages / 2)), (step / (L::kStages / 2)) & 1u,
                      ctl, kSiteMmaK);
        if (!ok) break;
        for (int g = 0; g < 2; ++g) {
          // ---- O_g += P_g(j-1) V(j-1)
          if (prev_valid && prev_active[g]) {
            const uint32_t par = p_par[g];
            p_par[g] ^= 1u;
            if constexpr (FP8) {
              // the FP8 softmax arrives on both halves after all of P: one
              // wait (every wait in this thread delays the tensor pipe)
              ok = wait_bar(bar(L::kPFull + 2 * g + 1), par, ctl, kSiteMmaP);
              if (!ok) break;
              tc_fence_after_sync();
              mma_f8_ts_kmajor_x4(tmem + L::o_col(g), tmem + L::s_col(g),
                                  v_desc0 + prev_vslot * kSlotStep, kIdescO,
                                  prev_acc[g] ? 1u : 0u);
            } else {
              ok = wait_bar(bar(L::kPFull + 2 * g), par, ctl, kSiteMmaP);
              if (!ok) break;
              tc_fence_after_sync();
              // keys 0-63: P columns +0, V rows 0-63
              mma_ts_mnmajor_x4(tmem + L::o_col(g), tmem + L::s_col(g),
                                v_desc0 + prev_vslot * kSlotStep, kIdescO, prev_acc[g] ? 1u : 0u);
              ok = wait_bar(bar(L::kPFull + 2 * g + 1), par, ctl, kSiteMmaP);
              if (!ok) break;
              tc_fence_after_sync();
              // keys 64-127: P columns +32, V rows 64-127 (4 steps of 2 KB on)
              mma_ts_mnmajor_x4(tmem + L::o_col(g), tmem + L::s_col(g) + 32,
                                v_desc0 + prev_vslot * kSlotStep + 512, kIdescO, 1u);
            }
            tc_commit(bar(L::kODone + g));
            ++o_cnt[g];
          }
          // ---- S_g = Q_g K_j^T.  It overwrites the columns every earlier
          //      P_g V read its A operand from: wait for the latest one's
          //      commit (the commit tracks all earlier MMAs of this thread).
          if (cur_valid && n >= w.n0[g] && n < w.n1[g]) {
            if (o_seen[g] != o_cnt[g]) {
              ok = wait_bar(bar(L::kODone + g), (o_cnt[g] - 1) & 1u, ctl, kSiteMmaO);
              if (!ok) break;
              o_seen[g] = o_cnt[g];
            }
            tc_fence_after_sync();
            const uint64_t a = q_desc0 + g * kSlotStep;
            const uint64_t b = k_desc0 + kslot * kSlotStep;
            if constexpr (FP8)
              mma_f8_ss_kmajor_x4(tmem + L::s_col(g), a, b, kIdescS, 0u);
            else if constexpr (D == 128)
              mma_ss_kmajor_x8(tmem + L::s_col(g), a, b, kIdescS, 0u);
            else
              mma_ss_kmajor_x4(tmem + L::s_col(g), a, b, kIdescS, 0u);
            tc_commit(bar(L::kSFull + g));
            if (n == w.n1[g] - 1) tc_commit(bar(L::kQEmpty + g));
          }
        }
        if (!ok) break;
        // one commit per step releases K(j) and V(j-1) (release group
        // step % h); the last V goes with the final, K-less step
        tc_commit(bar(L::kKVEmpty + step % (L::kStages / 2)));
        ++step;
        if (!cur_valid) break;
        if (++slot == (uint32_t)L::kStages) slot = 0;
        // V(j): used (and released) in step j+1, whose barrier covers it
        const uint32_t vslot = slot;
        if (++slot == (uint32_t)L::kStages) slot = 0;
        prev_valid = true;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          prev_active[g] = n >= w.n0[g] && n < w.n1[g];
          prev_acc[g] = n > w.n0[g];  // the first tile of a unit overwrites O_g
        }
        prev_vslot = vslot;
        if (++n == w.n_end) {
          do {
            u += gridDim.x;
            if (u < p.num_units) w = decode_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
          } while (u < p.num_units && w.n_end == w.n_beg);
          n = w.n_beg;
        }
      }
      // Every MMA issued must complete before tensor memory is released.
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < 8) {
    regs_increase<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int g = warp / 4;
    const int t = threadIdx.x % 128;  // row within the query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::s_col(g);
    const uint32_t tO = tmem + lane_base + L::o_col(g);
    const uint32_t stage = sbase + L::kStageOff;
    const float scale_log2 = p.scale_log2;
    uint32_t s_par = 0, pv_cnt = 0;
    uint32_t n_stores = 0;  // O tiles staged so far by both warpgroups, in order
    bool ok = true;

    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      const Unit w = decode_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
      // the staging tile is used by tile 0 then tile 1 of each unit (tiles of
      // packed batches are written directly)
      const bool staged0 = staged_tile<CAUSAL, PACKED>(p, w, 0), staged1 = staged_tile<CAUSAL, PACKED>(p, w, 1);
      const uint32_t my_store = n_stores + ((g == 1 && staged0) ? 1u : 0u);
      n_stores += (staged0 ? 1u : 0u) + (staged1 ? 1u : 0u);
      // this warpgroup's tile (g is per warp: selects, not indexed loads)
      const int t_n0 = g ? w.n0[1] : w.n0[0];
      const int t_n1 = g ? w.n1[1] : w.n1[0];
      const int t_row0 = g ? w.row0[1] : w.row0[0];
      if (t_n1 == t_n0) continue;
      // this thread's query position and output head (with grouped-query
      // packing, tile row t is head t % group of position t / group)
      const int gq = PACKED ? p.gqa_log2 : 0;
      const int row = t_row0 + (t >> gq);
      const int o_head = w.sv.o_head + (t & ((1 << gq) - 1));
      float m_ref = -INFINITY;  // reference maximum (log2 units, scaled)
      float l = 0.f;            // running row sum relative to m_ref

      const int len = w.sv.len;
      const int k_len = w.sv.k_len, k_off = w.sv.k_off;
      const int row_end = min(len, t_row0 + (kBlockM >> gq));
      for (int n = t_n0; n < t_n1; ++n) {
        ok = wait_bar(bar(L::kSFull + g), s_par, ctl, kSiteSoftmaxS);
        s_par ^= 1u;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();

        uint32_t sraw[kBlockN];
        float mblk[4];  // per-32-column maxima, reduced by the load itself
        tmem_ld_max_x32x4_sync(tS, sraw, mblk);
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sraw[c]);

        // keys pos - win_left .. pos + win_right below k_len, where
        // pos = row + k_off is the row's key position
        const int kbase = n * kBlockN;
        const bool need_mask = (kbase + kBlockN > k_len) ||
                               (kbase + kBlockN - 1 > t_row0 + k_off + p.win_right) ||
                               (kbase < row_end - 1 + k_off - p.win_left);
        if (need_mask) {
          const int pos = row + k_off;
          const int hi = min(k_len - kbase, pos + p.win_right + 1 - kbase);  // c < hi
          const int lo = pos - p.win_left - kbase;                           // c >= lo
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c >= hi || c < lo) s[c] = -INFINITY;
        }
        // a masked tile takes its maximum over the kept columns only
        const float m_tile =
            (need_mask ? tile_max(s)
                       : fmaxf(fmaxf(mblk[0], mblk[1]), fmaxf(mblk[2], mblk[3]))) *
            scale_log2;
        if (__any_sync(0xffffffffu, m_tile > m_ref + kThreshold)) {
          const float m_new = fmaxf(m_ref, m_tile);
          const float factor = (m_new == -INFINITY) ? 1.f : ex2_approx(m_ref - m_new);
          if (n > t_n0) {
            // O_g holds the previous tiles' sum: wait for the last P_g V MMA,
            // then rescale this warp's 32 rows in tensor memory.
            ok = wait_bar(bar(L::kODone + g), (pv_cnt - 1) & 1u, ctl, kSiteSoftmaxO);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld_x32_sync(tO + c, o);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
              tmem_st_x32(tO + c, o);
            }
            tmem_wait_st();
          }
          l *= factor;
          m_ref = m_new;
        }
        if constexpr (FP8) {
          l += exp_tile_to_tmem_e4m3(s, scale_log2,
                                     ((m_ref == -INFINITY) ? 0.f : m_ref) - kFp8POffset, tS);
          tmem_wait_st();
          tc_fence_before_sync();
          mbar_arrive(bar(L::kPFull + 2 * g));
        } else {
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          // keys 0-63 first: their P V product can start while the rest runs
          float lsum = exp_tile_to_tmem<BF16, 0, kBlockN / 2>(s, scale_log2, m_use, tS);
          tmem_wait_st();
          tc_fence_before_sync();
          mbar_arrive(bar(L::kPFull + 2 * g));
          lsum += exp_tile_to_tmem<BF16, kBlockN / 2, kBlockN>(s, scale_log2, m_use, tS);
          l += lsum;
          tmem_wait_st();
        }
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPFull + 2 * g + 1));
        ++pv_cnt;
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      ok = wait_bar(bar(L::kODone + g), (pv_cnt - 1) & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();

      // O_g is final: read the row (one wait for all its loads), normalise
      // and pack it before waiting for the staging tile, so that this work
      // overlaps the store of the other warpgroup's tile.
      // (FP8: l carries the 2^offset of P; O also takes the V descale)
      const float inv_l = (l > 0.f) ? (FP8 ? p.descale_v : 1.f) / l : 0.f;
      uint32_t pk[D / 2];
      {
        uint32_t o[D];
        if constexpr (D == 128)
          tmem_ld_x32x4_sync(tO, o);
        else
          tmem_ld_2x32_sync(tO, o, tO + 32, o + 32);
#pragma unroll
        for (int e = 0; e < D / 2; ++e)
          pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                              __uint_as_float(o[2 * e + 1]) * inv_l);
      }
      if (p.lse != nullptr && row < len) {
        p.lse[(PACKED ? static_cast<long long>(o_head) * p.total_rows + w.sv.row_base
                      : lse_base<PACKED>(p, w.sv)) + row] =
            (l > 0.f) ? (m_ref + log2f(l) - (FP8 ? kFp8POffset : 0.f)) * 0.6931471805599453f
                      : -INFINITY;
      }
      if constexpr (PACKED) {
        // a packed tile (whose 128-row TMA box could run into the next
        // sequence's rows): the warp stores its rows itself, 64 contiguous
        // bytes per row and store; no staging, no store warp
        const int t_warp = t & ~31;  // tile row of lane 0
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 16) {  // 16 packed words = 32 columns
          uint32_t w16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w16[e] = pk[c0 + e];
          store_rows_x32(w16, threadIdx.x & 31, [&](int rl) -> uint16_t* {
            const int tr = t_warp + rl;
            const int r_row = t_row0 + (tr >> gq);
            if (r_row >= len) return nullptr;
            const int r_head = w.sv.o_head + (tr & ((1 << gq) - 1));
            return p.o_ptr +
                   ((static_cast<long long>(w.sv.row_base) + r_row) * p.H + r_head) * D + 2 * c0;
          });
        }
        continue;
      } else if (!(g ? staged1 : staged0)) {
        // a dense tile not staged (tile 1 of a causal unit): the warp stores
        // its rows of [heads][N][d] itself, 64 contiguous bytes per row and
        // store
        const int t_warp = t & ~31;  // tile row of lane 0
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 16) {  // 16 packed words = 32 columns
          uint32_t w16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w16[e] = pk[c0 + e];
          store_rows_x32(w16, threadIdx.x & 31, [&](int rl) -> uint16_t* {
            const int r_row = t_row0 + t_warp + rl;
            if (r_row >= len) return nullptr;
            return p.o_ptr + (static_cast<long long>(w.sv.o_head) * p.N + r_row) * D + 2 * c0;
          });
        }
        continue;
      }
      // the staging tile must have been read by the store before this one
      ok = wait_bar(bar(L::kStageEmpty), (my_store - 1) & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
#pragma unroll
      for (int c16 = 0; c16 < D / 8; ++c16) {  // 16-byte chunks along the row
        const uint32_t addr = stage + (c16 / 8) * (kBlockM * 128) + t * 128 +
                              (((c16 % 8) ^ (t & 7)) << 4);
        st_shared_v4(addr, pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kStageFull));
    }
    __syncwarp();
  } else if (warp == kStoreWarp) {
    regs_decrease<kControlRegs>();
    // ------------------------------------------------------------ O store
    // Lane 0 waits and issues the TMA store of each staged tile (tiles of
    // packed batches are stored by the softmax threads).
    uint32_t full_par = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok && lane == 0; u += gridDim.x) {
      const Unit w = decode_unit<CAUSAL, PACKED, TABLE>(u, p, tab);
      for (int g = 0; g < 2 && ok; ++g) {
        if (!staged_tile<CAUSAL, PACKED>(p, w, g)) continue;
        ok = wait_bar(bar(L::kStageFull), full_par, ctl, kSiteStore);
        full_par ^= 1u;
        if (!ok) break;
        if (PACKED && p.gqa_log2)
          tma_store_5d(&p.tm_o, sbase + L::kStageOff, 0, 0, w.sv.row_base + w.row0[g], 0,
                       w.sv.kv_head);
        else
          tma_store_4d(&p.tm_o, sbase + L::kStageOff, 0, w.sv.row_base + w.row0[g], 0,
                       w.sv.o_head);
        bulk_commit_group();
        bulk_wait_read_all();  // the staging tile may be rewritten
        mbar_arrive(bar(L::kStageEmpty));
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    regs_decrease<kControlRegs>();  // spare warps of the third warpgroup
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
