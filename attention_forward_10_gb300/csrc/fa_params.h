// fa_params.h -- launch parameters shared by the host launcher and the
// sm_103a kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (header-only use; no driver link needed)
#include <cstdint>

namespace fa {

// Tile shape of the kernels: 128 query rows (the M of one tcgen05 MMA with
// cta_group::1) by 128 keys per K/V tile.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Two query tiles (256 rows) per work unit: one per softmax warpgroup.
constexpr int kRowsPerUnit = 2 * kBlockM;
// Limits of the per-CTA unit table of packed causal launches.
constexpr int kTableSeqs = 64;
constexpr int kTablePairs = 256;
constexpr int kBwdTableTiles = 128;  // backward: tiles per problem

// Site codes recorded in the status word when a bounded wait runs out.
enum WaitSite : int {
  kSiteProducerQ = 1,
  kSiteProducerKV = 2,
  kSiteMmaQ = 3,
  kSiteMmaK = 4,
  kSiteMmaV = 5,
  kSiteMmaO = 6,
  kSiteMmaP = 7,
  kSiteSoftmaxS = 8,
  kSiteSoftmaxO = 9,
  kSiteEpilogueO = 10,
  kSiteStore = 12,
  kSiteSelftest = 15,
};

struct FaParams {  // 64-byte aligned through CUtensorMap
  CUtensorMap tm_q;  // 4-D views {64, N, d/64, B*H} of [B,H,N,d] (see launcher)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;
  float* lse;        // [B*H, N] fp32 or nullptr
  int* status;       // device status word (first timeout wins)
  unsigned long long timeout_ns;
  int N;             // sequence length
  int num_bh;        // B*H
  int num_pairs;     // ceil(N / 256): work units per (b,h)
  int num_units;     // work units (see num_pair_units)
  int num_pair_units;  // units below this index are query-tile pairs; the
                       // rest are single tiles (d <= 128 kernel)
  int n_ktiles;      // number of K/V tiles along N
  int H;             // query heads per batch entry
  int group;         // query heads per K/V head (H / H_kv)
  int win_left;      // query i sees keys i - win_left .. i + win_right,
  int win_right;     //   both clamped to [0, N]; win_right = 0 when causal
  int num_splits;    // key splits per query tile (1: no split)
  int split_tiles;   // K/V tiles per key split
  float scale_log2;  // softmax scale * log2(e)
  // Variable-length batches (packed rows; nullptr / 0 otherwise): sequence
  // b holds query rows [cu_seqlens[b], cu_seqlens[b+1]) of the packed
  // [rows][H][d] Q and O and key rows [cu_seqlens_k[b], cu_seqlens_k[b+1])
  // of the packed K and V (the same array for self-attention); seqused_q /
  // seqused_k (nullptr: all rows) cut each to its first used rows.  N is
  // then the longest query sequence, N_k the longest key sequence and
  // num_bh = batch * H.
  const int* cu_seqlens;
  const int* cu_seqlens_k;
  const int* seqused_q;
  const int* seqused_k;
  int total_rows;    // rows of the packed Q and O
  int total_rows_k;  // rows of the packed K and V
  int N_k;           // longest key sequence (N when not packed)
  // Grouped-query packing (packed batches, d <= 128; 0 otherwise): log2 of
  // the query heads of one K/V head that share a 128-row tile.  A tile then
  // holds 128 >> gqa_log2 positions of all those heads (row = position *
  // heads + head), units count (b, K/V head) problems, tm_q / tm_o are 5-D
  // views {64, heads of a group, rows, d/64, K/V heads} and num_bh = batch
  // * H_kv.
  int gqa_log2;
  // Packed causal launches of the d <= 128 kernel with at most
  // kTableSeqs sequences and 2 .. kTablePairs units per problem: 1 when
  // every CTA builds the unit table (units ordered by their pair index from
  // the sequence start, heaviest first; see the kernel), 0 otherwise.
  int unit_table;
  uint16_t* o_ptr;   // O (packed rows), for the row-by-row store of the last
                     // query tile of a sequence
  float descale_v;   // FP8 kernels: V descale, applied to O in the epilogue
};

// Split-KV: unit u is split u % num_splits of base unit u / num_splits; the
// split covers K/V tiles [s * split_tiles, (s + 1) * split_tiles).  Its O and
// LSE go to head s * num_bh + bh of the partial outputs.
__host__ __device__ inline void clip_to_split(int s, int split_tiles, int* n0, int* n1) {
  const int lo = s * split_tiles, hi = lo + split_tiles;
  if (*n0 < lo) *n0 = lo;
  if (*n1 > hi) *n1 = hi;
  if (*n1 < *n0) *n1 = *n0;
}

// Launch parameters of the backward kernels ([B][H][N][d] layout, d <= 128).
struct BwdParams {  // 64-byte aligned through CUtensorMap
  CUtensorMap tm_q;   // {64, N, d/64, B*H}, box {64, 128, d/64, 1}
  CUtensorMap tm_k;   // {64, N, d/64, B*H_kv}
  CUtensorMap tm_v;
  CUtensorMap tm_do;  // like tm_q
  const float* lse2;  // [B*H][n_pad]: -LSE * log2(e); -inf on padding rows
  const float* dsum;  // [B*H][n_pad]: -rowsum(dO * O); 0 on padding rows
  uint16_t* dq;       // [B*H][N][d]
  uint16_t* dk;       // [B*H_kv][N][d]
  uint16_t* dv;
  int* status;
  unsigned long long timeout_ns;
  int N, n_pad, n_tiles;  // rows, rows rounded up to 128, 128-row tiles
  int num_bh, num_bkv;    // B*H, B*H_kv
  int num_units;          // work units of the launched kernel
  int H, H_kv, group;
  int win_left, win_right;  // clamped to [0, N + N_k]; win_right = 0 when causal
  float scale, scale_log2;
  // packed variable-length batches (nullptr / 0 otherwise): Q, O, dO, dQ are
  // [total_rows][H][d] and K, V, dK, dV [total_rows_k][H_kv][d]; sequence b
  // owns query rows cu_seqlens[b] .. cu_seqlens[b+1]-1 and key rows
  // cu_seqlens_k[b] .. (the same offsets for self-attention), cut to
  // seqused_q[b] / seqused_k[b] rows when given; N and N_k are the longest
  // query and key lengths and num_bh = batch * H.  Masks are aligned
  // bottom-right: query i of a sequence sits at key position i + k_len - len.
  const int* cu_seqlens;
  const int* cu_seqlens_k;
  const int* seqused_q;
  const int* seqused_k;
  int total_rows, total_rows_k;
  int N_k, n_tiles_k;  // longest key length (N unless packed) and its 128-key tiles
  // Packed causal launches with at most kTableSeqs sequences and 2 ..
  // kBwdTableTiles tiles per problem: 1 when every CTA orders its units from
  // a unit table (see the kernels), 0 otherwise.
  int unit_table;
};

// Rows of one (b, h) attention problem: the first packed row and the length
// of its queries and of its keys, the head coordinates of its Q, O and K/V
// in the tensor maps, and the bottom-right alignment of the masks: query i
// sits at key position i + k_off (flash-attention's causal and local masks
// shift the query row by seqlen_k - seqlen_q).
struct SeqView {
  int row_base;   // 0, or the sequence's first packed query row
  int len;        // N, or the sequence's used query rows (clamped to the buffers)
  int k_row_base; // 0, or the sequence's first packed key row
  int k_len;      // N, or the sequence's used key rows (clamped to the buffers)
  int k_off;      // k_len - len (0 for self-attention)
  int q_head;     // head coordinate of Q (bh, or h when packed)
  int o_head;     // head coordinate of O (out_head, or h when packed)
  int kv_head;    // head coordinate of K and V
};

// K/V head of query head bh = b*H + h (grouped heads: h / group).
// Order in which a persistent grid of `grid` CTAs takes its work units: CTA
// c runs slots c, c + grid, c + 2 grid, ... and slot s runs unit
// wave_order(s).  Causal units are numbered heaviest first, so slots taken
// round robin would hand CTA 0 the heaviest unit of every wave; every other
// wave is reversed instead (CTA 0 takes the heaviest unit of even waves and
// the lightest of odd ones), which evens out the CTAs' totals.  A bijection
// of [0, num_units): a last, partial wave is reversed within itself.
__host__ __device__ inline int wave_order(int s, int num_units, int grid) {
  const int k = s / grid;
  if ((k & 1) == 0) return s;
  const int first = k * grid;
  const int size = (num_units - first < grid) ? num_units - first : grid;
  return first + (size - 1 - (s - first));
}

__host__ __device__ inline int kv_head(int bh, int H, int group) {
  const int H_kv = H / group;
  return (bh / H) * H_kv + (bh % H) / group;
}

// Geometry of the (b,h) problem bh; `out_head` is the output head of the
// non-packed layout (bh, or a split's partial head).  PACKED kernels serve
// variable-length batches (cu_seqlens set).  For packed batches the
// offsets are clamped so that a malformed cu_seqlens can only shorten a
// sequence (to at most N rows), never move a row outside [0, total_rows).
// First row and used length of sequence b under offsets cu (clamped to
// [0, total]) and optional used lengths, capped at cap rows.
__device__ __forceinline__ void packed_rows(const int* cu, const int* used, int b, int total,
                                            int cap, int* first, int* len) {
  int r0 = cu[b], r1 = cu[b + 1];
  r0 = r0 < 0 ? 0 : (r0 > total ? total : r0);
  r1 = r1 < r0 ? r0 : (r1 > total ? total : r1);
  int n = r1 - r0;
  if (used != nullptr) {
    const int u = used[b];
    n = u < 0 ? 0 : (u < n ? u : n);
  }
  *first = r0;
  *len = n < cap ? n : cap;
}

// Query rows (first packed row and used length) and key rows of sequence b
// of a backward launch, clamped as packed_rows clamps them.
template <bool PACKED>
__device__ __forceinline__ void bwd_sequence(const BwdParams& p, int b, int* row_base,
                                             int* len) {
  if constexpr (!PACKED) {
    *row_base = 0;
    *len = p.N;
  } else {
    packed_rows(p.cu_seqlens, p.seqused_q, b, p.total_rows, p.N, row_base, len);
  }
}

template <bool PACKED>
__device__ __forceinline__ void bwd_keys(const BwdParams& p, int b, int* k_row_base,
                                         int* k_len) {
  if constexpr (!PACKED) {
    *k_row_base = 0;
    *k_len = p.N;
  } else {
    packed_rows(p.cu_seqlens_k, p.seqused_k, b, p.total_rows_k, p.N_k, k_row_base, k_len);
  }
}

template <bool PACKED>
__device__ __forceinline__ SeqView seq_view(const FaParams& p, int bh, int out_head) {
  SeqView v;
  if constexpr (!PACKED) {
    v.row_base = 0;
    v.len = p.N;
    v.k_row_base = 0;
    v.k_len = p.N;
    v.k_off = 0;
    v.q_head = bh;
    v.o_head = out_head;
    v.kv_head = kv_head(bh, p.H, p.group);
    return v;
  }
  // (grouped-query packing: problem bh is K/V head hk of sequence b, and
  // its tiles hold all the query heads hk * group .. of that K/V head)
  const int heads = p.H >> p.gqa_log2;
  const int b = bh / heads, h = bh % heads;
  packed_rows(p.cu_seqlens, p.seqused_q, b, p.total_rows, p.N, &v.row_base, &v.len);
  packed_rows(p.cu_seqlens_k, p.seqused_k, b, p.total_rows_k, p.N_k, &v.k_row_base, &v.k_len);
  v.k_off = v.k_len - v.len;
  v.q_head = h << p.gqa_log2;
  v.o_head = h << p.gqa_log2;
  v.kv_head = p.gqa_log2 ? h : h / p.group;
  return v;
}

// Index in the LSE output of row 0 of the problem seen through `v`:
// [heads][N] rows, or [H][total_rows] for packed batches.
template <bool PACKED>
__device__ __forceinline__ long long lse_base(const FaParams& p, const SeqView& v) {
  if constexpr (PACKED) return static_cast<long long>(v.o_head) * p.total_rows + v.row_base;
  return static_cast<long long>(v.o_head) * p.N;
}

// K/V tiles [n0, n1) of `tile` keys that query rows [r0, r_end) can see.
__host__ __device__ inline void key_tile_range(int r0, int r_end, int N, int win_left,
                                               int win_right, int tile, int* n0, int* n1) {
  const long long lo = r0 - static_cast<long long>(win_left);
  const long long hi = static_cast<long long>(r_end) + win_right;  // exclusive
  const int key_lo = lo < 0 ? 0 : static_cast<int>(lo);
  const int key_hi = hi > N ? N : static_cast<int>(hi);
  *n0 = key_lo / tile;
  *n1 = key_hi > key_lo ? (key_hi + tile - 1) / tile : *n0;
}

}  // namespace fa
