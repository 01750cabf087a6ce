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
  kSitePair = 11,
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

// K/V head of query head bh = b*H + h (grouped heads: h / group).
__host__ __device__ inline int kv_head(int bh, int H, int group) {
  const int H_kv = H / group;
  return (bh / H) * H_kv + (bh % H) / group;
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
