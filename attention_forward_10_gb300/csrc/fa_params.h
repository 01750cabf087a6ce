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
  int n_ktiles;      // ceil(N / 128)
  float scale_log2;  // softmax scale * log2(e)
};

}  // namespace fa
