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
//   warps 0-3  softmax warpgroup 0   (query tile 0 of the unit, row = thread)
//   warps 4-7  softmax warpgroup 1   (query tile 1)
//   warp  8    TMA producer          (Q tiles, then K_j / V_j into a ring)
//   warp  9    MMA issuer            (S_g = Q_g K_j^T, O_g += P_g V_j)
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
//   O staging      one tile per softmax warpgroup (TMA store source)
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

#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

constexpr int kNumThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kStatusTimeout = 5;           // == FA_ERR_DEVICE_TIMEOUT

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr uint32_t kTileBytes = kBlockM * D * 2;  // == kBlockN * D * 2
  static constexpr int kStages = (D == 64) ? 6 : 3;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kQOff + 2 * kTileBytes;
  static constexpr uint32_t kStageOff = kKVOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kStageOff + 2 * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 2;
  static constexpr int kKVFull = 4;
  static constexpr int kKVEmpty = kKVFull + kStages;
  static constexpr int kSFull = kKVEmpty + kStages;
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kODone = kPFull + 2;
  static constexpr int kDrain = kODone + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr uint32_t kCtlOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kUsedBytes = kCtlOff + 16;
  static constexpr uint32_t kSmemBytes = kUsedBytes + 1024;  // alignment slack
  // tensor-memory columns of S_g / P_g and of O_g
  __device__ static constexpr uint32_t s_col(int g) { return g * 128u; }
  __device__ static constexpr uint32_t o_col(int g) { return 256u + g * D; }
};

// One work unit: 256 query rows of one (b,h) = two 128-row query tiles.
struct Unit {
  int bh;
  int row0[2];  // first query row of each tile
  int nt[2];    // K/V tiles each query tile visits (0 if the tile is empty)
  int ntot;     // K/V tiles streamed for the unit = max(nt)
};

template <bool CAUSAL>
__device__ __forceinline__ Unit decode_unit(int u, const FaParams& p) {
  Unit w;
  int pair;
  if (CAUSAL) {
    // heaviest first: the last query pairs of every head come first
    pair = p.num_pairs - 1 - u / p.num_bh;
    w.bh = u % p.num_bh;
  } else {
    // consecutive units share a head, so its K/V stay hot in L2
    w.bh = u / p.num_pairs;
    pair = u % p.num_pairs;
  }
  w.ntot = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int r0 = pair * kRowsPerUnit + g * kBlockM;
    w.row0[g] = r0;
    if (r0 >= p.N) {
      w.nt[g] = 0;
    } else if (CAUSAL) {
      const int last = min(p.N, r0 + kBlockM);  // rows r0..last-1 see keys < last
      w.nt[g] = (last + kBlockN - 1) / kBlockN;
    } else {
      w.nt[g] = p.n_ktiles;
    }
    w.ntot = max(w.ntot, w.nt[g]);
  }
  return w;
}

struct Ctl {
  volatile int* abort_flag;  // shared memory, CTA-wide
  int* status;               // global status word
  unsigned long long timeout_ns;
};

static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl& c,
                                       int site) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      *c.abort_flag = 1;
      atomicCAS(c.status, 0, kStatusTimeout | (site << 8));
      return false;
    }
  }
}

// Bounded wait for the phase of `bar` with the given parity.  False means the
// wait ran out (or another role gave up): the caller must stop its work.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                         int site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c, site);
}

// Bounded wait that ignores the abort flag (used while draining on exit).
static __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                        unsigned long long limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FaParams p) {
  using L = Layout<D>;
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
      mbar_init(bar(L::kPFull + g), 128);
      mbar_init(bar(L::kODone + g), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kKVFull + s), 1);
      mbar_init(bar(L::kKVEmpty + s), 1);
    }
    mbar_init(bar(L::kDrain), 1);
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

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      uint32_t kv_it = 0, q_it[2] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL>(u, p);
        for (int g = 0; g < 2 && ok; ++g) {
          if (w.nt[g] == 0) continue;
          ok = wait_bar(bar(L::kQEmpty + g), (q_it[g] & 1u) ^ 1u, ctl, kSiteProducerQ);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kQFull + g), L::kTileBytes);
          tma_load_4d(sbase + L::kQOff + g * L::kTileBytes, &p.tm_q, bar(L::kQFull + g), 0,
                      w.row0[g], 0, w.bh);
          ++q_it[g];
        }
        for (int n = 0; n < w.ntot && ok; ++n) {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t slot = kv_it % L::kStages;
            const uint32_t phase = (kv_it / L::kStages) & 1u;
            ok = wait_bar(bar(L::kKVEmpty + slot), phase ^ 1u, ctl, kSiteProducerKV);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(L::kKVFull + slot), L::kTileBytes);
            tma_load_4d(sbase + L::kKVOff + slot * L::kTileBytes, kv ? &p.tm_v : &p.tm_k,
                        bar(L::kKVFull + slot), 0, n * kBlockN, 0, w.bh);
            ++kv_it;
          }
        }
      }
      // Let every copy this warp issued land before the CTA may exit.
      const uint32_t first = kv_it > (uint32_t)L::kStages ? kv_it - L::kStages : 0u;
      for (uint32_t it = first; it < kv_it; ++it)
        wait_drain(bar(L::kKVFull + it % L::kStages), (it / L::kStages) & 1u,
                   p.timeout_ns);
      for (int g = 0; g < 2; ++g)
        if (q_it[g] > 0) wait_drain(bar(L::kQFull + g), (q_it[g] - 1) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_f16(kBlockM, kBlockN, BF16, false);
      constexpr uint32_t kIdescO = make_idesc_f16(kBlockM, D, BF16, true);
      uint32_t kv_it = 0, q_it[2] = {0, 0}, p_it[2] = {0, 0}, o_cnt[2] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL>(u, p);
        for (int g = 0; g < 2 && ok; ++g) {
          if (w.nt[g] == 0) continue;
          ok = wait_bar(bar(L::kQFull + g), q_it[g] & 1u, ctl, kSiteMmaQ);
          ++q_it[g];
        }
        for (int n = 0; n < w.ntot && ok; ++n) {
          // S_g = Q_g K_n^T for every query tile that still visits tile n
          const uint32_t kslot = kv_it % L::kStages;
          ok = wait_bar(bar(L::kKVFull + kslot), (kv_it / L::kStages) & 1u, ctl, kSiteMmaK);
          ++kv_it;
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t k_smem = sbase + L::kKVOff + kslot * L::kTileBytes;
          for (int g = 0; g < 2; ++g) {
            if (n >= w.nt[g]) continue;
            // P_g (aliasing S_g) must have been consumed by the last O_g MMA
            if (o_cnt[g] > 0) {
              ok = wait_bar(bar(L::kODone + g), (o_cnt[g] - 1) & 1u, ctl, kSiteMmaO);
              if (!ok) break;
              tc_fence_after_sync();
            }
            const uint32_t q_smem = sbase + L::kQOff + g * L::kTileBytes;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              // K-major operands: 64-element column blocks of 128 rows x 128 B;
              // 16-element steps advance 32 B inside the swizzled row.
              const uint32_t koff = (k / 4) * (kBlockM * 128) + (k % 4) * 32;
              const uint64_t a = smem_desc_sw128(q_smem + koff, 16, 1024);
              const uint64_t b = smem_desc_sw128(k_smem + koff, 16, 1024);
              mma_ss(tmem + L::s_col(g), a, b, kIdescS, k > 0 ? 1u : 0u);
            }
            tc_commit(bar(L::kSFull + g));
            if (n == w.nt[g] - 1) tc_commit(bar(L::kQEmpty + g));
          }
          if (!ok) break;
          tc_commit(bar(L::kKVEmpty + kslot));

          // O_g += P_g V_n
          const uint32_t vslot = kv_it % L::kStages;
          ok = wait_bar(bar(L::kKVFull + vslot), (kv_it / L::kStages) & 1u, ctl, kSiteMmaV);
          ++kv_it;
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t v_smem = sbase + L::kKVOff + vslot * L::kTileBytes;
          for (int g = 0; g < 2; ++g) {
            if (n >= w.nt[g]) continue;
            ok = wait_bar(bar(L::kPFull + g), p_it[g] & 1u, ctl, kSiteMmaP);
            ++p_it[g];
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int k = 0; k < kBlockN / 16; ++k) {
              // V is MN-major (d contiguous): 64-wide d blocks 128 keys apart
              // (LBO), 8-key groups 1024 B apart (SBO); 16 keys per step.
              const uint64_t b = smem_desc_sw128(v_smem + k * 16 * 128, kBlockN * 128, 1024);
              mma_ts(tmem + L::o_col(g), tmem + L::s_col(g) + k * 8, b, kIdescO,
                     (n > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(bar(L::kODone + g));
            ++o_cnt[g];
          }
          if (!ok) break;
          tc_commit(bar(L::kKVEmpty + vslot));
        }
      }
      // Every MMA issued must complete before tensor memory is released.
      tc_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int g = warp / 4;
    const int t = threadIdx.x % 128;  // row within the query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::s_col(g);
    const uint32_t tO = tmem + lane_base + L::o_col(g);
    const uint32_t stage = sbase + L::kStageOff + g * L::kTileBytes;
    const float scale_log2 = p.scale_log2;
    uint32_t s_it = 0, pv_cnt = 0;
    bool ok = true, store_pending = false;

    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      const Unit w = decode_unit<CAUSAL>(u, p);
      if (w.nt[g] == 0) continue;
      const int row = w.row0[g] + t;
      float m_ref = -INFINITY;  // reference maximum (log2 units, scaled)
      float l = 0.f;            // running row sum relative to m_ref

      for (int n = 0; n < w.nt[g]; ++n) {
        ok = wait_bar(bar(L::kSFull + g), s_it & 1u, ctl, kSiteSoftmaxS);
        ++s_it;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();

        uint32_t sraw[kBlockN];
        tmem_ld_x128_sync(tS, sraw);
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sraw[c]);

        const int kbase = n * kBlockN;
        const bool need_mask =
            (kbase + kBlockN > p.N) || (CAUSAL && kbase + kBlockN - 1 > w.row0[g]);
        if (need_mask) {
          int lim = p.N - kbase;
          if (CAUSAL) lim = min(lim, row - kbase + 1);
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < kBlockN; c += 4) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
          mx2 = fmaxf(mx2, s[c + 2]);
          mx3 = fmaxf(mx3, s[c + 3]);
        }
        const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;

        const bool need = m_tile > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_ref, m_tile);
          const float factor = (m_new == -INFINITY) ? 1.f : ex2_approx(m_ref - m_new);
          if (n > 0) {
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

        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < kBlockN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2_approx(fmaf(s[c0 + 2 * e], scale_log2, -m_use));
            const float p1 = ex2_approx(fmaf(s[c0 + 2 * e + 1], scale_log2, -m_use));
            sum0 += p0;
            sum1 += p1;
            pk[e] = pack2<BF16>(p0, p1);
          }
          tmem_st_x16(tS + c0 / 2, pk);
        }
        tmem_wait_st();
        l += sum0 + sum1;
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPFull + g));
        ++pv_cnt;
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      ok = wait_bar(bar(L::kODone + g), (pv_cnt - 1) & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      if (t == 0 && store_pending) bulk_wait_read_all();  // staging tile free again
      named_bar_sync(1 + g, 128);

      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld_x32_sync(tO + c, o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w4[e] = pack2<BF16>(__uint_as_float(o[8 * j + 2 * e]) * inv_l,
                                __uint_as_float(o[8 * j + 2 * e + 1]) * inv_l);
          const int c16 = c / 8 + j;  // 16-byte chunk index along the row
          const uint32_t addr = stage + (c16 / 8) * (kBlockM * 128) + t * 128 +
                                (((c16 % 8) ^ (t & 7)) << 4);
          st_shared_v4(addr, w4[0], w4[1], w4[2], w4[3]);
        }
      }
      if (p.lse != nullptr && row < p.N) {
        p.lse[static_cast<size_t>(w.bh) * p.N + row] =
            (l > 0.f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + g, 128);
      if (t == 0) {
        tma_store_4d(&p.tm_o, stage, 0, w.row0[g], 0, w.bh);
        bulk_commit_group();
        store_pending = true;
      }
    }
    if (t == 0 && store_pending) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
