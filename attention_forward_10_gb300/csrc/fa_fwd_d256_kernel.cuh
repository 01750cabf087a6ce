// fa_fwd_d256_kernel.cuh -- attention forward for head dimension 256 on
// sm_103a (tcgen05, tensor memory, TMA); persistent and warp-specialised.
//
// Same computation as the d <= 128 kernel (the FlashAttention-2 forward of
// LeetCUDA "flash_attn_mma_tiling_qk.cu": tile Q by rows, stream K/V tiles,
// online row max / row sum with the running output rescaled by
// exp(m_old - m_new), division by the row sum at the end; O stored with the
// row LSE as in flash-attention "hopper/flash_fwd_kernel.h"), with a layout
// chosen for d = 256, where the fp32 output tile alone takes half of tensor
// memory:
//
//   work unit  one 128-row query tile of one (b,h)
//   K/V tiles  64 keys (32 KB each at d = 256), a 4-slot ring in shared memory
//   tensor memory (512 columns):
//     [0,64) ... [192,256)        S buffers 0-3 (scores of four
//                                  consecutive K tiles; P, packed 16-bit,
//                                  is written over the first 32 columns)
//     [256,512)                   O (running output, fp32)
//
//   warps 0-3  softmax (one query row per thread)
//   warp  4    TMA producer of Q and the K tiles
//   warp  5    S issuer: S(G) = Q K_G^T into buffer G mod 4, over the
//              stream of K tiles G
//   warp  6    O store (TMA store of the 128x128 staging tile: columns
//              0-127 of a dense tile, both halves of a whole packed tile;
//              the softmax threads store the rest themselves)
//   warp  7    P V issuer: O += P(G) V_G once the softmax has written P(G)
//   warp  8    TMA producer of the V tiles
//
// The tensor pipe accepts only a few MMAs ahead of the one it executes, so
// a single issuing thread that waits on a barrier (a K tile, a P tile) lets
// the pipe run dry; with the two products issued from two warps, one
// issuer's waits overlap the other's MMAs.  The two streams meet only
// through barriers: P V(G) waits for the softmax of tile G (which waited for
// S(G)), and with four S buffers S(G) overwrites the columns of P(G-4), the
// A operand of P(G-4) V, so S(G) first waits for that product's commit
// (barrier ODone of the buffer; the PTX ISA orders tcgen05.mma of one thread
// only when they share the accumulator and shape, and these are issued by
// different threads).  The softmax of tile G-1 runs while S(G) executes.
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_params.h"
#include "ptx.cuh"

namespace fa {

namespace d256 {

constexpr int D = 256;
constexpr int kBN = 64;                 // keys per K/V tile
constexpr int kThreads = 288;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStoreWarp = 6;
constexpr int kPvWarp = 7;
constexpr int kVProducerWarp = 8;
constexpr int kSBufs = 4;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kQBytes = kBlockM * D * 2;   // 64 KB
constexpr uint32_t kKVBytes = kBN * D * 2;      // 32 KB
constexpr int kStages = 4;
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKVOff = kQOff + kQBytes;
constexpr uint32_t kStageOff = kKVOff + kStages * kKVBytes;
constexpr uint32_t kStageBytes = kBlockM * 128 * 2;  // two 64-column blocks
constexpr uint32_t kBarOff = kStageOff + kStageBytes;
// barrier indices
constexpr int kQFull = 0;
constexpr int kQEmpty = 1;
constexpr int kKVFull = 2;
constexpr int kKVEmpty = kKVFull + kStages;
constexpr int kSFull = kKVEmpty + kStages;    // per S buffer
constexpr int kPFull = kSFull + kSBufs;       // per S buffer
constexpr int kODone = kPFull + kSBufs;       // per S buffer: P(G) V done
constexpr int kStageFull = kODone + kSBufs;
constexpr int kStageEmpty = kStageFull + 1;
constexpr int kDrain = kStageEmpty + 1;
constexpr int kDrainPv = kDrain + 1;
constexpr int kNumBars = kDrainPv + 1;
constexpr uint32_t kCtlOff = kBarOff + kNumBars * 8;
constexpr uint32_t kUsedBytes = kCtlOff + 16;
constexpr uint32_t kSmemBytes = kUsedBytes + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the shared memory of one CTA");
constexpr uint32_t kOCol = 256;

struct Unit {
  int bh;     // query head
  SeqView sv; // its rows and tensor-map heads
  int row0;   // first query row of the tile (within the sequence)
  int n0, n1; // K/V tiles visited: [n0, n1); empty only for a key split
              // that the tile's rows cannot see
};

template <bool CAUSAL, bool PACKED>
__device__ __forceinline__ Unit decode_unit(int u, const FaParams& p) {
  Unit w;
  if (CAUSAL && !PACKED && u < p.num_units) u = wave_order(u, p.num_units, gridDim.x);
  int split = 0;
  if (p.num_splits > 1) {
    split = u % p.num_splits;
    u /= p.num_splits;
  }
  int qt;
  if (CAUSAL) {
    qt = p.num_pairs - 1 - u / p.num_bh;  // heaviest first
    w.bh = u % p.num_bh;
  } else {
    w.bh = u / p.num_pairs;
    qt = u % p.num_pairs;
  }
  w.sv = seq_view<PACKED>(p, w.bh, split * p.num_bh + w.bh);
  const int len = w.sv.len;
  if (PACKED && CAUSAL) {
    // sequences differ in length: count the tiles from each sequence's end,
    // so that every sequence's heaviest (last) tiles come first
    qt = (len + kBlockM - 1) / kBlockM - 1 - (p.num_pairs - 1 - qt);
    if (qt < 0) qt = p.num_pairs;  // no such tile: an empty unit
  }
  w.row0 = qt * kBlockM;
  if (w.row0 >= len) {
    w.n0 = w.n1 = 0;  // past the end of a shorter packed sequence
    return w;
  }
  // rows row0 .. sit at key positions row0 + k_off .. (bottom-right alignment)
  key_tile_range(w.row0 + w.sv.k_off, min(len, w.row0 + kBlockM) + w.sv.k_off, w.sv.k_len,
                 p.win_left, p.win_right, kBN, &w.n0, &w.n1);
  if (p.num_splits > 1) {
    clip_to_split(split, p.split_tiles, &w.n0, &w.n1);
  } else if (w.n1 == w.n0) {
    // no row of the tile has a key: one fully masked key tile gives its rows
    // O = 0 and LSE = -inf through the ordinary path
    w.n0 = 0;
    w.n1 = 1;
  }
  return w;
}

}  // namespace d256

// p.num_pairs holds the number of 128-row query tiles per (b,h) and
// p.n_ktiles the number of 64-key tiles for this kernel.
template <bool CAUSAL, bool BF16, bool PACKED>
__global__ void __launch_bounds__(d256::kThreads, 1)
    fa_fwd_d256_kernel(const __grid_constant__ FaParams p) {
  using namespace d256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  auto bar = [&](int i) -> uint32_t { return sbase + kBarOff + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kCtlOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kCtlOff + 4);
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kKVFull + s), 1);
      mbar_init(bar(kKVEmpty + s), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kPFull + b), 128);
      mbar_init(bar(kODone + b), 1);
    }
    mbar_init(bar(kStageFull), 128);
    mbar_init(bar(kStageEmpty), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kDrainPv), 1);
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

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ---------------------------------------------------------------- TMA
    // K(G) goes to ring slot 2 (G mod 2), V(G) to slot 2 (G mod 2) + 1; warp
    // 4 loads Q and the K tiles, warp 8 the V tiles, so that a K tile never
    // waits behind a V tile whose slot the slower P V chain still holds.
    if (lane == 0) {
      const bool is_v = warp == kVProducerWarp;
      uint32_t q_it = 0, G = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL, PACKED>(u, p);
        if (w.n1 == w.n0) continue;
        if (!is_v) {
          ok = wait_bar(bar(kQEmpty), (q_it & 1u) ^ 1u, ctl, kSiteProducerQ);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kQFull), kQBytes);
          tma_load_4d(sbase + kQOff, &p.tm_q, bar(kQFull), 0, w.sv.row_base + w.row0, 0,
                      w.sv.q_head);
          ++q_it;
        }
        for (int n = w.n0; n < w.n1 && ok; ++n, ++G) {
          const uint32_t slot = 2u * (G % 2u) + (is_v ? 1u : 0u);
          ok = wait_bar(bar(kKVEmpty + slot), ((G / 2u) & 1u) ^ 1u, ctl, kSiteProducerKV);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kKVFull + slot), kKVBytes);
          tma_load_4d(sbase + kKVOff + slot * kKVBytes, is_v ? &p.tm_v : &p.tm_k,
                      bar(kKVFull + slot), 0, w.sv.k_row_base + n * kBN, 0, w.sv.kv_head);
        }
      }
      // Let every copy this thread issued land before the CTA may exit.
      for (uint32_t g = G > 2u ? G - 2u : 0u; g < G; ++g)
        wait_drain(bar(kKVFull + 2u * (g % 2u) + (is_v ? 1u : 0u)), (g / 2u) & 1u, p.timeout_ns);
      if (q_it > 0) wait_drain(bar(kQFull), (q_it - 1) & 1u, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ S = Q K^T
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_f16(kBlockM, kBN, BF16, false);
      constexpr uint32_t kSlotStep = kKVBytes >> 4;  // descriptor units
      const uint64_t q_desc = smem_desc_sw128(sbase + kQOff, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(sbase + kKVOff, 16, 1024);
      uint32_t q_par = 0;
      uint32_t G = 0;  // global index of this CTA's K tiles (S tiles)
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL, PACKED>(u, p);
        if (w.n1 == w.n0) continue;  // empty key split: nothing to do
        ok = wait_bar(bar(kQFull), q_par, ctl, kSiteMmaQ);
        q_par ^= 1u;
        for (int n = w.n0; n < w.n1 && ok; ++n, ++G) {
          // K(G) is load 2G of the ring
          const uint32_t b = G % kSBufs;
          const uint32_t kslot = (2u * G) % kStages;
          ok = wait_bar(bar(kKVFull + kslot), ((2u * G) / kStages) & 1u, ctl, kSiteMmaK);
          if (!ok) break;
          // P(G-4) occupied buffer b: its P V product must have read it
          // before this product overwrites it
          if (G >= (uint32_t)kSBufs) {
            ok = wait_bar(bar(kODone + b), ((G - kSBufs) / kSBufs) & 1u, ctl, kSiteMmaO);
            if (!ok) break;
          }
          tc_fence_after_sync();
          mma_ss_kmajor_x16_q128_k64(tmem + b * kBN, q_desc, k_desc0 + kslot * kSlotStep,
                                     kIdescS, 0u);
          tc_commit(bar(kSFull + b));
          tc_commit(bar(kKVEmpty + kslot));
          if (n == w.n1 - 1) tc_commit(bar(kQEmpty));
        }
      }
      tc_commit(bar(kDrain));
      wait_drain(bar(kDrain), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ----------------------------------------------------------- O += P V
    if (lane == 0) {
      constexpr uint32_t kIdescO = make_idesc_f16(kBlockM, D, BF16, true);
      constexpr uint32_t kSlotStep = kKVBytes >> 4;  // descriptor units
      // V (64 keys x 256): MN-major, 64-wide d blocks 64 keys x 128 B apart
      // (LBO), 8-key groups 1024 B apart (SBO)
      const uint64_t v_desc0 = smem_desc_sw128(sbase + kKVOff, kBN * 128, 1024);
      uint32_t G = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
        const Unit w = decode_unit<CAUSAL, PACKED>(u, p);
        if (w.n1 == w.n0) continue;
        for (int n = w.n0; n < w.n1 && ok; ++n, ++G) {
          // V(G) is load 2G + 1 of the ring; P(G) sits in buffer G mod 4
          const uint32_t pb = G % kSBufs;
          const uint32_t vslot = (2u * G + 1u) % kStages;
          ok = wait_bar(bar(kKVFull + vslot), ((2u * G + 1u) / kStages) & 1u, ctl, kSiteMmaV);
          ok = ok && wait_bar(bar(kPFull + pb), (G / kSBufs) & 1u, ctl, kSiteMmaP);
          if (!ok) break;
          tc_fence_after_sync();
          mma_ts_mnmajor_x4(tmem + kOCol, tmem + pb * kBN, v_desc0 + vslot * kSlotStep, kIdescO,
                            n > w.n0 ? 1u : 0u);
          tc_commit(bar(kODone + pb));
          tc_commit(bar(kKVEmpty + vslot));
        }
      }
      tc_commit(bar(kDrainPv));
      wait_drain(bar(kDrainPv), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;  // row within the query tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + kOCol;
    const uint32_t stage = sbase + kStageOff;
    const float scale_log2 = p.scale_log2;
    uint32_t G = 0, n_stores = 0;
    bool ok = true;

    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      const Unit w = decode_unit<CAUSAL, PACKED>(u, p);
      if (w.n1 == w.n0) continue;
      const int row = w.row0 + t;
      float m_ref = -INFINITY, l = 0.f;
      const int len = w.sv.len;
      const int k_len = w.sv.k_len, k_off = w.sv.k_off;
      const int row_end = min(len, w.row0 + kBlockM);
      for (int n = w.n0; n < w.n1; ++n, ++G) {
        const uint32_t b = G % kSBufs;
        const uint32_t tS = tmem + lane_base + b * kBN;
        ok = wait_bar(bar(kSFull + b), (G / kSBufs) & 1u, ctl, kSiteSoftmaxS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        float s[kBN];
        float mblk[2];  // per-32-column maxima, reduced by the load itself
        {
          uint32_t r[kBN];
          tmem_ld_max_x32x2_sync(tS, r, mblk);
#pragma unroll
          for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(r[c]);
        }
        // keys pos - win_left .. pos + win_right below k_len, where
        // pos = row + k_off is the row's key position
        const int kbase = n * kBN;
        const bool need_mask = (kbase + kBN > k_len) ||
                               (kbase + kBN - 1 > w.row0 + k_off + p.win_right) ||
                               (kbase < row_end - 1 + k_off - p.win_left);
        if (need_mask) {
          const int pos = row + k_off;
          const int hi = min(k_len - kbase, pos + p.win_right + 1 - kbase);  // c < hi
          const int lo = pos - p.win_left - kbase;                           // c >= lo
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= hi || c < lo) s[c] = -INFINITY;
        }
        float m_raw = fmaxf(mblk[0], mblk[1]);
        if (need_mask) {
          // a masked tile takes its maximum over the kept columns only
          float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
          for (int c = 4; c < kBN; c += 4) {
            mx0 = fmaxf(mx0, s[c]);
            mx1 = fmaxf(mx1, s[c + 1]);
            mx2 = fmaxf(mx2, s[c + 2]);
            mx3 = fmaxf(mx3, s[c + 3]);
          }
          m_raw = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        }
        const float m_tile = m_raw * scale_log2;

        const bool need = m_tile > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_ref, m_tile);
          const float factor = (m_new == -INFINITY) ? 1.f : ex2_approx(m_ref - m_new);
          if (n > w.n0) {
            // O holds the previous tiles' sum: wait for P(G-1) V, rescale
            const uint32_t pb = (G - 1) % kSBufs;
            ok = wait_bar(bar(kODone + pb), ((G - 1) / kSBufs) & 1u, ctl, kSiteSoftmaxO);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll 1
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
        const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
        const uint64_t neg_m2 = pack_f32x2(-m_use, -m_use);
        uint64_t acc_a = pack_f32x2(0.f, 0.f), acc_b = acc_a;
#pragma unroll
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            unpack_f32x2(fma_f32x2(pack_f32x2(s[c0 + 2 * e], s[c0 + 2 * e + 1]), scale2, neg_m2),
                         x0, x1);
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
        tmem_wait_st();
        {
          float a0, a1;
          unpack_f32x2(add_f32x2(acc_a, acc_b), a0, a1);
          l += a0 + a1;
        }
        tc_fence_before_sync();
        mbar_arrive(bar(kPFull + b));
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      const uint32_t last = G - 1;
      ok = wait_bar(bar(kODone + last % kSBufs), (last / kSBufs) & 1u, ctl, kSiteEpilogueO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if (PACKED && len - w.row0 < kBlockM) {
        // the last tile of a packed sequence, whose 128-row TMA box would
        // run into the next sequence's rows: each thread stores its own row
        // (16-byte stores); no staging, no store warp
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t o[32];
          tmem_ld_x32_sync(tO + c, o);
          if (row < len) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.o_ptr + ((static_cast<long long>(w.sv.row_base) + row) * p.H + w.sv.o_head) *
                              256 + c);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack2<BF16>(__uint_as_float(o[8 * j + 2 * e]) * inv_l,
                                    __uint_as_float(o[8 * j + 2 * e + 1]) * inv_l);
              dst[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
      // Dense layout: columns 0-127 through the staging tile and a TMA
      // store, columns 128-255 stored by the warps themselves (coalesced
      // 64-byte row segments), so that the second half does not wait for
      // the first half's store to free the staging tile.  Whole packed
      // tiles stage both halves.
      const int staged_halves = PACKED ? 2 : 1;
      for (int half = 0; half < staged_halves && ok && !(PACKED && len - w.row0 < kBlockM);
           ++half) {
        // the staging tile must have been read by the store before this one
        ok = wait_bar(bar(kStageEmpty), (n_stores - 1) & 1u, ctl, kSiteEpilogueO);
        ok = __all_sync(0xffffffffu, ok);
        ++n_stores;
        if (!ok) break;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t o[32];
          tmem_ld_x32_sync(tO + half * 128 + c, o);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = pack2<BF16>(__uint_as_float(o[8 * j + 2 * e]) * inv_l,
                                  __uint_as_float(o[8 * j + 2 * e + 1]) * inv_l);
            const int c16 = c / 8 + j;  // 16-byte chunk within the half row
            const uint32_t addr = stage + (c16 / 8) * (kBlockM * 128) + t * 128 +
                                  (((c16 % 8) ^ (t & 7)) << 4);
            st_shared_v4(addr, w4[0], w4[1], w4[2], w4[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kStageFull));
      }
      if (!PACKED && ok) {
        const int t_warp = t & ~31;  // tile row of lane 0
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t o[32];
          tmem_ld_x32_sync(tO + 128 + c, o);
          uint32_t w16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w16[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                                 __uint_as_float(o[2 * e + 1]) * inv_l);
          store_rows_x32(w16, lane, [&](int rl) -> uint16_t* {
            const int r_row = w.row0 + t_warp + rl;
            if (r_row >= len) return nullptr;
            return p.o_ptr + (static_cast<long long>(w.sv.o_head) * p.N + r_row) * 256 + 128 + c;
          });
        }
      }
      if (p.lse != nullptr && row < len) {
        p.lse[lse_base<PACKED>(p, w.sv) + row] =
            (l > 0.f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
    __syncwarp();
  } else if (warp == kStoreWarp) {
    // ------------------------------------------------------------ O store
    // Lane 0 waits and issues the TMA stores of the staged halves of each
    // tile: columns 0-127 of a dense tile, both halves of a whole packed
    // tile (the partial last tiles of packed sequences are stored by the
    // softmax threads).
    uint32_t full_par = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok && lane == 0; u += gridDim.x) {
      const Unit w = decode_unit<CAUSAL, PACKED>(u, p);
      if (w.n1 == w.n0) continue;
      if (PACKED && w.sv.len - w.row0 < kBlockM) continue;
      for (int half = 0; half < (PACKED ? 2 : 1) && ok; ++half) {
        ok = wait_bar(bar(kStageFull), full_par, ctl, kSiteStore);
        full_par ^= 1u;
        if (!ok) break;
        // columns [128*half, 128*half + 128) = d blocks 2*half, 2*half + 1
        tma_store_4d(&p.tm_o, sbase + kStageOff, 0, w.sv.row_base + w.row0, 2 * half,
                     w.sv.o_head);
        bulk_commit_group();
        bulk_wait_read_all();
        mbar_arrive(bar(kStageEmpty));
      }
    }
    if (lane == 0) bulk_wait_all();
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
