// CTA-pair variant of the FC GEMM: one tcgen05 MMA of M = 256, N = 256 is
// shared by the two CTAs of a cluster (cta_group::2).
//
// Tile = 256 x 256 output elements per CTA pair.  CTA rank r of the pair
//   * TMA-loads rows [128 r, 128 r + 128) of the A tile and columns
//     [128 r, 128 r + 128) of the B tile into its OWN shared memory (no
//     multicast); both CTAs' loads complete on the even CTA's mbarrier,
//   * holds rows [128 r, 128 r + 128) x 256 columns of the fp32 accumulator
//     in its own TMEM (double-buffered: 2 x 256 columns),
//   * runs its own epilogue over those rows.
// The even CTA (rank 0) issues every MMA and commits stage releases and
// accumulator-ready signals to both CTAs with one multicast commit; the odd
// CTA's epilogue reports a drained accumulator to the even CTA's barrier.
//
// Per CTA and 64-deep stage: 16 KB of A + 16 KB of B, so 6 stages fit in
// 192 KB.  Every wait is bounded exactly as in the single-CTA kernel.
#pragma once
#include "gemm_kernel.cuh"

namespace axonn {

constexpr int kPairBM = 256;  // output rows per CTA pair
constexpr int kPairBN = 256;  // output columns per CTA pair

template <int STAGES>
struct PairSmemLayout {
  static constexpr int kABytes = 128 * kBK * 2;
  static constexpr int kBBytes = (kPairBN / 2) * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kBytes = 1024 + STAGES * kStageBytes + kNumBars * 8 + 16;
};

template <int STAGES, int MAXP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fc_gemm_tcgen05_pair_kernel(const __grid_constant__ GemmParams<MAXP> P) {
  using L = PairSmemLayout<STAGES>;
  constexpr uint32_t kTmemCols = 2 * kPairBN;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  uint8_t* ring_ptr = smem_raw + (ring - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + STAGES * L::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_addr(bars + 2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_addr(bars + 2 * STAGES + 2 + b); };
  const uint32_t mma_done_bar = smem_addr(bars + 2 * STAGES + 4);
  auto a_tile = [&](int s) { return ring + s * L::kStageBytes; };
  auto b_tile = [&](int s) { return ring + s * L::kStageBytes + L::kABytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P.num_problems; ++p) {
      prefetch_tmap(&P.tma[p]);
      prefetch_tmap(&P.tmb[p]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t tmo = P.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && P.inject != 1) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t loads = 0;
      bool ok = true;
      for (int t = pair; ok && t < P.total_tiles; t += num_pairs) {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        const CUtensorMap* ma = &P.tma[tc.p];
        const CUtensorMap* mb = &P.tmb[tc.p];
        const int m0 = tc.m_blk * kPairBM + static_cast<int>(rank) * 128;
        const int n0 = tc.n_blk * kPairBN + static_cast<int>(rank) * (kPairBN / 2);
        for (int k = 0; k < d.num_k; ++k) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, tmo, abort_flag, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * L::kStageBytes);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const int r0 = k * kBK;
          if (d.a_mn) {
            tma_load_2d_pair(a_tile(stage), ma, fb, m0, r0);
            tma_load_2d_pair(a_tile(stage) + 8192, ma, fb, m0 + 64, r0);
          } else {
            tma_load_2d_pair(a_tile(stage), ma, fb, r0, m0);
          }
          if (d.b_mn) {
            tma_load_2d_pair(b_tile(stage), mb, fb, n0, r0);
            tma_load_2d_pair(b_tile(stage) + 8192, mb, fb, n0 + 64, r0);
          } else {
            tma_load_2d_pair(b_tile(stage), mb, fb, r0, n0);
          }
          ++loads;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain (even CTA): the full barriers count both CTAs' bytes, so the
      // last phase of each stage completing means every copy has landed.
      if (leader) {
        for (int s = 0; s < STAGES; ++s) {
          if (loads > static_cast<uint32_t>(s)) {
            const uint32_t n_s = (loads - s + STAGES - 1) / STAGES;
            wait_bounded(full_bar(s), (n_s - 1) & 1u, tmo, abort_flag, kSiteDrainLoads, false);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc = 0;
      bool ok = true;
      for (int t = pair; ok && t < P.total_tiles; t += num_pairs) {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        if (d.num_k == 0) continue;
        const uint32_t b = acc & 1u;
        const uint32_t acc_phase = (acc >> 1) & 1u;
        if (!wait_bounded(tempty_bar(b), acc_phase ^ 1u, tmo, abort_flag, kSiteMmaTmemEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kPairBN;
        for (int k = 0; k < d.num_k; ++k) {
          if (!wait_bounded(full_bar(stage), phase, tmo, abort_flag, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = a_tile(stage);
          const uint32_t sb = b_tile(stage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = operand_desc<kBK>(sa, kk, d.a_mn);
            const uint64_t bd = operand_desc<kBK>(sb, kk, d.b_mn);
            umma_bf16_pair(d_tmem, ad, bd, d.idesc, (k | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(b), 0x3);
        ++acc;
      }
      umma_commit_pair(mma_done_bar);
      wait_bounded(mma_done_bar, 0, tmo, abort_flag, kSiteDrainMma, false);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint32_t acc = 0;
    for (int t = pair; t < P.total_tiles; t += num_pairs) {
      const TileCoord tc = decode_tile(P, t);
      const ProblemDesc& d = P.prob[tc.p];
      const int row = tc.m_blk * kPairBM + static_cast<int>(rank) * 128 + q * 32 + lane;
      const int n0 = tc.n_blk * kPairBN;
      if (d.num_k == 0) {
        if (row < d.M) store_zero_row(d, row, n0, kPairBN);
        continue;
      }
      const uint32_t b = acc & 1u;
      const uint32_t acc_phase = (acc >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull_bar(b), acc_phase, tmo, abort_flag, kSiteEpiTmemFull);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kPairBN;
#pragma unroll 1
      for (int c = 0; c < kPairBN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= d.N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        if (row < d.M) store_chunk(d, row, col0, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(b));
        else mbar_arrive_cluster(mapa_shared(tempty_bar(b), 0));
      }
      ++acc;
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace axonn
