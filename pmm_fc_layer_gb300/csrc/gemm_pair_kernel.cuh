// CTA-pair variant of the FC GEMM: each tcgen05 MMA of M = 256 rows and
// N = BN columns is shared by the two CTAs of a cluster (cta_group::2).
//
// Pair tile = MH*256 x BN output elements.  CTA rank r of the pair
//   * TMA-loads its own MH*128 rows [MH*128 r, MH*128 (r+1)) of the A tile
//     and columns [BN/2 r, BN/2 (r+1)) of the B tile into its OWN shared
//     memory (no multicast); both CTAs' loads complete on the even CTA's
//     mbarrier,
//   * holds its MH*128 rows x BN columns of the fp32 accumulator in its own
//     TMEM,
//   * runs its own epilogue over those rows.
// MMA hh (0 <= hh < MH) multiplies rows [128 hh, 128 hh + 128) of each
// CTA's A slice by the whole B tile, so one B slice serves MH MMAs.
// MH = 1: 256 x BN tiles, accumulator double-buffered (2 x BN columns),
//         6 stages of 32 KB.
// MH = 2: 512 x BN tiles; each SM loads 48 KB per 64-deep stage for
//         2 x 128 x BN x 64 multiply-adds (about 1.35x the FLOPs per loaded
//         byte of MH = 1), the two accumulators fill TMEM (single-buffered)
//         and 8 epilogue warps drain them; the CTA has 12 warps and moves
//         registers from warpgroup 0 to the epilogue (see cta_threads).
// The even CTA (rank 0) issues every MMA and commits stage releases and
// accumulator-ready signals to both CTAs with one multicast commit (an
// mbarrier signal, not a data copy); the odd CTA's epilogue reports a
// drained accumulator to the even CTA's barrier.  Every wait is bounded
// exactly as in the single-CTA kernel.
#pragma once
#include "gemm_kernel.cuh"

namespace axonn {

template <int BN, int STAGES, int MH>
struct PairSmemLayout {
  static constexpr int kAHalfBytes = 128 * kBK * 2;
  static constexpr int kABytes = MH * kAHalfBytes;
  static constexpr int kBBytes = (BN / 2) * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kBytes = 1024 + STAGES * kStageBytes + kNumBars * 8 + 16;
};

template <int BN, int STAGES, int MAXP, int MH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_threads<MH, MH == 2>(), 1)
    fc_gemm_tcgen05_pair_kernel(const __grid_constant__ GemmParams<MAXP> P) {
  using L = PairSmemLayout<BN, STAGES, MH>;
  static_assert(MH == 1 || MH == 2, "row halves per CTA");
  static_assert(BN == 128 || BN == 256, "each CTA's B slice is whole 64-column chunks");
  constexpr int kAccBufs = MH == 1 ? 2 : 1;
  constexpr uint32_t kHalfCols = BN;
  constexpr uint32_t kAccCols = MH * kHalfCols;
  constexpr uint32_t kTmemUsed = kAccBufs * kAccCols;
  constexpr uint32_t kTmemCols = kTmemUsed <= 128 ? 128 : (kTmemUsed <= 256 ? 256 : 512);
  constexpr int kCtaM = MH * 128;   // output rows of one CTA
  constexpr int kTileM = 2 * kCtaM;  // output rows of the pair
  static_assert(kTmemUsed <= 512, "TMEM columns");

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
      mbar_init(tempty_bar(b), 2 * kEpiWarps * MH);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P.num_maps; ++p) {
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
  // Barrier set-up, TMEM allocation and tensor-map prefetch above overlap
  // the previous kernel's tail; nothing below touches global memory before
  // that kernel is complete.
  griddep_wait();

  constexpr bool kSplit = MH == 2;  // 12 warps, registers moved to the epilogue
  if (warp < epi_first_warp<MH, kSplit>()) shrink_registers<MH, kSplit>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && P.inject != 1) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t loads = 0;
      for_each_work(P, pair, num_pairs, [&](int t, int k0, int k1, int) -> bool {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        // L2 priorities of this tile's operand lines (see ProblemDesc)
        const uint64_t pol_a = l2_policy(d.l2_keep == 1, d.l2_keep_frac);
        const uint64_t pol_b = l2_policy(d.l2_keep == 2, d.l2_keep_frac);
        ChainPos cp = chain_start(P, d, k0);
        const CUtensorMap* ma = &P.tma[d.map0 + cp.g];
        const CUtensorMap* mb = &P.tmb[d.map0 + cp.g];
        const int m0 = tc.m_blk * kTileM + static_cast<int>(rank) * kCtaM;
        const int n0 = tc.n_blk * BN + static_cast<int>(rank) * (BN / 2);
        const int kend = k1 < 0 ? d.num_k : k1;
        for (int k = k0; k < kend; ++k) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, tmo, abort_flag, kSiteProducerEmpty))
            return false;
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * L::kStageBytes);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const int r0 = cp.kl * kBK;
          if (d.a_3d) {
            tma_load_3d_pair(a_tile(stage), ma, fb, 0, r0, m0 / 64, pol_a);
          } else
#pragma unroll
          for (int hh = 0; hh < MH; ++hh) {
            const uint32_t at = a_tile(stage) + hh * L::kAHalfBytes;
            if (d.a_mn) {
              tma_load_2d_pair(at, ma, fb, m0 + 128 * hh, r0, pol_a);
              tma_load_2d_pair(at + kBK * 128, ma, fb, m0 + 128 * hh + 64, r0, pol_a);
            } else {
              tma_load_2d_pair(at, ma, fb, r0, m0 + 128 * hh, pol_a);
            }
          }
          if (d.b_3d) {
            tma_load_3d_pair(b_tile(stage), mb, fb, 0, r0, n0 / 64, pol_b);
          } else if (d.b_mn) {
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d_pair(b_tile(stage) + h * (kBK * 128), mb, fb, n0 + 64 * h, r0, pol_b);
          } else {
            tma_load_2d_pair(b_tile(stage), mb, fb, r0, n0, pol_b);
          }
          if (chain_next(P, d, cp)) {
            ma = &P.tma[d.map0 + cp.g];
            mb = &P.tmb[d.map0 + cp.g];
          }
          ++loads;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      });
      // Every load of this CTA is issued: the next kernel may begin its
      // set-up on SMs as they free up.
      griddep_launch_dependents();
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
      for_each_work(P, pair, num_pairs, [&](int t, int k0, int k1, int) -> bool {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        const int kend = k1 < 0 ? d.num_k : k1;
        if (kend <= k0) return true;
        const uint32_t b = acc % kAccBufs;
        const uint32_t acc_phase = (acc / kAccBufs) & 1u;
        if (!wait_bounded(tempty_bar(b), acc_phase ^ 1u, tmo, abort_flag, kSiteMmaTmemEmpty)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kAccCols;
        for (int k = k0; k < kend; ++k) {
          if (!wait_bounded(full_bar(stage), phase, tmo, abort_flag, kSiteMmaFull)) return false;
          tc_fence_after();
          const uint32_t sa = a_tile(stage);
          const uint32_t sb = b_tile(stage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = operand_desc<kBK>(sb, kk, d.b_mn);
#pragma unroll
            for (int hh = 0; hh < MH; ++hh) {
              const uint64_t ad = operand_desc<kBK>(sa + hh * L::kAHalfBytes, kk, d.a_mn);
              umma_bf16_pair(d_tmem + hh * kHalfCols, ad, bd, d.idesc,
                             (k != k0 || kk != 0) ? 1u : 0u);
            }
          }
          umma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit_pair_mc(tfull_bar(b), 0x3);
        ++acc;
        return true;
      });
      umma_commit_pair(mma_done_bar);
      wait_bounded(mma_done_bar, 0, tmo, abort_flag, kSiteDrainMma, false);
    }
  } else if (warp >= epi_first_warp<MH, kSplit>()) {
    grow_registers<MH, kSplit>();
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int hh = (warp - epi_first_warp<MH, kSplit>()) >> 2;  // row half it drains
    uint32_t acc = 0;
    for_each_work(P, pair, num_pairs, [&](int t, int k0, int k1, int kind) -> bool {
      const TileCoord tc = decode_tile(P, t);
      const ProblemDesc& d = P.prob[tc.p];
      const int row =
          tc.m_blk * kTileM + static_cast<int>(rank) * kCtaM + hh * 128 + q * 32 + lane;
      const int n0 = tc.n_blk * BN;
      if ((k1 < 0 ? d.num_k : k1) <= k0) {
        if (row < d.M) store_zero_row(d, row, n0, BN);
        return true;
      }
      const uint32_t b = acc % kAccBufs;
      const uint32_t acc_phase = (acc / kAccBufs) & 1u;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull_bar(b), acc_phase, tmo, abort_flag, kSiteEpiTmemFull);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) return false;
      tc_fence_after();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kAccCols + hh * kHalfCols;
      epilogue_item<BN>(P, d, kind, pair,
                        static_cast<int>(rank) * kEpiWarps * MH + (warp - epi_first_warp<MH, kSplit>()),
                        tc.m_blk * kTileM, n0, t_row, row,
                        leader ? tempty_bar(b) : mapa_shared(tempty_bar(b), 0), !leader);
      ++acc;
      return true;
    });
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
