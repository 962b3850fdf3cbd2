// Persistent, warp-specialised bf16 GEMM on the sm_103a tensor cores, with an
// epilogue that can fold in earlier fp32 partial products (the fixed-order
// reduction of 3D-grid partials and of split reduction ranges).
//
//   C[M x N] (op)= A[M x R] . B[R x N]      bf16 in, fp32 accumulate in TMEM
//
// One launch processes a list of independent "problems" (one per block
// product of the 3D grid, or a single full-layer GEMM).  Every problem has
// its own pair of TMA tensor maps whose extents are the block's own extents,
// so tile boxes that run past a block edge read zeros exactly as a GPU that
// held only that shard would.
//
// One CTA per SM, persistent over a static tile schedule:
//   warp 0      TMA producer (one thread): smem ring of STAGES x (A | B) tiles
//   warp 1      TMEM owner + MMA issuer (one thread): tcgen05.mma 128 x BN x 16
//   epilogue    4 warps per 128-row half: tcgen05.ld -> fp32 -> bf16 RNE (or
//               fp32) -> global
// The accumulator is double-buffered in TMEM (2 x BN columns) so the epilogue
// of tile i overlaps the mainloop of tile i+1.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records an error word in device memory, all roles leave their loops, the
// producer's outstanding copies and the issued MMAs are drained (each drain
// bounded too) and TMEM is released before the CTA exits.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace axonn {

constexpr int kBM = 128;       // rows of one UMMA (cta_group::1)
constexpr int kBK = 64;        // reduction depth per stage of the CTA-pair kernel
constexpr int kEpiWarps = 4;

// A CTA may own MH row halves of 128 (an MH*128 x BN tile).  Warp roles:
//   MH = 1:            6 warps: producer, MMA issuer, 4 epilogue warps (2..5).
//   MH = 2:           10 warps: producer, MMA issuer, 8 epilogue warps (2..9).
//   MH = 2, SPLIT:    12 warps in 3 warpgroups: warpgroup 0 holds the producer
//                     (warp 0) and the MMA issuer (warp 1) and gives registers
//                     to warpgroups 1 and 2 (setmaxnreg), which drain row
//                     halves 0 and 1 holding a whole bf16 accumulator row of
//                     up to 128 words per thread.
// The split is used only where it measures faster (the CTA-pair kernel with
// 256-column tiles); in the single-CTA kernel it slowed the operand supply.
template <int MH, bool SPLIT = false>
constexpr int cta_threads() { return MH == 1 ? 192 : (SPLIT ? 384 : 320); }
template <int MH, bool SPLIT = false>
constexpr int epi_first_warp() { return MH == 2 && SPLIT ? 4 : 2; }
constexpr int kRegsAtLaunch = 168;  // 384 threads, one CTA per SM
constexpr int kRegsControl = 56;    // warpgroup 0 after the split
constexpr int kRegsEpilogue = 224;  // warpgroups 1 and 2 after the split
static_assert(128 * kRegsControl + 256 * kRegsEpilogue <= 384 * kRegsAtLaunch,
              "register split exceeds the launch allocation");

// Register split of a 12-warp CTA (no-ops otherwise), made inside each
// role's branch so that the compiler allocates each branch for its budget.
template <int MH, bool SPLIT>
__device__ __forceinline__ void shrink_registers() {
  if constexpr (MH == 2 && SPLIT) setmaxnreg_dec<kRegsControl>();
}
template <int MH, bool SPLIT>
__device__ __forceinline__ void grow_registers() {
  if constexpr (MH == 2 && SPLIT) setmaxnreg_inc<kRegsEpilogue>();
}

// Output modes of the epilogue.  kOutF32Red adds the tile into an fp32
// output with atomic adds, for products of which several write the same
// output rows in one launch (the grid's partial products summed in no fixed
// order).
enum OutMode : int32_t { kOutBF16 = 0, kOutF32 = 1, kOutF32Accum = 2, kOutF32Red = 3 };

struct ProblemDesc {
  void* C;            // output base (element (0,0) of this problem)
  int64_t ldc;        // output row stride, elements
  int32_t M, N, R;    // problem extents
  int32_t tiles_m, tiles_n;
  int32_t tile_start;  // first global tile index of this problem
  int32_t num_k;       // ceil(R / kBK)
  uint32_t idesc;      // tcgen05 instruction descriptor
  int32_t a_mn;        // A stored M-contiguous (else R-contiguous)
  int32_t b_mn;        // B stored N-contiguous (else R-contiguous)
  int32_t out_mode;
  int32_t red_count;      // > 0: add red_count fp32 partials before storing
  const float* red_src;   // partial 0 of this problem's output, element (0,0)
  int64_t red_stride;     // elements between consecutive partials
  int64_t red_ld;         // row stride of a partial, elements
  int32_t a_3d, b_3d;     // MN-major operand whose tile comes in one 3-D box
  int32_t fast_bf16;      // bf16 output, no partials, every row 32-byte aligned
  // The reduction of every tile runs through `chain` block products in
  // order, tensor-map pairs map0 .. map0+chain-1 (map_nk[] steps each), all
  // into one accumulator: the virtual grid's sum over the reduced axis kept
  // in TMEM.  chain = 1 for a single product.  num_k is the chain's total.
  int32_t chain;
  int32_t map0;
  // The problem computes the transpose of the caller's product (operand
  // roles swapped, C^T = B^T . A^T): its tile element (i, j) is the
  // caller's output element (j, i), stored at C + j * ldc + i.
  int32_t out_t;
  // L2 priorities of the operand loads: l2_keep = 1 keeps A's lines (a
  // fraction l2_keep_frac of them evict-last), 2 keeps B's, 0 neither; the
  // other operand loads at the default priority.  A rasterisation group
  // walks its tile rows (or columns) across the whole product, so the
  // group's panel of the one operand is read again by every later wave of
  // the group while the other operand's panels pass through once.
  int32_t l2_keep;
  float l2_keep_frac;
};

template <int MAXP>
struct GemmParams {
  CUtensorMap tma[MAXP];  // A operand of each block product (map index)
  CUtensorMap tmb[MAXP];  // B operand of each block product
  int32_t map_nk[MAXP];   // 64-deep reduction steps of each block product
  ProblemDesc prob[MAXP];
  int32_t num_problems;
  int32_t num_maps;
  int32_t total_tiles;
  int32_t group_m;     // tile rows per rasterisation group
  int32_t inject;      // test-only: 1 = the producer withholds every load
  uint64_t timeout_ns; // bound on any single mbarrier wait
  // Stream-K tail (single-problem launches only; sk_tiles = 0 disables it).
  // The last sk_tiles tiles of the tile order are not given whole to CTAs:
  // their sk_tiles * num_k reduction steps are cut into gridDim equal,
  // consecutive ranges, one per CTA (or CTA pair).  sk_tiles >= gridDim, so
  // a range covers at least one tile and each tile is cut into at most two
  // pieces: a head (steps 0..k1) at the end of unit u's range and a tail
  // (k1..num_k) at the start of unit u+1's.  How the two are summed is in
  // epilogue_item.
  int32_t sk_tiles;
  int32_t sk_slot_floats;  // floats per partial slot (one tile)
  float* sk_partials;      // 2 slots per unit (CTA or CTA pair)
  uint32_t* sk_flags;      // kSkCountersPerUnit counters per unit, zero at launch
};

// Kinds of work item: a whole tile, or the head or tail piece of a stream-K
// tile (see GemmParams).
enum WorkKind : int { kWhole = 0, kHead = 1, kTail = 2 };

// Calls f(t, k0, k1, kind) for each work item of unit `u` of `units` (a CTA,
// or a CTA pair), in order, until f returns false: first the whole tiles
// u, u + units, ... below the stream-K tiles (k0 = 0, k1 = -1 meaning the
// tile's own num_k), then the unit's range of stream-K steps.  Every role of
// a unit walks the same sequence.  The whole-tile rounds are a plain strided
// loop: with the item's bounds known at that call site, the roles' loops
// compile as they do without stream-K (an iterator object there slowed the
// producer's issue loop by 14 %).  The host keeps sk_tiles * num_k below
// 2^31.
//
// The reduction-split kernel (kSplit) walks instead the tiles c, c + C, ...
// of its cluster c (C clusters), this CTA taking piece `rank` of each: steps
// [nk rank / S, nk (rank + 1) / S) of S, S the cluster's size.
template <bool kSplit = false, int MAXP, typename F>
__device__ __forceinline__ void for_each_work(const GemmParams<MAXP>& P, int u, int units, F&& f) {
  if constexpr (kSplit) {
    const int S = static_cast<int>(cluster_nctarank());
    const int rank = static_cast<int>(cluster_ctarank());
    const int nk = P.prob[0].num_k;
    const int k0 = nk * rank / S, k1 = nk * (rank + 1) / S;
    const int nc = static_cast<int>(num_clusters_x());
    for (int t = static_cast<int>(cluster_id_x()); t < P.total_tiles; t += nc)
      if (!f(t, k0, k1, kWhole)) return;
    return;
  }
  const int dp_end = P.total_tiles - P.sk_tiles;
  for (int t = u; t < dp_end; t += units)
    if (!f(t, 0, -1, kWhole)) return;
  if (P.sk_tiles == 0) return;
  const int nk = P.prob[0].num_k;
  const int64_t steps = static_cast<int64_t>(P.sk_tiles) * nk;
  int s = static_cast<int>(steps * u / units);
  const int s_end = static_cast<int>(steps * (u + 1) / units);
  while (s < s_end) {
    const int st = s / nk;
    const int k0 = s - st * nk;
    const int k1 = min(nk, k0 + (s_end - s));
    const int kind = (k0 == 0 && k1 == nk) ? kWhole : (k0 == 0 ? kHead : kTail);
    if (!f(dp_end + st, k0, k1, kind)) return;
    s += k1 - k0;
  }
}

// Device-side error word: 0 = no error.  Layout of a timeout record:
// bits 32..39 = 0x7E, bits 8..31 = CTA index, bits 0..7 = wait site.  Each
// translation unit that instantiates kernels has its own copy (no
// relocatable device code); the host reads them through kernels_take_status.
__device__ unsigned long long g_status_word;

enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiTmemFull = 4,
  kSiteDrainLoads = 5,
  kSiteDrainMma = 6,
  kSiteSplitFree = 7,
  kSiteSplitInbox = 8,
  kSiteSplitStaged = 9,
};

__device__ __forceinline__ void record_timeout(uint32_t site) {
  const unsigned long long code =
      (0x7EULL << 32) | (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 8) | site;
  atomicCAS(&g_status_word, 0ULL, code);
}

// Bounded wait on the phase of `bar` with the given parity.  Returns false
// if the limit passed (error recorded, CTA abort flag raised) or, when
// `honor_abort` is set, another role of this CTA aborted first.  Drains of
// in-flight copies and MMAs pass honor_abort = false: they must wait for the
// hardware even after an abort, still within the limit.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             volatile int* abort_flag, uint32_t site,
                                             bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    // Suspended up to 20 us per poll: epilogue warps wait most of a tile,
    // and fewer issued instructions leave more of the power budget to the
    // tensor cores.  The limit and abort checks still run every poll.
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (honor_abort && *abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      record_timeout(site);
      return false;
    }
  }
}

// Bounded wait that polls without ever suspending the thread, for the
// reduction split's waits, which are short and on its critical path: a
// warp whose thread has come back from a suspending try_wait was measured
// to run the code after it several times slower for thousands of cycles
// (the split's band sums, on GB300).  `cluster` gives the test acquire
// semantics at cluster scope (a phase completed by other CTAs).  The clock
// and abort flag are read every 256 polls.
template <bool kCluster>
__device__ __forceinline__ bool wait_polling(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             volatile int* abort_flag, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (kCluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      record_timeout(site);
      return false;
    }
  }
}

struct TileCoord {
  int p, m_blk, n_blk;
};

// Where reduction step k of a problem falls in its chain of block products:
// member g, step kl of that member's nk steps.
struct ChainPos {
  int g, kl, nk;
};

template <int MAXP>
__device__ __forceinline__ ChainPos chain_start(const GemmParams<MAXP>& P, const ProblemDesc& d,
                                                int k) {
  ChainPos c{0, k, P.map_nk[d.map0]};
#pragma unroll 1
  while (c.g + 1 < d.chain && c.kl >= c.nk) {
    c.kl -= c.nk;
    ++c.g;
    c.nk = P.map_nk[d.map0 + c.g];
  }
  return c;
}

// Moves to the next reduction step; true when it starts the next member
// (whose tensor maps the producer then loads from).
template <int MAXP>
__device__ __forceinline__ bool chain_next(const GemmParams<MAXP>& P, const ProblemDesc& d,
                                           ChainPos& c) {
  if (++c.kl < c.nk || c.g + 1 >= d.chain) return false;
  ++c.g;
  c.kl = 0;
  c.nk = P.map_nk[d.map0 + c.g];
  return true;
}

template <int MAXP>
__device__ __forceinline__ TileCoord decode_tile(const GemmParams<MAXP>& P, int t) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < P.num_problems && t >= P.prob[p + 1].tile_start) ++p;
  const ProblemDesc& d = P.prob[p];
  const int lt = t - d.tile_start;
  // Grouped rasterisation, so that concurrently running CTAs share operand
  // panels in L2.  group_m > 0: walk group_m tile rows down one tile column
  // before moving right.  group_m < 0: walk -group_m tile columns along one
  // tile row before moving down.
  TileCoord c;
  c.p = p;
  if (P.group_m > 0) {
    const int per_group = P.group_m * d.tiles_n;
    const int group = lt / per_group;
    const int first_m = group * P.group_m;
    const int gsize = min(P.group_m, d.tiles_m - first_m);
    const int in_group = lt - group * per_group;
    c.m_blk = first_m + in_group % gsize;
    c.n_blk = in_group / gsize;
  } else {
    const int gn = -P.group_m;
    const int per_group = gn * d.tiles_m;
    const int group = lt / per_group;
    const int first_n = group * gn;
    const int gsize = min(gn, d.tiles_n - first_n);
    const int in_group = lt - group * per_group;
    c.n_blk = first_n + in_group % gsize;
    c.m_blk = in_group / gsize;
  }
  return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
  __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&v);
}

// Sum, in order, the fp32 partials 0..red_count-1 of 32 columns of one row
// and then this problem's own accumulator: the fixed-order reduction of the
// grid's partial products, fused into the epilogue of the last one.
__device__ __forceinline__ void add_partials(const ProblemDesc& d, int row, int col0, int ncols,
                                             uint32_t (&r)[32]) {
  float s[32];
  const float* src = d.red_src + row * d.red_ld + col0;
  if (ncols == 32) {
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 a = reinterpret_cast<const float4*>(src)[v];
      s[4 * v] = a.x; s[4 * v + 1] = a.y; s[4 * v + 2] = a.z; s[4 * v + 3] = a.w;
    }
    for (int g = 1; g < d.red_count; ++g) {
      const float* pg = src + g * d.red_stride;
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 a = reinterpret_cast<const float4*>(pg)[v];
        s[4 * v] += a.x; s[4 * v + 1] += a.y; s[4 * v + 2] += a.z; s[4 * v + 3] += a.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) s[j] = j < ncols ? src[j] : 0.0f;
    for (int g = 1; g < d.red_count; ++g)
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncols) s[j] += src[g * d.red_stride + j];
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(s[j] + __uint_as_float(r[j]));
}

// Writes 16 packed bf16 pairs, columns [col0, col0+32) of one output row.
// Each thread writes its own row, so a warp's store instruction touches 32
// rows: 32-byte stores (whole L2 sectors) take half the time of 16-byte ones
// and are used whenever the address is 32-byte aligned.
__device__ __forceinline__ void store_bf16_32(const ProblemDesc& d, int row, int col0,
                                              const uint32_t* pk) {
  const int ncols = min(32, d.N - col0);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(d.C) + row * d.ldc + col0;
  if (ncols == 32) {
    if ((reinterpret_cast<uintptr_t>(out) & 31u) == 0) {
      st_global_v8(out, pk);
      st_global_v8(out + 16, pk + 8);
    } else {
#pragma unroll
      for (int v = 0; v < 4; ++v)
        reinterpret_cast<uint4*>(out)[v] =
            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  } else {
    unsigned short* o16 = reinterpret_cast<unsigned short*>(out);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < ncols) o16[j] = static_cast<unsigned short>((pk[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu);
  }
}

// Writes 32 accumulator columns of a transposed problem: tile row `row` is
// output column `row`, tile column col0 + j is output row col0 + j.  The
// warp's lanes hold consecutive tile rows, so each store instruction writes
// 32 consecutive elements of one output row.
__device__ __forceinline__ void store_chunk_t(const ProblemDesc& d, int row, int col0, int ncols,
                                              const uint32_t (&r)[32]) {
  if (d.out_mode == kOutBF16) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(d.C) + row;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < ncols) out[static_cast<int64_t>(col0 + j) * d.ldc] = __float2bfloat16_rn(__uint_as_float(r[j]));
  } else {
    float* out = reinterpret_cast<float*>(d.C) + row;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j >= ncols) continue;
      float* o = out + static_cast<int64_t>(col0 + j) * d.ldc;
      if (d.out_mode == kOutF32Red || d.out_mode == kOutF32Accum) red_add_f32(o, r[j]);
      else *o = __uint_as_float(r[j]);
    }
  }
}

// Writes 32 accumulator columns [col0, col0+32) of one output row.
__device__ __forceinline__ void store_chunk(const ProblemDesc& d, int row, int col0,
                                            uint32_t (&r)[32]) {
  const int ncols = min(32, d.N - col0);
  if (d.red_count > 0) add_partials(d, row, col0, ncols, r);
  if (d.out_t) {
    store_chunk_t(d, row, col0, ncols, r);
    return;
  }
  if (d.out_mode == kOutBF16) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(r[2 * j], r[2 * j + 1]);
    store_bf16_32(d, row, col0, pk);
  } else {
    float* out = reinterpret_cast<float*>(d.C) + row * d.ldc + col0;
    if (d.out_mode == kOutF32Red || d.out_mode == kOutF32Accum) {
      // 16-byte vector reductions (row stride and column offset keep every
      // 4-column group 16-byte aligned).  They return nothing, so the warp
      // issues them and moves on, and the L2 performs the adds: an
      // accumulating tile never waits for the old output.  With one writer
      // per element (kOutF32Accum) the result is the single rounded sum of
      // the old value and the tile's, as a load-add-store would give (up to
      // the reduction's flush of subnormals to zero).
      if (ncols == 32) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          red_add_v4_f32(out + 4 * v, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncols) red_add_f32(out + j, r[j]);
      }
    } else if (ncols == 32 && (reinterpret_cast<uintptr_t>(out) & 31u) == 0) {
#pragma unroll
      for (int v = 0; v < 4; ++v) st_global_v8(out + 8 * v, &r[8 * v]);
    } else if (ncols == 32) {
#pragma unroll
      for (int v = 0; v < 8; ++v)
        reinterpret_cast<float4*>(out)[v] =
            make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncols) out[j] = __uint_as_float(r[j]);
    }
  }
}

// Row of a tile whose reduction range is empty: the product is zero (plus
// any partials to add).
__device__ __forceinline__ void store_zero_row(const ProblemDesc& d, int row, int n0, int BN) {
  // nothing to add into an accumulating output: leave it as it is
  if ((d.out_mode == kOutF32Accum || d.out_mode == kOutF32Red) && d.red_count == 0) return;
  for (int col0 = n0; col0 < min(d.N, n0 + BN); col0 += 32) {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = 0u;
    store_chunk(d, row, col0, r);
  }
}

// Epilogue of one warp: its 32 accumulator rows x BN columns (TMEM lanes
// of t_row) to global memory, then one arrive on `tempty` by the lanes with
// `arrive` set (a shared::cluster address of the peer CTA's barrier when
// `remote`).  A plain bf16 tile that lies wholly inside the output is first
// packed into registers (BN / 2 words per thread) and TMEM is released
// before any store, so the next tile's MMAs start while the stores drain;
// its rows are stored as 32-byte vectors.  With kTransFast a transposed
// bf16 tile (operand roles exchanged) whose warp rows and columns all lie
// inside a 4-byte-aligned output does the same and stores column pairs as
// 32-bit words.  Other tiles (partials to add, fp32 output, ragged edges,
// misaligned rows) are stored chunk by chunk and release TMEM afterwards.
template <int BN, bool kTransFast>
__device__ __forceinline__ void drain_accumulator(const ProblemDesc& d, uint32_t t_row, int row,
                                                  int n0, uint32_t tempty, bool arrive,
                                                  bool remote) {
  if (d.fast_bf16 && n0 + BN <= d.N) {
    uint32_t pk[BN / 2];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[16 * c + j] = cvt_bf16x2_ordered(r[2 * j], r[2 * j + 1]);
    }
    tc_fence_before();
    __syncwarp();
    if (arrive) {
      if (remote) mbar_arrive_cluster(tempty);
      else mbar_arrive(tempty);
    }
    if (row < d.M) {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(d.C) + row * d.ldc + n0;
#pragma unroll
      for (int v = 0; v < BN / 16; ++v) st_global_v8(out + 16 * v, &pk[8 * v]);
    }
    return;
  }
  if (kTransFast && d.out_t && d.out_mode == kOutBF16 && d.red_count == 0 && n0 + BN <= d.N &&
      (row | 31) < d.M &&
      ((reinterpret_cast<uintptr_t>(d.C) & 3) | (d.ldc & 1)) == 0) {
    // Transposed bf16 output (exchanged operand roles): as above, the row is
    // packed in registers and TMEM released before any store, so the next
    // tile's MMAs do not wait for the stores.  Accumulator column j is output
    // row n0 + j.  Lanes 2i and 2i+1 (adjacent accumulator rows) swap their
    // packed column pairs, after which the even lane holds column 2w of both
    // rows and the odd lane column 2w+1: one 32-bit store each per pair of
    // columns, the warp covering 64 consecutive bytes of two output rows.
    const int odd = row & 1;
    // even lane: (own low half, partner's low half); odd: (partner's high, own high)
    const uint32_t sel = odd ? 0x3276u : 0x5410u;
    uint32_t pk[BN / 2];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t mine = cvt_bf16x2_ordered(r[2 * j], r[2 * j + 1]);
        pk[16 * c + j] = __byte_perm(mine, __shfl_xor_sync(0xffffffffu, mine, 1), sel);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (arrive) {
      if (remote) mbar_arrive_cluster(tempty);
      else mbar_arrive(tempty);
    }
    const int64_t ld = d.ldc;
    uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned short*>(d.C) +
                                                (n0 + odd) * ld + (row - odd));
#pragma unroll
    for (int w = 0; w < BN / 2; ++w) {
      *out = pk[w];
      out += ld;  // two output rows of 16-bit elements
    }
    return;
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int col0 = n0 + c * 32;
    if (col0 >= d.N) break;
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c * 32, r);
    tmem_ld_wait();
    if (row < d.M) store_chunk(d, row, col0, r);
  }
  tc_fence_before();
  __syncwarp();
  if (arrive) {
    if (remote) mbar_arrive_cluster(tempty);
    else mbar_arrive(tempty);
  }
}

// Counters per unit for the stream-K pieces: one per epilogue warp of the
// unit (up to 2 CTAs x 8 warps).
constexpr int kSkCountersPerUnit = 16;

// Epilogue of one work item (see for_each_work) by one warp, which owns 32
// rows of the tile (its TMEM lane quarter of one row half).  Whole tiles go
// to the output.  The two pieces of a stream-K tile never wait for each
// other.  Each piece first stores its rows of the accumulator, in fp32, to
// its own partial slot: the head in slot 2u+1 of its unit u, the tail in
// slot 2(u+1) of the next unit.  TMEM stays held.  Then the warp adds one to
// the counter of its rows (counter index: the head's unit, this warp's
// place `warp_slot` in the unit).  The warp that finds the other piece
// already counted adds the other piece's partial to its own accumulator
// and stores the output rows.  Two fp32 terms sum to the same value in
// either order, so the output does not depend on which piece comes second.
// Co-residency of the units is not needed, so launches on other streams
// cannot stall it.
template <int BN, int MAXP, bool kTransFast = true>
__device__ __forceinline__ void epilogue_item(const GemmParams<MAXP>& P, const ProblemDesc& d,
                                              int kind, int unit, int warp_slot, int tile_m0,
                                              int n0, uint32_t t_row, int row, uint32_t tempty,
                                              bool remote) {
  const int lane = threadIdx.x & 31;
  if (kind == kWhole) {
    drain_accumulator<BN, kTransFast>(d, t_row, row, n0, tempty, lane == 0, remote);
    return;
  }
  const bool head = kind == kHead;
  const int head_unit = head ? unit : unit - 1;
  const int64_t origin = static_cast<int64_t>(tile_m0) * BN + n0;
  float* mine = P.sk_partials + static_cast<int64_t>(2 * unit + (head ? 1 : 0)) * P.sk_slot_floats;
  const float* other =
      P.sk_partials + static_cast<int64_t>(head ? 2 * (unit + 1) : 2 * (unit - 1) + 1) * P.sk_slot_floats;
  // 1. this piece's rows, fp32, to its slot (tile-local, BN floats a row)
  ProblemDesc dp = d;
  dp.C = mine - origin;
  dp.ldc = BN;
  dp.out_mode = kOutF32;
  dp.red_count = 0;
  dp.fast_bf16 = 0;
  dp.out_t = 0;  // partial slots are tile-local, in the problem's own orientation
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int col0 = n0 + c * 32;
    if (col0 >= d.N) break;
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c * 32, r);
    tmem_ld_wait();
    if (row < d.M) store_chunk(dp, row, col0, r);
  }
  // 2. count this warp's rows as done; the second piece finishes them
  __threadfence();
  __syncwarp();
  uint32_t before = 0;
  if (lane == 0) before = atomicAdd(&P.sk_flags[head_unit * kSkCountersPerUnit + warp_slot], 1u);
  before = __shfl_sync(0xFFFFFFFFu, before, 0);
  __syncwarp();
  if (before == 1u) {
    __threadfence();
    ProblemDesc ds = d;
    ds.fast_bf16 = 0;
    ds.red_count = 1;
    ds.red_src = other - origin;
    ds.red_ld = BN;
    ds.red_stride = 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = n0 + c * 32;
      if (col0 >= d.N) break;
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c * 32, r);
      tmem_ld_wait();
      if (row < d.M) store_chunk(ds, row, col0, r);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (remote) mbar_arrive_cluster(tempty);
    else mbar_arrive(tempty);
  }
}

// Four consecutive output columns col..col+3 of one row (the reduction
// split's epilogue): one vector access where all four exist and the address
// allows it, else one per column.  Rounding and output modes as store_chunk,
// transposed (out_t) as store_chunk_t.
__device__ __forceinline__ void store_quad(const ProblemDesc& d, int row, int col, float4 v) {
  const int n = min(4, d.N - col);
  const float x[4] = {v.x, v.y, v.z, v.w};
  if (d.out_t) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j >= n) continue;
      const int64_t at = static_cast<int64_t>(col + j) * d.ldc + row;
      if (d.out_mode == kOutBF16) {
        reinterpret_cast<__nv_bfloat16*>(d.C)[at] = __float2bfloat16_rn(x[j]);
      } else {
        float* o = reinterpret_cast<float*>(d.C) + at;
        if (d.out_mode == kOutF32Red || d.out_mode == kOutF32Accum) red_add_f32(o, __float_as_uint(x[j]));
        else *o = x[j];
      }
    }
    return;
  }
  if (d.out_mode == kOutBF16) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(d.C) + row * d.ldc + col;
    if (n == 4 && (reinterpret_cast<uintptr_t>(o) & 7u) == 0) {
      __stwb(reinterpret_cast<uint2*>(o), make_uint2(pack_bf16x2(__float_as_uint(v.x), __float_as_uint(v.y)),
                                                     pack_bf16x2(__float_as_uint(v.z), __float_as_uint(v.w))));
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < n) o[j] = __float2bfloat16_rn(x[j]);
    }
    return;
  }
  float* o = reinterpret_cast<float*>(d.C) + row * d.ldc + col;
  const bool add = d.out_mode == kOutF32Red || d.out_mode == kOutF32Accum;
  if (n == 4 && (reinterpret_cast<uintptr_t>(o) & 15u) == 0) {
    if (add)
      red_add_v4_f32(o, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                     __float_as_uint(v.w));
    else
      *reinterpret_cast<float4*>(o) = v;
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j >= n) continue;
    if (add) red_add_f32(o + j, __float_as_uint(x[j]));
    else o[j] = x[j];
  }
}

// The reduction split's band sum for S pieces (S a compile-time constant,
// so that all S loads of a row are issued before the adds): warp q takes
// band rows q, q + 4, ...; a lane four consecutive columns.  Piece g's rows
// are this CTA's staged rows when g == me, else block g (g < me) or g - 1
// (g > me) of the inbox (shared-memory addresses); rows are kLd floats
// apart.  The sum runs over
// pieces 0, 1, ..., S-1 in that order.
template <int S, int BN, int kLd>
__device__ __forceinline__ void split_band_sum(uint32_t own, uint32_t inboxed, int me, int q,
                                               int lane, int row0, int n0, const ProblemDesc& od) {
  constexpr int band = kBM / S;
  const bool bf16_rows = od.out_mode == kOutBF16 && !od.out_t;
  for (int i = q; i < band; i += kEpiWarps) {
    const int row = row0 + i;
    if (row >= od.M) break;
#pragma unroll
    for (int cb = 0; cb < BN; cb += 128) {
      const int col = cb + 4 * lane;
      if (col >= BN || n0 + col >= od.N) continue;
      float4 x[S];
#pragma unroll
      for (int g = 0; g < S; ++g) {
        const int at = g == me ? i * kLd + col : ((g < me ? g : g - 1) * band + i) * kLd + col;
        x[g] = ld_shared_v4((g == me ? own : inboxed) + static_cast<uint32_t>(at * 4));
      }
      float4 a = x[0];
#pragma unroll
      for (int g = 1; g < S; ++g) {
        a.x += x[g].x;
        a.y += x[g].y;
        a.z += x[g].z;
        a.w += x[g].w;
      }
      // bf16 rows with all four columns present and the address aligned:
      // one 8-byte store (measured a third cheaper than store_quad's
      // general path here); the other cases through store_quad.
      __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(od.C) + row * od.ldc + n0 + col;
      if (bf16_rows && n0 + col + 4 <= od.N && (reinterpret_cast<uintptr_t>(o) & 7u) == 0)
        *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(__float_as_uint(a.x), __float_as_uint(a.y)),
                                                  pack_bf16x2(__float_as_uint(a.z), __float_as_uint(a.w)));
      else
        store_quad(od, row, n0 + col, a);
    }
  }
}

// kSplit adds the reduction split's staging tile (this piece's 128 x BN
// fp32 rows, each padded by 16 bytes so that a warp's row-per-lane stores
// and row-wise loads meet no bank conflict), its inbox (the other pieces'
// rows of this CTA's band: at most 7 bands of 16 rows, or 1 of 64, i.e.
// 128 - 128/S rows for S = 2, 4, 8) and three barriers.
constexpr int kSplitMaxPieces = 8;
template <int BN, int BK, int STAGES, int MH = 1, bool kSplit = false>
struct SmemLayout {
  static constexpr int kAHalfBytes = kBM * BK * 2;
  static constexpr int kABytes = MH * kAHalfBytes;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSplitLd = BN + 4;  // floats per staged row
  static constexpr int kStagingBytes = kSplit ? kBM * kSplitLd * 4 : 0;
  static constexpr int kInboxBytes = kSplit ? (kBM - kBM / kSplitMaxPieces) * kSplitLd * 4 : 0;
  static constexpr int kNumBars = 2 * STAGES + 5 + (kSplit ? 3 : 0);
  // 1024 B of slack for aligning the tile ring, the ring, the staging tile
  // and inbox, barriers, TMEM slot and the abort flag.
  static constexpr int kBytes =
      1024 + STAGES * kStageBytes + kStagingBytes + kInboxBytes + kNumBars * 8 + 16;
};

// Shared-memory descriptor of the K=16 slice kk of a stage's operand tile.
// K-major tiles hold rows of BK elements (128 B with 128-byte swizzle for
// BK = 64, 64 B with 64-byte swizzle for BK = 32); MN-major tiles hold
// 64-element MN chunks of BK rows of 128 B, BK * 128 bytes apart.
template <int BK>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile, int kk, bool mn_major) {
  if (mn_major) return sdesc_sw128(tile + kk * 2048, BK * 128, 1024);
  if (BK == 64) return sdesc_sw128(tile + kk * 32, 16, 1024);
  return sdesc_sw64(tile + kk * 32, 16, 512);
}

// MH = 1: 128 x BN tiles, accumulator double-buffered in TMEM (2 x BN
// columns), so the epilogue of a tile overlaps the next mainloop.
// MH = 2: 256 x BN tiles as two M = 128 MMAs sharing each B slice (a third
// fewer operand bytes per FLOP); the two accumulators fill TMEM (2 x BN
// columns, single-buffered) and 8 epilogue warps drain them.
//
// kSplit (MH = 1, one problem): the reduction split.  The launch is made
// of clusters of S CTAs (S = 2, 4 or 8); a cluster owns whole tiles and its
// CTA of rank p computes piece p of each (see for_each_work) into TMEM.  The
// 128 rows of a tile are dealt out in S bands of 128/S, band o finished by
// CTA o.  Each CTA pushes its piece's rows, fp32, into the inbox of the
// band's CTA (st.async into that CTA's shared memory, counted in bytes on
// its inbox barrier), at block p of that inbox.  Once its inbox is full a
// CTA adds blocks 0, 1, ..., S-1 in that order -- the pieces in reduction
// order, whatever order they arrived in -- and writes its band to the
// output; then it tells every CTA of the cluster (their "free" barriers)
// that their blocks have been read and the inbox may take the next tile.
// No workspace and no second launch; pieces meet only inside the cluster,
// whose CTAs the hardware schedules together.
template <int BN, int BK, int STAGES, int MAXP, int MH = 1, bool kSplit = false>
__global__ void __launch_bounds__(cta_threads<MH>(), 1)
    fc_gemm_tcgen05_kernel(const __grid_constant__ GemmParams<MAXP> P) {
  using L = SmemLayout<BN, BK, STAGES, MH, kSplit>;
  static_assert(!kSplit || (MH == 1 && MAXP == 1), "reduction split: 128-row tiles, one problem");
  static_assert(BK == 64 || BK == 32, "stage depth");
  static_assert(MH == 1 || MH == 2, "row halves per CTA");
  constexpr int kAccBufs = MH == 1 ? 2 : 1;
  // Each row half's accumulator starts on a 128-column boundary of TMEM
  // (a 192-wide one takes 256 columns); TMEM is allocated in powers of two.
  constexpr uint32_t kHalfCols = BN <= 128 ? 128 : 256;
  constexpr uint32_t kAccCols = MH * kHalfCols;  // TMEM columns of one accumulator
  constexpr uint32_t kTmemUsed = kAccBufs * kAccCols;
  constexpr uint32_t kTmemCols = kTmemUsed <= 128 ? 128 : (kTmemUsed <= 256 ? 256 : 512);
  constexpr int kTileM = MH * kBM;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "UMMA N: 64, 128, 192 or 256");
  static_assert(kTmemUsed <= 512, "TMEM columns");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  uint8_t* ring_ptr = smem_raw + (ring - raw);
  // kSplit only: staging tile, then inbox, after the ring
  const uint32_t staging = ring + STAGES * L::kStageBytes;
  const uint32_t inbox = staging + L::kStagingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + STAGES * L::kStageBytes +
                                               L::kStagingBytes + L::kInboxBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // barrier indices
  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_addr(bars + 2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_addr(bars + 2 * STAGES + 2 + b); };
  const uint32_t mma_done_bar = smem_addr(bars + 2 * STAGES + 4);
  const uint32_t inbox_full = smem_addr(bars + 2 * STAGES + 5);  // kSplit only
  const uint32_t split_free = smem_addr(bars + 2 * STAGES + 6);  // kSplit only
  const uint32_t staged_bar = smem_addr(bars + 2 * STAGES + 7);  // kSplit only
  auto a_tile = [&](int s) { return ring + s * L::kStageBytes; };
  auto b_tile = [&](int s) { return ring + s * L::kStageBytes + L::kABytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps * MH);
    }
    mbar_init(mma_done_bar, 1);
    if constexpr (kSplit) {
      mbar_init(inbox_full, 1);
      mbar_init(split_free, kEpiWarps * cluster_nctarank());
      mbar_init(staged_bar, kEpiWarps);
    }
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
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The cluster's barriers exist before any CTA signals or stores into them.
  if constexpr (kSplit) cluster_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t tmo = P.timeout_ns;
  // The pipeline's waits: suspending ones, except in the reduction split,
  // whose pieces are a few stages long (see wait_polling).
  auto wait_pipe = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
    if constexpr (kSplit) return wait_polling<false>(bar, parity, tmo, abort_flag, site);
    else return wait_bounded(bar, parity, tmo, abort_flag, site);
  };
  // Barrier set-up, TMEM allocation and tensor-map prefetch above overlap
  // the previous kernel's tail; nothing below touches global memory before
  // that kernel is complete.
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && P.inject != 1) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t loads = 0;
      for_each_work<kSplit>(P, blockIdx.x, gridDim.x, [&](int t, int k0, int k1, int) -> bool {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        // L2 priorities of this tile's operand lines (see ProblemDesc)
        const uint64_t pol_a = l2_policy(d.l2_keep == 1, d.l2_keep_frac);
        const uint64_t pol_b = l2_policy(d.l2_keep == 2, d.l2_keep_frac);
        ChainPos cp = chain_start(P, d, k0);
        const CUtensorMap* ma = &P.tma[d.map0 + cp.g];
        const CUtensorMap* mb = &P.tmb[d.map0 + cp.g];
        const int m0 = tc.m_blk * kTileM;
        const int n0 = tc.n_blk * BN;
        const int kend = k1 < 0 ? d.num_k : k1;
        for (int k = k0; k < kend; ++k) {
          if (!wait_pipe(empty_bar(stage), phase ^ 1u, kSiteProducerEmpty)) return false;
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, L::kStageBytes);
          const int r0 = cp.kl * BK;
          // An MN-major tile is (rows or columns / 64) chunks of BK rows of
          // 128 B; with a 3-D tensor map {64, R, MN/64} one box brings all of
          // them (fewer TMA operations per stage), else one box per chunk.
          if (d.a_3d) {
            tma_load_3d(a_tile(stage), ma, fb, 0, r0, m0 / 64, pol_a);
          } else
#pragma unroll
          for (int hh = 0; hh < MH; ++hh) {
            const uint32_t at = a_tile(stage) + hh * L::kAHalfBytes;
            if (d.a_mn) {
#pragma unroll
              for (int h = 0; h < kBM / 64; ++h)
                tma_load_2d(at + h * (BK * 128), ma, fb, m0 + kBM * hh + 64 * h, r0, pol_a);
            } else {
              tma_load_2d(at, ma, fb, r0, m0 + kBM * hh, pol_a);
            }
          }
          if (d.b_3d) {
            tma_load_3d(b_tile(stage), mb, fb, 0, r0, n0 / 64, pol_b);
          } else if (d.b_mn) {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_2d(b_tile(stage) + h * (BK * 128), mb, fb, n0 + 64 * h, r0, pol_b);
          } else {
            tma_load_2d(b_tile(stage), mb, fb, r0, n0, pol_b);
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
      // Drain: the last load issued on each stage must have landed before
      // the CTA may exit.
      for (int s = 0; s < STAGES; ++s) {
        if (loads > static_cast<uint32_t>(s)) {
          const uint32_t n_s = (loads - s + STAGES - 1) / STAGES;
          wait_bounded(full_bar(s), (n_s - 1) & 1u, tmo, abort_flag, kSiteDrainLoads, false);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc = 0;
      for_each_work<kSplit>(P, blockIdx.x, gridDim.x, [&](int t, int k0, int k1, int) -> bool {
        const TileCoord tc = decode_tile(P, t);
        const ProblemDesc& d = P.prob[tc.p];
        const int kend = k1 < 0 ? d.num_k : k1;
        if (kend <= k0) return true;
        const uint32_t b = acc % kAccBufs;
        const uint32_t acc_phase = (acc / kAccBufs) & 1u;
        if (!wait_pipe(tempty_bar(b), acc_phase ^ 1u, kSiteMmaTmemEmpty)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kAccCols;
        for (int k = k0; k < kend; ++k) {
          if (!wait_pipe(full_bar(stage), phase, kSiteMmaFull)) return false;
          tc_fence_after();
          const uint32_t sa = a_tile(stage);
          const uint32_t sb = b_tile(stage);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = operand_desc<BK>(sb, kk, d.b_mn);
#pragma unroll
            for (int hh = 0; hh < MH; ++hh) {
              const uint64_t ad = operand_desc<BK>(sa + hh * L::kAHalfBytes, kk, d.a_mn);
              umma_bf16(d_tmem + hh * kHalfCols, ad, bd, d.idesc, (k != k0 || kk != 0) ? 1u : 0u);
            }
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(tfull_bar(b));
        ++acc;
        return true;
      });
      // Drain every MMA issued by this thread before TMEM is released.
      umma_commit(mma_done_bar);
      wait_bounded(mma_done_bar, 0, tmo, abort_flag, kSiteDrainMma, false);
    }
  } else if (kSplit && warp >= epi_first_warp<MH>()) {
    // ------------------------------------------- epilogue, reduction split
    // Per tile: this piece's rows go to the staging tile; one bulk copy per
    // other CTA o of the cluster sends band o of them into o's inbox,
    // counted on o's inbox barrier; this CTA's own band stays in place.
    // The inbox holds the other pieces' blocks of this CTA's band in piece
    // order, piece g at block g (g < me) or g - 1 (g > me).
    constexpr int kLd = L::kSplitLd;
    const int q = warp & 3;  // TMEM lane quarter: tile rows 32q .. 32q+31
    const uint32_t S = cluster_nctarank();
    const uint32_t me = cluster_ctarank();
    const int band = kBM / static_cast<int>(S);  // rows each CTA finishes
    const int r = q * 32 + lane;                  // the tile row this lane stages
    const uint32_t band_bytes = static_cast<uint32_t>(band * kLd * 4);
    uint32_t acc = 0, item = 0;
    for_each_work<kSplit>(P, blockIdx.x, gridDim.x, [&](int t, int k0, int k1, int) -> bool {
      const TileCoord tc = decode_tile(P, t);
      const ProblemDesc& d = P.prob[tc.p];
      const int m0 = tc.m_blk * kTileM;
      const int n0 = tc.n_blk * BN;
      // 1. Every CTA has finished with this CTA's staging tile and inbox of
      // the previous tile; the inbox (its previous phase complete) is told
      // what this tile brings.
      int ok = 1;
      if (lane == 0) {
        if (item > 0)
          ok = wait_polling<true>(split_free, (item - 1) & 1u, tmo, abort_flag, kSiteSplitFree);
        if (ok && q == 0) mbar_arrive_expect_tx(inbox_full, (S - 1) * band_bytes);
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) return false;
      // 2. This piece's rows, fp32, to the staging tile (the whole tile,
      // ragged edges included: the copies are whole bands).
      const bool has = (k1 < 0 ? d.num_k : k1) > k0;
      const uint32_t b = acc % kAccBufs;
      if (has) {
        if (lane == 0)
          ok = wait_polling<false>(tfull_bar(b), (acc / kAccBufs) & 1u, tmo, abort_flag, kSiteEpiTmemFull);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) return false;
        tc_fence_after();
      }
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kAccCols;
      const uint32_t my_row = staging + static_cast<uint32_t>(r * kLd * 4);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        if (has) {
          tmem_ld_32x32b_x32(t_row + c * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(my_row + static_cast<uint32_t>((c * 32 + 4 * j) * 4), v[4 * j], v[4 * j + 1],
                       v[4 * j + 2], v[4 * j + 3]);
      }
      if (has) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(b));
        ++acc;
      }
      // 3. The staged rows are made visible to the copy engine and counted
      // on the staged barrier; once all four warps have staged theirs, one
      // thread sends each other CTA its band.
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(staged_bar);
      if (q == 0) {
        if (lane == 0) {
          ok = wait_polling<false>(staged_bar, item & 1u, tmo, abort_flag, kSiteSplitStaged);
          for (uint32_t o = 0; ok && o < S; ++o) {
            if (o == me) continue;
            const uint32_t blk = me < o ? me : me - 1;
            bulk_copy_to_cluster(mapa_shared(inbox + blk * band_bytes, o), staging + o * band_bytes,
                                 band_bytes, mapa_shared(inbox_full, o));
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) return false;
      }
      // 4. Every other piece of this CTA's band has arrived.
      if (lane == 0) ok = wait_polling<true>(inbox_full, item & 1u, tmo, abort_flag, kSiteSplitInbox);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) return false;
      // 5. Pieces 0..S-1 added in that order, the band written out (see
      // split_band_sum).  The output's fields are copied out of the
      // parameter block first (the stores go through generic pointers,
      // after which the compiler would read them again from there every
      // row).
      ProblemDesc od{};
      od.C = d.C;
      od.ldc = d.ldc;
      od.M = d.M;
      od.N = d.N;
      od.out_mode = d.out_mode;
      od.out_t = d.out_t;
      const int row0 = m0 + static_cast<int>(me) * band;
      const uint32_t own = staging + me * band_bytes;
      if (S == 2) split_band_sum<2, BN, kLd>(own, inbox, static_cast<int>(me), q, lane, row0, n0, od);
      else if (S == 4) split_band_sum<4, BN, kLd>(own, inbox, static_cast<int>(me), q, lane, row0, n0, od);
      else split_band_sum<8, BN, kLd>(own, inbox, static_cast<int>(me), q, lane, row0, n0, od);
      // 6. This warp is done with the staging tile and inbox: one arrival
      // on every CTA's free barrier (kEpiWarps per CTA).
      __syncwarp();
      if (lane == 0)
        for (uint32_t g = 0; g < S; ++g) mbar_arrive_cluster(mapa_shared(split_free, g));
      ++item;
      return true;
    });
  } else if (!kSplit && warp >= epi_first_warp<MH>()) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int hh = (warp - epi_first_warp<MH>()) >> 2;  // row half it drains
    uint32_t acc = 0;
    for_each_work(P, blockIdx.x, gridDim.x, [&](int t, int k0, int k1, int kind) -> bool {
      const TileCoord tc = decode_tile(P, t);
      const ProblemDesc& d = P.prob[tc.p];
      const int row = tc.m_blk * kTileM + hh * kBM + q * 32 + lane;
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
      // The transposed register-resident epilogue only where its registers
      // fit: 320 threads leave 168 a thread, too few beside the plain one.
      epilogue_item<BN, MAXP, MH == 1>(P, d, kind, blockIdx.x, warp - epi_first_warp<MH>(),
                                       tc.m_blk * kTileM, n0, t_row, row, tempty_bar(b), false);
      ++acc;
      return true;
    });
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // No CTA leaves while another may still store into its inbox or arrive
  // on its barriers.
  if constexpr (kSplit) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace axonn
