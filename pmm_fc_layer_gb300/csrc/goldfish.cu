// Goldfish-loss masked cross-entropy over bf16 logits, with its gradient.
//
// The pith.science review of arXiv 2502.08145 ("What carries the argument")
// has the paper train against memorisation with Goldfish Loss, which leaves
// tokens out of the cross-entropy at random; its "Assumptions & free
// parameters" give the mask parameters k = 2 and h = 13.  The rule taken
// here, from the method's own paper that the pages cite (a hash of the h
// tokens before a label picks one label in k to leave out):
//   label (b, t) is dropped when FNV-1a-64(input_ids[b, t-h+1 .. t]) mod k
//   == 0 (each id as 4 little-endian bytes, oldest first); labels with fewer
//   than h tokens before them are kept; k = 0 keeps every label; labels
//   outside [0, V) are padding and never counted.
//   CE_t = logsumexp(z_t) - z_t[y_t];  loss = sum_kept CE_t / n (0 if n = 0)
//   dloss/dz_t = G_t (softmax(z_t) - e_{y_t}) / n.
//
// Three launches on the caller's stream:
//  1. goldfish_mask_kernel: one CTA hashes every window, writes keep[] and
//     the count n (a block reduction, so no atomics and no zeroing).
//  2. goldfish_rows_kernel: a cluster of C CTAs per row of logits,
//     persistent over rows.  CTA c of the cluster holds elements
//     [c*L, (c+1)*L) of the row in shared memory, brought in by one 1-D bulk
//     copy (cp.async.bulk) and double-buffered so the next kept row loads
//     while this one is computed.  Each CTA reduces its slice to (max, sum
//     of exp), the owner of the label also its logit, and publishes them in
//     its shared memory; after one cluster barrier every CTA reads the C
//     triples through distributed shared memory and has logsumexp.  The
//     gradient slice is then computed from shared memory and streamed out.
//     The logits of a row are read from HBM once; rows of dropped labels are
//     not read at all (their gradient is zero).
//  3. goldfish_mean_kernel: one CTA sums token_loss[] in a fixed order and
//     divides by n.
// Every wait on a copy is bounded by a wall-clock limit; on expiry the CTA
// records an error word (read by axonn_sync_status), stops issuing copies,
// keeps taking part in the cluster barriers and drains before exiting.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "goldfish.h"
#include "ptx.cuh"

namespace axonn {

namespace {

constexpr int kGfConsumerWarps = 8;
constexpr int kGfConsumers = 32 * kGfConsumerWarps;
constexpr int kGfThreads = kGfConsumers + 32;  // + the producer warp
constexpr int kGfStages = 4;                   // slice buffers per CTA, at most
constexpr int kMaskThreads = 1024;
// Shared memory for one slice buffer: rows are split over as many CTAs as it
// takes (up to a cluster of 8) to keep a slice within kTargetSliceBytes, so
// that a ring of four buffers keeps 128 KB of copies in flight per SM; a
// row needs at most kMaxSliceBytes per CTA (then with two buffers).
constexpr int64_t kTargetSliceBytes = 32 * 1024;
constexpr int64_t kMaxSliceBytes = 96 * 1024;
constexpr int64_t kRingBytes = 200 * 1024;  // buffers of the ring fit in this
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ unsigned long long g_goldfish_status;

__device__ __forceinline__ void gf_record(uint32_t site) {
  const unsigned long long code =
      (0x7DULL << 32) | (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 8) | site;
  atomicCAS(&g_goldfish_status, 0ULL, code);
}

// Bounded wait on an mbarrier phase; false (and an error word) on expiry.
__device__ __forceinline__ bool gf_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                        uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      gf_record(site);
      return false;
    }
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on
// `bar` in bytes (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ mask
// 64-bit FNV-1a (Fowler, Noll and Vo): state starts at the offset basis;
// each byte is xor-ed in, then the state is multiplied by the prime mod 2^64.
__device__ __forceinline__ uint64_t fnv1a64_ids(const int32_t* w, int h) {
  uint64_t s = 0xCBF29CE484222325ull;
  for (int j = 0; j < h; ++j) {
    const uint32_t v = static_cast<uint32_t>(w[j]);
#pragma unroll
    for (int byte = 0; byte < 4; ++byte) {
      s ^= (v >> (8 * byte)) & 0xFFu;
      s *= 0x100000001B3ull;
    }
  }
  return s;
}

__global__ void __launch_bounds__(kMaskThreads) goldfish_mask_kernel(GoldfishArgs a) {
  __shared__ int counts[kMaskThreads / 32];
  const int64_t T = a.batch * a.seq;
  int count = 0;
  for (int64_t i = threadIdx.x; i < T; i += blockDim.x) {
    const int64_t b = i / a.seq, t = i - b * a.seq;
    const int32_t y = a.labels[i];
    uint8_t g = 0;
    if (y >= 0 && y < a.vocab) {
      if (a.k == 0 || t < a.h - 1) {
        g = 1;
      } else {
        const uint64_t H = fnv1a64_ids(a.input_ids + b * a.seq + t - a.h + 1, a.h);
        g = (H % static_cast<uint64_t>(a.k)) != 0 ? 1 : 0;
      }
    }
    a.keep[i] = g;
    count += g;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) count += __shfl_xor_sync(0xFFFFFFFFu, count, o);
  if ((threadIdx.x & 31) == 0) counts[threadIdx.x >> 5] = count;
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    for (int w = 0; w < kMaskThreads / 32; ++w) n += counts[w];
    *a.kept = n;
  }
}

// ------------------------------------------------------------------ rows
struct RowParams {
  GoldfishArgs a;
  int cluster;    // CTAs per row
  int stages;     // slice buffers in the ring (2 to kGfStages)
  int64_t slice;  // elements per CTA (multiple of 8)
};

// Shared memory after the slice buffers.
struct alignas(16) GfTail {
  float4 inbox[2][8];  // [row parity][sending CTA]: max, sum of exp, label logit, has label
  uint64_t full[kGfStages];
  uint64_t empty[kGfStages];
  uint64_t inbox_bar[2];
  int64_t meta_row[kGfStages];
  int32_t meta_y[kGfStages];
  int32_t meta_keep[kGfStages];
  float red_m[kGfConsumerWarps];
  float red_s[kGfConsumerWarps];
  float lse;
  int aborted;
};

// Barrier among the consumer warps only (the producer warp runs ahead).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGfConsumers) : "memory");
}

// 16-byte store into (possibly another CTA's) shared memory whose
// completion is counted, in bytes, on an mbarrier of that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float4 v, uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          cluster_addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cluster_bar)
      : "memory");
}

// Element j (0..7) of eight packed bf16 values.
__device__ __forceinline__ float lane_bf16(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : (j < 4 ? v.y : (j < 6 ? v.z : v.w));
  return bf16_to_f32(static_cast<uint16_t>(w >> (16 * (j & 1))));
}

// Writes zeros to elements [c0, c1) of a gradient row (16-byte stores for
// the part whose start is 8-aligned, single elements for the tail), by the
// consumer threads.
__device__ __forceinline__ void zero_row(uint16_t* row, int64_t c0, int64_t c1, int ct) {
  const int64_t v1 = c0 + ((c1 - c0) & ~int64_t{7});
  for (int64_t i = c0 + 8 * ct; i < v1; i += 8 * kGfConsumers)
    __stcs(reinterpret_cast<int4*>(row + i), make_int4(0, 0, 0, 0));
  for (int64_t i = v1 + ct; i < c1; i += kGfConsumers) row[i] = 0;
}

// Warp 0 is the producer: lane 0 walks the cluster's rows, records each
// row's label and mask in a ring of kGfStages entries and, for a kept row,
// bulk-copies this CTA's slice of its logits into the entry's buffer (a
// dropped row gets a plain arrival: nothing to read).  Warps 1..8 consume
// the ring in order.  For a kept row each CTA reduces its slice to (max,
// sum of exp) and pushes it, with the label's logit if it owns it, into
// every peer's inbox with st.async, completing on the peer's inbox barrier;
// when its own inbox has all C entries it forms logsumexp and writes its
// gradient slice.  A CTA pushes row i+2's entry (same inbox parity as row
// i) only after it received every peer's entry for row i+1, which each
// peer sends after it read row i's inbox: so two inbox slots suffice and no
// cluster barrier is needed per row.
__global__ void __launch_bounds__(kGfThreads, 1)
    goldfish_rows_kernel(const __grid_constant__ RowParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GoldfishArgs& a = p.a;
  const int C = p.cluster;
  const uint32_t rank = C > 1 ? cluster_ctarank() : 0u;
  const int64_t cl = blockIdx.x / C;
  const int64_t ncl = gridDim.x / C;
  const int64_t T = a.batch * a.seq;
  const int64_t V = a.vocab;
  const int64_t vpad = (V + 7) & ~int64_t{7};
  const int64_t s0 = static_cast<int64_t>(rank) * p.slice;
  const int64_t n_load = s0 < vpad ? min(p.slice, vpad - s0) : 0;  // elements copied
  const int64_t n_valid = s0 < V ? min(p.slice, V - s0) : 0;       // elements of the row
  const int64_t buf_bytes = p.slice * 2;
  GfTail* tl = reinterpret_cast<GfTail*>(smem + p.stages * buf_bytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < p.stages; ++b) {
      mbar_init(smem_addr(&tl->full[b]), 1);
      mbar_init(smem_addr(&tl->empty[b]), kGfConsumerWarps);
    }
    mbar_init(smem_addr(&tl->inbox_bar[0]), 1);
    mbar_init(smem_addr(&tl->inbox_bar[1]), 1);
    tl->aborted = 0;
    fence_mbarrier_init();
  }
  // every CTA's barriers are set up before any peer pushes to them
  cluster_sync();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int NB = p.stages;
    int b = 0;
    uint32_t ph = 0;
    int issued[kGfStages] = {};  // phases of each stage that carried a copy
    int uses[kGfStages] = {};
    for (int64_t base = cl; base < T; base += 32 * ncl) {
      // 32 rows' labels and mask flags at once, one per lane
      const int64_t rr = base + lane * ncl;
      const int32_t keep_l = rr < T ? a.keep[rr] : 0;
      const int32_t y_l = rr < T ? a.labels[rr] : 0;
      const int64_t left = (T - base + ncl - 1) / ncl;
      const int cnt = left < 32 ? static_cast<int>(left) : 32;
      for (int j = 0; j < cnt; ++j) {
        const int32_t keep = __shfl_sync(0xFFFFFFFFu, keep_l, j);
        const int32_t y = __shfl_sync(0xFFFFFFFFu, y_l, j);
        if (lane == 0) {
          const int64_t r = base + j * ncl;
          if (!gf_wait(smem_addr(&tl->empty[b]), ph ^ 1u, tmo, 3)) tl->aborted = 1;
          tl->meta_row[b] = r;
          tl->meta_y[b] = y;
          tl->meta_keep[b] = keep;
          const uint32_t fb = smem_addr(&tl->full[b]);
          if (keep && n_load > 0 && !tl->aborted) {
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(n_load * 2));
            bulk_load(smem_addr(smem + b * buf_bytes), a.logits + r * a.ld_logits + s0,
                      static_cast<uint32_t>(n_load * 2), fb);
            issued[b] = uses[b] + 1;
          } else {
            mbar_arrive(fb);  // publishes the entry; nothing to copy
          }
          ++uses[b];
        }
        __syncwarp();
        if (++b == NB) {
          b = 0;
          ph ^= 1u;
        }
      }
    }
    // Copies not consumed exist only after an expired wait: let them land
    // (bounded) before this CTA's shared memory goes away.
    if (lane == 0 && tl->aborted) {
      for (int s = 0; s < NB; ++s)
        if (issued[s] > 0) gf_wait(smem_addr(&tl->full[s]), (issued[s] - 1) & 1u, tmo, 2);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;            // consumer warp 0..7
    const int ct = threadIdx.x - 32;    // consumer thread 0..255
    const int NB = p.stages;
    const int32_t n = *a.kept;
    const float inv_n = n > 0 ? 1.0f / static_cast<float>(n) : 0.0f;
    int b = 0;
    uint32_t ph = 0;
    int kc = 0;  // kept rows so far
    for (int64_t r = cl; r < T; r += ncl) {
      if (!gf_wait(smem_addr(&tl->full[b]), ph, tmo, 1)) tl->aborted = 1;
      const int32_t y = tl->meta_y[b];
      const int keep = tl->meta_keep[b];
      const uint16_t* x = reinterpret_cast<const uint16_t*>(smem + b * buf_bytes);
      if (!keep) {
        if (a.dlogits && n_valid > 0) zero_row(a.dlogits + r * a.ld_dlogits, s0, s0 + n_valid, ct);
        if (rank == 0 && ct == 0) a.token_loss[r] = 0.0f;
      } else {
        const bool have = n_load > 0 && !tl->aborted;
        // this slice's max, then its sum of exp(x - max)
        float m = -INFINITY;
        if (have) {
          for (int64_t i = 8 * ct; i < n_valid; i += 8 * kGfConsumers) {
            const uint4 v = *reinterpret_cast<const uint4*>(x + i);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (i + j < n_valid) m = fmaxf(m, lane_bf16(v, j));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) tl->red_m[cw] = m;
        consumer_sync();
        m = tl->red_m[0];
#pragma unroll
        for (int w = 1; w < kGfConsumerWarps; ++w) m = fmaxf(m, tl->red_m[w]);
        float sum = 0.0f;
        if (have && m > -INFINITY) {
          const float mb = m * kLog2e;
          for (int64_t i = 8 * ct; i < n_valid; i += 8 * kGfConsumers) {
            const uint4 v = *reinterpret_cast<const uint4*>(x + i);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (i + j < n_valid) sum += exp2f(fmaf(lane_bf16(v, j), kLog2e, -mb));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane == 0) tl->red_s[cw] = sum;
        consumer_sync();
        if (ct == 0) {
          float s = 0.0f;
#pragma unroll
          for (int w = 0; w < kGfConsumerWarps; ++w) s += tl->red_s[w];
          const bool mine = have && y >= s0 && y < s0 + n_valid;
          const float4 entry = make_float4(m, s, mine ? bf16_to_f32(x[y - s0]) : 0.0f,
                                           mine ? 1.0f : 0.0f);
          const int par = kc & 1;
          const uint32_t ib = smem_addr(&tl->inbox_bar[par]);
          mbar_arrive_expect_tx(ib, static_cast<uint32_t>(16 * C));
          const uint32_t slot = smem_addr(&tl->inbox[par][rank]);
          for (int c = 0; c < C; ++c)
            st_async_v4(mapa_shared(slot, static_cast<uint32_t>(c)), entry,
                        mapa_shared(ib, static_cast<uint32_t>(c)));
          if (!gf_wait(ib, (kc >> 1) & 1u, tmo, 4)) tl->aborted = 1;
          float M = -INFINITY, zy = 0.0f;
          for (int c = 0; c < C; ++c) {
            const float4 e = tl->inbox[par][c];
            M = fmaxf(M, e.x);
            if (e.w != 0.0f) zy = e.z;
          }
          float S = 0.0f;
          for (int c = 0; c < C; ++c) {
            const float4 e = tl->inbox[par][c];
            if (e.x > -INFINITY) S += e.y * exp2f((e.x - M) * kLog2e);
          }
          const float lse = M + log2f(S) * kLn2;
          tl->lse = lse;
          if (rank == 0) a.token_loss[r] = lse - zy;
        }
        consumer_sync();
        const float lse = tl->lse;
        // gradient slice: (softmax - onehot) / n, from shared memory
        if (a.dlogits && n_valid > 0) {
          uint16_t* out = a.dlogits + r * a.ld_dlogits + s0;
          const float lb = lse * kLog2e;
          const int64_t yl = y - s0;  // the label's place in this slice (may be outside)
          const int64_t vfull = n_valid & ~int64_t{7};
          for (int64_t i = 8 * ct; i < vfull; i += 8 * kGfConsumers) {
            const uint4 v = have ? *reinterpret_cast<const uint4*>(x + i) : make_uint4(0, 0, 0, 0);
            float g[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              g[j] = exp2f(fmaf(lane_bf16(v, j), kLog2e, -lb)) * inv_n;
              if (i + j == yl) g[j] -= inv_n;
            }
            __stcs(reinterpret_cast<int4*>(out + i),
                   make_int4(static_cast<int>(pack2(g[0], g[1])), static_cast<int>(pack2(g[2], g[3])),
                             static_cast<int>(pack2(g[4], g[5])), static_cast<int>(pack2(g[6], g[7]))));
          }
          for (int64_t i = vfull + ct; i < n_valid; i += kGfConsumers) {
            const float z = have ? bf16_to_f32(x[i]) : 0.0f;
            float g = exp2f(fmaf(z, kLog2e, -lb)) * inv_n;
            if (i == yl) g -= inv_n;
            __nv_bfloat16 h = __float2bfloat16_rn(g);
            out[i] = *reinterpret_cast<uint16_t*>(&h);
          }
        }
        ++kc;
      }
      // this warp is done with the stage's buffer
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tl->empty[b]));
      if (++b == NB) {
        b = 0;
        ph ^= 1u;
      }
    }
  }
  // no CTA leaves while a peer may still push into its inbox
  cluster_sync();
}

// ------------------------------------------------------------------ mean
__global__ void __launch_bounds__(1024) goldfish_mean_kernel(GoldfishArgs a) {
  __shared__ float part[32];
  const int64_t T = a.batch * a.seq;
  float s = 0.0f;
  for (int64_t i = threadIdx.x; i < T; i += blockDim.x) s += a.token_loss[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < 32; ++w) t += part[w];
    const int32_t n = *a.kept;
    *a.loss = n > 0 ? t / static_cast<float>(n) : 0.0f;
  }
}

}  // namespace

int64_t goldfish_slice(int64_t vocab, int cluster) {
  const int64_t vpad = (vocab + 7) / 8 * 8;
  const int64_t per = (vpad + cluster - 1) / cluster;
  return (per + 7) / 8 * 8;
}

int goldfish_cluster(int64_t vocab) {
  for (int c = 1; c <= 8; c *= 2)
    if (goldfish_slice(vocab, c) * 2 <= kTargetSliceBytes) return c;
  for (int c = 1; c <= 8; c *= 2)
    if (goldfish_slice(vocab, c) * 2 <= kMaxSliceBytes) return c;
  return 0;
}

cudaError_t goldfish_launch(const GoldfishArgs& a, int cluster, int sms, cudaStream_t stream) {
  const int64_t T = a.batch * a.seq;
  goldfish_mask_kernel<<<1, kMaskThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  RowParams p;
  p.a = a;
  p.cluster = cluster;
  p.slice = goldfish_slice(a.vocab, cluster);
  p.stages = static_cast<int>(std::min<int64_t>(kGfStages, kRingBytes / (p.slice * 2)));
  const size_t smem = static_cast<size_t>(p.stages * p.slice * 2) + sizeof(GfTail);
  e = cudaFuncSetAttribute(goldfish_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // Persistent clusters: as many as fit at once (no cluster waits for
  // another, so a larger grid would only queue), at most one per row.
  const int per_sm = static_cast<int>(std::min<size_t>(4, (227 * 1024) / (smem + 1024)));
  int64_t clusters = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1) / cluster;
  if (clusters < 1) clusters = 1;
  if (clusters > T) clusters = T;
  if (T > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cluster), 1, 1);
    cfg.blockDim = dim3(kGfThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, goldfish_rows_kernel, p);
    if (e != cudaSuccess) return e;
  }
  goldfish_mean_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t goldfish_take_status(unsigned long long* word, cudaStream_t stream) {
  *word = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_goldfish_status, sizeof(*word), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned long long zero = 0;
  e = cudaMemcpyToSymbolAsync(g_goldfish_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace axonn
