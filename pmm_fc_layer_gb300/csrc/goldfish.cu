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
//     [c*L, (c+1)*L) of a row in shared memory, brought in by one 1-D bulk
//     copy (cp.async.bulk) into a ring of up to four buffers filled by a
//     producer warp, so copies of the next kept rows are in flight while one
//     is computed.  Sixteen consumer warps reduce the slice to (max, sum of
//     exp) in one pass, the owner of the label adds its logit, and the entry
//     is pushed into every CTA of the cluster through distributed shared
//     memory (st.async onto an mbarrier); with all C entries a CTA has
//     logsumexp and writes its gradient slice from shared memory.  The
//     exchange of one row overlaps the gradient pass of the previous one.
//     The logits of a row are read from HBM once; rows of dropped labels are
//     not read at all (their gradient rows are written as zeros first).
//  3. goldfish_mean_kernel: one CTA sums token_loss[] in a fixed order and
//     divides by n.
// Every wait on a copy is bounded by a wall-clock limit; on expiry the CTA
// records an error word (read by axonn_sync_status), stops issuing copies,
// keeps taking part in the cluster barriers and drains before exiting.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "goldfish.h"
#include "ptx.cuh"

namespace axonn {

namespace {

constexpr int kGfConsumerWarps = 16;
constexpr int kGfConsumers = 32 * kGfConsumerWarps;
constexpr int kGfThreads = kGfConsumers + 32;  // + the producer warp
constexpr int kGfStages = 4;                   // slice buffers per CTA, at most
constexpr int kMaskThreads = 1024;
// Shared memory: a row is split over a cluster of C CTAs (C in {1, 2, 4,
// 8}); each CTA's slice is at most kMaxSliceBytes, and its ring holds as
// many slices (up to kGfStages) as fit in kRingBytes.
constexpr int64_t kMaxSliceBytes = 96 * 1024;
constexpr int64_t kRingBytes = 200 * 1024;
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

// 2^x by the SFU's approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22; results below 2^-126 flush to zero, far below any bound the
// loss or its bf16 gradient is held to).  The softmax's exponents are never
// positive, so no overflow path is needed.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

constexpr int kInbox = 3;  // inbox slots: rows kc, kc+1 and kc+2 may be in flight

// Shared memory after the slice buffers.
struct alignas(16) GfTail {
  float4 inbox[kInbox][8];  // [row % kInbox][sending CTA]: max, sum of exp, label logit, has it
  uint64_t full[kGfStages];
  uint64_t empty[kGfStages];
  uint64_t inbox_bar[kInbox];
  int64_t meta_row[kGfStages];
  int32_t meta_y[kGfStages];
  float red_m[kGfConsumerWarps];
  float red_s[kGfConsumerWarps];
  int red_n[kGfConsumerWarps];
  float lse;
  int aborted;
  uint8_t flags[kGfConsumers];  // mask flags of a chunk of the cluster's rows
};

// Barrier among the consumer warps only (the producer warp runs ahead).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGfConsumers) : "memory");
}

// The eight bf16 values of a 16-byte vector as floats (exact): a bf16 is
// the high half of a float, so the high half of each 32-bit word is masked
// out in place and the low half shifted up.
__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xFFFF0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xFFFF0000u);
  x[4] = __uint_as_float(v.z << 16);
  x[5] = __uint_as_float(v.z & 0xFFFF0000u);
  x[6] = __uint_as_float(v.w << 16);
  x[7] = __uint_as_float(v.w & 0xFFFF0000u);
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

// Number of consumer threads whose `pred` is true (a barrier among the
// consumers; every consumer thread gets the count).
__device__ __forceinline__ int consumers_count(bool pred, GfTail* tl);

// Adds values to one thread's running (max, sum of exp(x - max)).
__device__ __forceinline__ void online_add8(float& m, float& s, const float (&x)[8]) {
  const float vm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                         fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
  if (vm > m) {
    s *= fast_exp2((m - vm) * kLog2e);  // 2^-inf = 0 on the first values
    m = vm;
  }
  const float mb = m * kLog2e;
  float t0 = 0.0f, t1 = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    t0 += fast_exp2(fmaf(x[j], kLog2e, -mb));
    t1 += fast_exp2(fmaf(x[j + 1], kLog2e, -mb));
  }
  s += t0 + t1;
}

__device__ __forceinline__ void online_add1(float& m, float& s, float x) {
  if (x > m) {
    s *= fast_exp2((m - x) * kLog2e);
    m = x;
  }
  s += fast_exp2((x - m) * kLog2e);
}

__device__ __forceinline__ int consumers_count(bool pred, GfTail* tl) {
  const int w = (threadIdx.x >> 5) - 1;
  const int c = __popc(__ballot_sync(0xFFFFFFFFu, pred));
  if ((threadIdx.x & 31) == 0) tl->red_n[w] = c;
  consumer_sync();
  int n = 0;
#pragma unroll
  for (int i = 0; i < kGfConsumerWarps; ++i) n += tl->red_n[i];
  return n;
}

// Warp 0 is the producer: lane 0 bulk-copies this CTA's slice of every kept
// row of the cluster, in order, into a ring of `stages` buffers.  Warps
// 1..16 are the consumers.  They first write the zero gradient rows (and
// zero losses) of the cluster's dropped labels, which need no logits.  Then,
// for kept row kc, each CTA reduces its slice to (max, sum of exp), adds the
// label's logit if it owns it, and pushes that entry with st.async into the
// same inbox slot (kc mod 3) of every CTA of the cluster, completing on that
// CTA's inbox barrier.  Row kc+1 is reduced and pushed before row kc's inbox
// is read and its gradient written, so the exchange overlaps a gradient
// pass.  A CTA pushes row kc+3 into slot kc mod 3 only after it has every
// peer's entry for row kc+2, which each peer pushes after reading its row
// kc entries: three slots suffice and no cluster barrier is needed per row.
__global__ void __launch_bounds__(kGfThreads, 1)
    goldfish_rows_kernel(const __grid_constant__ RowParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GoldfishArgs& a = p.a;
  const int C = p.cluster;
  const int NB = p.stages;
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
  GfTail* tl = reinterpret_cast<GfTail*>(smem + NB * buf_bytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(smem_addr(&tl->full[b]), 1);
      mbar_init(smem_addr(&tl->empty[b]), kGfConsumerWarps);
    }
    for (int q = 0; q < kInbox; ++q) mbar_init(smem_addr(&tl->inbox_bar[q]), 1);
    tl->aborted = 0;
    fence_mbarrier_init();
  }
  // every CTA's barriers are set up before any peer pushes to them
  cluster_sync();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int b = 0;
    uint32_t ph = 0;
    int issued[kGfStages] = {};  // 1 + the last use of each stage that carried a copy
    int uses[kGfStages] = {};
    for (int64_t base = cl; base < T; base += 32 * ncl) {
      // 32 rows' labels and mask flags at once, one per lane
      const int64_t rr = base + lane * ncl;
      const int32_t keep_l = rr < T ? a.keep[rr] : 0;
      const int32_t y_l = rr < T ? a.labels[rr] : 0;
      uint32_t kept_bits = __ballot_sync(0xFFFFFFFFu, keep_l != 0);
      while (kept_bits) {
        const int j = __ffs(kept_bits) - 1;
        kept_bits &= kept_bits - 1;
        const int32_t y = __shfl_sync(0xFFFFFFFFu, y_l, j);
        if (lane == 0) {
          const int64_t r = base + j * ncl;
          if (!gf_wait(smem_addr(&tl->empty[b]), ph ^ 1u, tmo, 3)) tl->aborted = 1;
          tl->meta_row[b] = r;
          tl->meta_y[b] = y;
          const uint32_t fb = smem_addr(&tl->full[b]);
          if (n_load > 0 && !tl->aborted) {
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
      for (int q = 0; q < NB; ++q)
        if (issued[q] > 0) gf_wait(smem_addr(&tl->full[q]), (issued[q] - 1) & 1u, tmo, 2);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;          // consumer warp
    const int ct = threadIdx.x - 32;  // consumer thread
    const int32_t n = *a.kept;
    const float inv_n = n > 0 ? 1.0f / static_cast<float>(n) : 0.0f;
    const float log2n = n > 0 ? log2f(static_cast<float>(n)) : 0.0f;

    // 1. rows of dropped labels: zero gradient slices and losses; count the
    //    kept rows of this cluster.  The mask flags of kGfConsumers rows at a
    //    time are read in parallel (one per thread) into shared memory.
    int nk = 0;
    for (int64_t base = cl; base < T; base += static_cast<int64_t>(kGfConsumers) * ncl) {
      const int64_t rr = base + static_cast<int64_t>(ct) * ncl;
      const int kf = rr < T ? a.keep[rr] : 1;
      tl->flags[ct] = static_cast<uint8_t>(kf != 0);
      nk += consumers_count(rr < T && kf != 0, tl);
      for (int j = 0; j < kGfConsumers; ++j) {
        const int64_t r = base + static_cast<int64_t>(j) * ncl;
        if (r >= T) break;
        if (tl->flags[j]) continue;
        if (a.dlogits && n_valid > 0) zero_row(a.dlogits + r * a.ld_dlogits, s0, s0 + n_valid, ct);
        if (rank == 0 && ct == 0) a.token_loss[r] = 0.0f;
      }
      consumer_sync();  // flags are rewritten for the next chunk
    }

    // 2. kept rows, software-pipelined by one row
    auto stage_of = [&](int kc) { return kc % NB; };
    auto wait_full = [&](int kc) {
      if (!gf_wait(smem_addr(&tl->full[stage_of(kc)]), static_cast<uint32_t>((kc / NB) & 1), tmo, 1))
        tl->aborted = 1;
    };
    // reduce kept row kc to this slice's entry and push it to every CTA
    auto reduce_push = [&](int kc) {
      wait_full(kc);
      const int b = stage_of(kc);
      const uint16_t* x = reinterpret_cast<const uint16_t*>(smem + b * buf_bytes);
      const int32_t y = tl->meta_y[b];
      const bool have = n_load > 0 && !tl->aborted;
      float m0 = -INFINITY, s0_ = 0.0f, m1 = -INFINITY, s1 = 0.0f;
      if (have) {
        // whole 8-element vectors, two per iteration, then the ragged tail
        const int64_t vfull = n_valid & ~int64_t{7};
        for (int64_t i = 16 * ct; i < vfull; i += 16 * kGfConsumers) {
          float xa[8];
          unpack8(*reinterpret_cast<const uint4*>(x + i), xa);
          online_add8(m0, s0_, xa);
          if (i + 8 < vfull) {
            float xb[8];
            unpack8(*reinterpret_cast<const uint4*>(x + i + 8), xb);
            online_add8(m1, s1, xb);
          }
        }
        for (int64_t i = vfull + ct; i < n_valid; i += kGfConsumers)
          online_add1(m1, s1, bf16_to_f32(x[i]));
      }
      // thread's (max, sum), then the slice's
      float m = fmaxf(m0, m1);
      float sm = (m0 > -INFINITY ? s0_ * fast_exp2((m0 - m) * kLog2e) : 0.0f) +
                 (m1 > -INFINITY ? s1 * fast_exp2((m1 - m) * kLog2e) : 0.0f);
      float wm = m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, o));
      if (lane == 0) tl->red_m[cw] = wm;
      consumer_sync();
      float M = tl->red_m[0];
#pragma unroll
      for (int w = 1; w < kGfConsumerWarps; ++w) M = fmaxf(M, tl->red_m[w]);
      float ws = m > -INFINITY ? sm * fast_exp2((m - M) * kLog2e) : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, o);
      if (lane == 0) tl->red_s[cw] = ws;
      consumer_sync();
      if (ct == 0) {
        float S = 0.0f;
#pragma unroll
        for (int w = 0; w < kGfConsumerWarps; ++w) S += tl->red_s[w];
        const bool mine = have && y >= s0 && y < s0 + n_valid;
        const float4 entry = make_float4(M, S, mine ? bf16_to_f32(x[y - s0]) : 0.0f,
                                         mine ? 1.0f : 0.0f);
        const int q = kc % kInbox;
        const uint32_t ib = smem_addr(&tl->inbox_bar[q]);
        mbar_arrive_expect_tx(ib, static_cast<uint32_t>(16 * C));
        const uint32_t slot = smem_addr(&tl->inbox[q][rank]);
        for (int c = 0; c < C; ++c)
          st_async_v4(mapa_shared(slot, static_cast<uint32_t>(c)), entry,
                      mapa_shared(ib, static_cast<uint32_t>(c)));
      }
    };
    if (nk > 0) reduce_push(0);
    for (int kc = 0; kc < nk; ++kc) {
      if (kc + 1 < nk) reduce_push(kc + 1);
      const int b = stage_of(kc);
      const int64_t r = tl->meta_row[b];
      const int32_t y = tl->meta_y[b];
      const uint16_t* x = reinterpret_cast<const uint16_t*>(smem + b * buf_bytes);
      const bool have = n_load > 0 && !tl->aborted;
      if (cw == 0) {
        // logsumexp of the row from the C entries of its inbox slot
        const int q = kc % kInbox;
        // every lane waits (each then sees the pushed entries)
        if (!gf_wait(smem_addr(&tl->inbox_bar[q]), static_cast<uint32_t>((kc / kInbox) & 1), tmo, 4))
          tl->aborted = 1;
        const float4 e = lane < C ? tl->inbox[q][lane] : make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
        float M = e.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        float S = e.x > -INFINITY ? e.y * fast_exp2((e.x - M) * kLog2e) : 0.0f;
        float zy = e.w != 0.0f ? e.z : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
          zy += __shfl_xor_sync(0xFFFFFFFFu, zy, o);
        }
        if (lane == 0) {
          const float lse = M + log2f(S) * kLn2;
          tl->lse = lse;
          if (rank == 0) a.token_loss[r] = lse - zy;
        }
      }
      consumer_sync();
      const float lse = tl->lse;
      // gradient slice: (softmax - onehot) / n, from shared memory
      if (a.dlogits && n_valid > 0) {
        uint16_t* out = a.dlogits + r * a.ld_dlogits + s0;
        // p / n = 2^(z log2e - (lse log2e + log2 n)): the 1/n folded into
        // the exponent
        const float lb = fmaf(lse, kLog2e, log2n);
        const int64_t yl = y - s0;  // the label's place in this slice (may be outside)
        const int64_t vfull = n_valid & ~int64_t{7};
        for (int64_t i = 8 * ct; i < vfull; i += 8 * kGfConsumers) {
          float g[8];
          unpack8(have ? *reinterpret_cast<const uint4*>(x + i) : make_uint4(0, 0, 0, 0), g);
#pragma unroll
          for (int j = 0; j < 8; ++j) g[j] = fast_exp2(fmaf(g[j], kLog2e, -lb));
          const int64_t d = yl - i;  // the label's element, if in this vector
          if (d >= 0 && d < 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (j == d) g[j] -= inv_n;
          }
          __stcs(reinterpret_cast<int4*>(out + i),
                 make_int4(static_cast<int>(pack2(g[0], g[1])), static_cast<int>(pack2(g[2], g[3])),
                           static_cast<int>(pack2(g[4], g[5])), static_cast<int>(pack2(g[6], g[7]))));
        }
        for (int64_t i = vfull + ct; i < n_valid; i += kGfConsumers) {
          const float z = have ? bf16_to_f32(x[i]) : 0.0f;
          float g = fast_exp2(fmaf(z, kLog2e, -lb));
          if (i == yl) g -= inv_n;
          __nv_bfloat16 h = __float2bfloat16_rn(g);
          out[i] = *reinterpret_cast<uint16_t*>(&h);
        }
      }
      // this warp is done with the stage's buffer
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tl->empty[b]));
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
    if (goldfish_slice(vocab, c) * 2 <= kMaxSliceBytes) return c;
  return 0;
}

namespace {

// Ring depth and shared memory of the rows kernel for a slice.
int ring_stages(int64_t slice) {
  return static_cast<int>(std::min<int64_t>(kGfStages, kRingBytes / (slice * 2)));
}
size_t rows_smem(int64_t slice) {
  return static_cast<size_t>(ring_stages(slice) * slice * 2) + sizeof(GfTail);
}

cudaLaunchConfig_t rows_config(int cluster, int64_t slice, int grid, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kGfThreads, 1, 1);
  cfg.dynamicSmemBytes = rows_smem(slice);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// The cluster size for a vocabulary: among the sizes whose slices fit a ring
// of at least two buffers, the one that keeps the most SMs busy when the
// GPU holds as many clusters as it can at once (a cluster must fit in one
// GPC, so fewer large clusters may fit than SMs / C), and its cluster
// count.  Decided once per device and vocabulary.
struct ClusterPick {
  int64_t vocab = -1;
  int device = -1;
  int cluster = 0;
  int resident = 0;
};
std::mutex g_pick_mu;
ClusterPick g_picks[16];

cudaError_t pick_cluster(int64_t vocab, int sms, int* cluster, int* resident) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_pick_mu);
  for (const ClusterPick& c : g_picks)
    if (c.vocab == vocab && c.device == dev) {
      *cluster = c.cluster;
      *resident = c.resident;
      return cudaSuccess;
    }
  int best_c = 0, best_r = 0;
  for (int c = 8; c >= 1; c /= 2) {
    const int64_t slice = goldfish_slice(vocab, c);
    if (slice * 2 > kMaxSliceBytes || ring_stages(slice) < 2) continue;
    e = cudaFuncSetAttribute(goldfish_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(rows_smem(slice)));
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = rows_config(c, slice, c * sms, nullptr, attr);
    int r = 0;
    if (cudaOccupancyMaxActiveClusters(&r, reinterpret_cast<const void*>(goldfish_rows_kernel),
                                       &cfg) != cudaSuccess || r < 1) {
      (void)cudaGetLastError();
      r = std::max(1, sms / c);
    }
    if (best_c == 0 || r * c > best_r * best_c) {
      best_c = c;
      best_r = r;
    }
  }
  if (best_c == 0) return cudaErrorInvalidValue;
  static int next = 0;
  g_picks[next] = ClusterPick{vocab, dev, best_c, best_r};
  next = (next + 1) % 16;
  *cluster = best_c;
  *resident = best_r;
  return cudaSuccess;
}

}  // namespace

cudaError_t goldfish_launch(const GoldfishArgs& a, int sms, cudaStream_t stream) {
  const int64_t T = a.batch * a.seq;
  goldfish_mask_kernel<<<1, kMaskThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (T > 0) {
    int cluster = 0, resident = 0;
    e = pick_cluster(a.vocab, sms, &cluster, &resident);
    if (e != cudaSuccess) return e;
    RowParams p;
    p.a = a;
    p.cluster = cluster;
    p.slice = goldfish_slice(a.vocab, cluster);
    p.stages = ring_stages(p.slice);
    e = cudaFuncSetAttribute(goldfish_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(rows_smem(p.slice)));
    if (e != cudaSuccess) return e;
    // Persistent clusters: as many as the GPU holds at once, at most one per
    // row (with more, the rest would run as a second wave).
    const int64_t clusters = std::min<int64_t>(resident, T);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = rows_config(cluster, p.slice, static_cast<int>(clusters * cluster),
                                         stream, attr);
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
