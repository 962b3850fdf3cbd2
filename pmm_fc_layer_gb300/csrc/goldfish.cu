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
//     the count n (a block reduction, so no atomics and no zeroing), and
//     zeroes the word of `loss`, which the rows kernel uses as its row
//     counter until the mean kernel writes the loss there.
//  2. goldfish_rows_kernel: one CTA per SM, persistent; each CTA claims the
//     next row with an atomic add on that counter, so the rows spread over
//     the SMs as they free up whatever the mix of kept and dropped labels.
//     A dropped label's gradient row is written as zeros and its logits are
//     never read.  A kept row is read twice through a ring of 32 KB chunks
//     filled by a producer warp with 1-D bulk copies: the first pass (from
//     HBM, lines marked evict-last in L2) reduces it to (max, sum of exp)
//     and picks the label's logit; the second pass (the same lines, still
//     in L2, marked evict-first) computes the gradient (softmax - onehot) / n
//     into the chunk's buffer, and a store warp copies it out with one bulk
//     copy per chunk (and zero-fills dropped rows the same way).  The HBM
//     traffic is the kept rows read once and every gradient row written
//     once.  The producer claims a row and starts its copies while the
//     consumer warps finish the previous one.
//  3. goldfish_mean_kernel: one CTA sums token_loss[] in a fixed order and
//     divides by n.
// Every wait is bounded by a wall-clock limit; on expiry the CTA records an
// error word (read by axonn_sync_status), stops claiming rows and issuing
// copies, and lets the copies already issued land before it exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "goldfish.h"
#include "ptx.cuh"

namespace axonn {

namespace {

constexpr int kGfConsumerWarps = 16;
constexpr int kGfConsumers = 32 * kGfConsumerWarps;
constexpr int kGfThreads = kGfConsumers + 64;  // + the producer and the store warp
constexpr int kMaskThreads = 1024;
constexpr int64_t kGfChunk = 16384;  // elements of one copy (32 KB)
constexpr int kGfRing = 6;           // chunk buffers (192 KB)
constexpr int kGfRowQ = 2;           // claimed rows handed to the consumers
constexpr int kGfZeroBytes = 16384;  // zeros the store warp copies over dropped rows
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ unsigned long long g_goldfish_status;

__device__ __forceinline__ void gf_record(uint32_t site) {
  const unsigned long long code =
      (0x7DULL << 32) | (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 8) | site;
  atomicCAS(&g_goldfish_status, 0ULL, code);
}

// Bounded wait on an mbarrier phase by polling (a suspended wait slows the
// code after it); false (and an error word) on expiry.
__device__ __forceinline__ bool gf_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                        uint32_t site) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) {
      gf_record(site);
      return false;
    }
  }
}

// 1-D bulk copy global -> this CTA's shared memory with an L2 cache policy,
// completion counted on `bar` in bytes (both addresses 16-byte aligned, size
// a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bounded wait of a whole warp: lane 0 polls, then every lane tests the
// completed phase once (each lane's own acquire of the data it guards).  The
// barriers waited on this way cannot complete their next phase before this
// warp has released them, so the phase lane 0 saw is still the one tested.
__device__ __forceinline__ bool gf_warp_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             uint32_t site) {
  bool got = true;
  if ((threadIdx.x & 31) == 0) got = gf_wait(bar, parity, timeout_ns, site);
  got = __shfl_sync(0xFFFFFFFFu, got, 0) != 0;
  if (got) (void)mbar_test_wait(bar, parity);
  return got;
}

// L2 policy marking every line of an access evict-first.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy of this CTA's shared memory to global memory with an L2
// cache policy, in the thread's current bulk group (both addresses 16-byte
// aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the bulk groups of this thread have read their shared-memory
// sources (the buffers may then be rewritten).
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until the bulk groups of this thread have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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
    *reinterpret_cast<unsigned int*>(a.loss) = 0u;  // the rows kernel's row counter
  }
}

// ------------------------------------------------------------------ rows
struct RowParams {
  GoldfishArgs a;
  int chunks;  // copies per row: ceil(vpad / kGfChunk), vpad = V rounded up to 8
};

// Shared memory after the chunk buffers and the zeros.
struct alignas(16) GfTail {
  uint64_t full[kGfRing];
  uint64_t consumed[kGfRing];  // the consumer warps are done with a chunk
  uint64_t empty[kGfRing];     // the buffer may be refilled
  uint64_t rq_full[kGfRowQ];
  uint64_t rq_empty[kGfRowQ];
  int64_t rq_row[kGfRowQ];  // claimed row, or -1: no more rows for this CTA
  int32_t rq_y[kGfRowQ];
  int32_t rq_keep[kGfRowQ];
  float red_m[kGfConsumerWarps];
  float red_s[kGfConsumerWarps];
  float zy;  // the label's logit of the row in progress
};

// Barrier among the consumer warps only (the producer and store warps run
// on their own).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGfConsumers) : "memory");
}

// Barrier among the consumer warps that also ORs a predicate over them: every
// consumer gets the same answer.
__device__ __forceinline__ bool consumers_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kGfConsumers)
      : "memory");
  return r != 0;
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

// Warp 0 is the producer: lane 0 claims rows (atomic add on the counter),
// hands each to the other warps through a queue of kGfRowQ entries and, for
// a kept row, copies its chunks in order into the ring: the whole row for
// the first pass, then the whole row again for the second (only the first
// when no gradient is asked for).  Warp 1 stores: it zero-fills the
// gradient rows of dropped labels by bulk copies from a buffer of zeros,
// and copies each gradient chunk the consumers left in shared memory to its
// row with one bulk copy; it frees a buffer for the producer once the
// consumers are done with it and its bulk copy has read it.  Warps 2..17
// are the consumers.  All consumer threads wait on the same barriers and
// take every decision that ends the loop together (consumers_any), so their
// barrier counts always match.
__global__ void __launch_bounds__(kGfThreads, 1)
    goldfish_rows_kernel(const __grid_constant__ RowParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GoldfishArgs& a = p.a;
  const int64_t T = a.batch * a.seq;
  const int64_t V = a.vocab;
  const int64_t vpad = (V + 7) & ~int64_t{7};
  const int64_t vfull = V & ~int64_t{7};  // elements in whole 8-element vectors
  const int nch = p.chunks;
  const int passes = a.dlogits ? 2 : 1;
  const uint32_t zeros = smem_addr(smem) + static_cast<uint32_t>(kGfRing * kGfChunk * 2);
  GfTail* tl = reinterpret_cast<GfTail*>(smem + kGfRing * kGfChunk * 2 + kGfZeroBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns;
  auto buf = [&](int b) { return smem_addr(smem) + static_cast<uint32_t>(b * kGfChunk * 2); };

  for (int i = threadIdx.x; i < kGfZeroBytes / 16; i += blockDim.x)
    reinterpret_cast<int4*>(smem + kGfRing * kGfChunk * 2)[i] = make_int4(0, 0, 0, 0);
  fence_proxy_async_shared();  // the zeros, for the bulk copies that read them
  if (threadIdx.x == 0) {
    for (int b = 0; b < kGfRing; ++b) {
      mbar_init(smem_addr(&tl->full[b]), 1);
      mbar_init(smem_addr(&tl->consumed[b]), kGfConsumerWarps);
      mbar_init(smem_addr(&tl->empty[b]), 1);
    }
    for (int q = 0; q < kGfRowQ; ++q) {
      mbar_init(smem_addr(&tl->rq_full[q]), 1);
      mbar_init(smem_addr(&tl->rq_empty[q]), kGfConsumerWarps + 1);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      unsigned int* counter = reinterpret_cast<unsigned int*>(a.loss);
      const uint64_t keep_pol = l2_policy(true, 1.0f);
      const uint64_t drop_pol = evict_first_policy();
      int b = 0, q = 0;
      uint32_t ph = 0, qph = 0;
      uint32_t uses[kGfRing] = {};  // copies issued into each buffer
      bool ok = true;
      while (true) {
        ok = ok && gf_wait(smem_addr(&tl->rq_empty[q]), qph ^ 1u, tmo, 1);
        const int64_t r = ok ? static_cast<int64_t>(atomicAdd(counter, 1u)) : T;
        const bool more = r < T;
        const int32_t keep = more ? a.keep[r] : 0;
        tl->rq_row[q] = more ? r : -1;
        tl->rq_y[q] = more ? a.labels[r] : 0;
        tl->rq_keep[q] = keep;
        mbar_arrive(smem_addr(&tl->rq_full[q]));
        if (++q == kGfRowQ) {
          q = 0;
          qph ^= 1u;
        }
        if (!more) break;
        if (!keep || a.inject == 1) continue;  // (the test hook withholds every copy)
        const uint16_t* src = a.logits + r * a.ld_logits;
        for (int pass = 0; pass < passes && ok; ++pass) {
          for (int c = 0; c < nch; ++c) {
            ok = gf_wait(smem_addr(&tl->empty[b]), ph ^ 1u, tmo, 2);
            if (!ok) break;
            const int64_t e0 = c * kGfChunk;
            const uint32_t bytes = static_cast<uint32_t>(min(kGfChunk, vpad - e0) * 2);
            const uint32_t fb = smem_addr(&tl->full[b]);
            mbar_arrive_expect_tx(fb, bytes);
            bulk_load(buf(b), src + e0, bytes, fb, pass == 0 ? keep_pol : drop_pol);
            ++uses[b];
            if (++b == kGfRing) {
              b = 0;
              ph ^= 1u;
            }
          }
        }
      }
      // Copies nobody took exist only after an expired wait: let them land
      // (bounded) before this CTA's shared memory goes away.
      if (!ok)
        for (int i = 0; i < kGfRing; ++i)
          if (uses[i] > 0) gf_wait(smem_addr(&tl->full[i]), (uses[i] - 1) & 1u, tmo, 3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ stores
    const uint64_t pol = evict_first_policy();
    int b = 0, q = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true;
    while (ok) {
      ok = gf_warp_wait(smem_addr(&tl->rq_full[q]), qph, tmo, 6);
      const int64_t r = tl->rq_row[q];
      const bool keep = tl->rq_keep[q] != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tl->rq_empty[q]));
      if (++q == kGfRowQ) {
        q = 0;
        qph ^= 1u;
      }
      if (!ok || r < 0) break;
      uint16_t* out = a.dlogits ? a.dlogits + r * a.ld_dlogits : nullptr;
      if (!keep) {
        if (out) {
          if (lane == 0) {
            for (int64_t e = 0; e < vfull; e += kGfZeroBytes / 2)
              bulk_store(out + e, zeros,
                         static_cast<uint32_t>(min(int64_t{kGfZeroBytes / 2}, vfull - e) * 2), pol);
            bulk_commit();
          }
          for (int64_t i = vfull + lane; i < V; i += 32) out[i] = 0;
        }
        continue;
      }
      for (int pass = 0; pass < passes && ok; ++pass) {
        for (int c = 0; c < nch; ++c) {
          ok = gf_warp_wait(smem_addr(&tl->consumed[b]), ph, tmo, 7);
          if (!ok) break;
          if (lane == 0) {
            if (pass == 1) {
              const int64_t e0 = c * kGfChunk;
              const int64_t nb = max(int64_t{0}, min(kGfChunk, vfull - e0));  // whole vectors
              if (nb > 0) {
                bulk_store(out + e0, buf(b), static_cast<uint32_t>(nb * 2), pol);
                bulk_commit();
                bulk_wait_read();
              }
            }
            mbar_arrive(smem_addr(&tl->empty[b]));
          }
          __syncwarp();
          if (++b == kGfRing) {
            b = 0;
            ph ^= 1u;
          }
        }
      }
    }
    // the gradient's bulk copies complete before the kernel does
    if (lane == 0) bulk_wait_all();
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 2;          // consumer warp
    const int ct = threadIdx.x - 64;  // consumer thread
    const int32_t n = *a.kept;
    const float inv_n = n > 0 ? 1.0f / static_cast<float>(n) : 0.0f;
    const float log2n = n > 0 ? log2f(static_cast<float>(n)) : 0.0f;
    int b = 0, q = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true;  // this thread's waits all completed
    // waits for chunk b, passes it to f(x, e0, n_valid) when it arrived, and
    // reports the warp done with it
    auto take_chunk = [&](int c, auto&& f) {
      const bool got = ok && gf_warp_wait(smem_addr(&tl->full[b]), ph, tmo, 4);
      ok = got;
      const int64_t e0 = c * kGfChunk;
      const int64_t nv = max(int64_t{0}, min(kGfChunk, V - e0));
      if (got) f(reinterpret_cast<uint16_t*>(smem + b * kGfChunk * 2), e0, nv);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tl->consumed[b]));
      if (++b == kGfRing) {
        b = 0;
        ph ^= 1u;
      }
    };
    while (true) {
      ok = ok && gf_warp_wait(smem_addr(&tl->rq_full[q]), qph, tmo, 5);
      const int64_t r = tl->rq_row[q];
      const int32_t y = tl->rq_y[q];
      const bool keep = tl->rq_keep[q] != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tl->rq_empty[q]));
      if (++q == kGfRowQ) {
        q = 0;
        qph ^= 1u;
      }
      if (consumers_any(!ok || r < 0)) break;
      if (!keep) {  // the store warp writes its zero gradient row
        if (ct == 0) a.token_loss[r] = 0.0f;
        continue;
      }
      // 1. (max, sum of exp) of the row, and the label's logit
      float m0 = -INFINITY, s0 = 0.0f, m1 = -INFINITY, s1 = 0.0f;
      for (int c = 0; c < nch; ++c)
        take_chunk(c, [&](const uint16_t* x, int64_t e0, int64_t nv) {
          const int64_t vf = nv & ~int64_t{7};
          for (int64_t i = 16 * ct; i < vf; i += 16 * kGfConsumers) {
            float xa[8];
            unpack8(*reinterpret_cast<const uint4*>(x + i), xa);
            online_add8(m0, s0, xa);
            if (i + 8 < vf) {
              float xb[8];
              unpack8(*reinterpret_cast<const uint4*>(x + i + 8), xb);
              online_add8(m1, s1, xb);
            }
          }
          for (int64_t i = vf + ct; i < nv; i += kGfConsumers) online_add1(m1, s1, bf16_to_f32(x[i]));
          if (ct == 0 && y >= e0 && y < e0 + nv) tl->zy = bf16_to_f32(x[y - e0]);
        });
      float m = fmaxf(m0, m1);
      float sm = (m0 > -INFINITY ? s0 * fast_exp2((m0 - m) * kLog2e) : 0.0f) +
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
      float S = 0.0f;
#pragma unroll
      for (int w = 0; w < kGfConsumerWarps; ++w) S += tl->red_s[w];
      const float lse = M + log2f(S) * kLn2;
      if (ct == 0) a.token_loss[r] = lse - tl->zy;
      // red_m, red_s and zy are rewritten only after every consumer has read
      // them: the next row's first write follows at least one more barrier
      // (consumers_any) that every consumer reaches after these reads.
      if (!a.dlogits) continue;
      // 2. gradient: p / n = 2^(z log2e - (lse log2e + log2 n)), the 1/n
      //    folded into the exponent; the label's entry less 1/n.  Whole
      //    vectors go back into the chunk's buffer for the store warp's bulk
      //    copy; the row's last (V mod 8) elements are stored here.
      const float lb = fmaf(lse, kLog2e, log2n);
      uint16_t* out = a.dlogits + r * a.ld_dlogits;
      for (int c = 0; c < nch; ++c)
        take_chunk(c, [&](uint16_t* x, int64_t e0, int64_t nv) {
          const int64_t yl = y - e0;  // the label's place in this chunk (may be outside)
          const int64_t vf = nv & ~int64_t{7};
          for (int64_t i = 8 * ct; i < vf; i += 8 * kGfConsumers) {
            float g[8];
            unpack8(*reinterpret_cast<const uint4*>(x + i), g);
#pragma unroll
            for (int j = 0; j < 8; ++j) g[j] = fast_exp2(fmaf(g[j], kLog2e, -lb));
            const int64_t d = yl - i;  // the label's element, if in this vector
            if (d >= 0 && d < 8) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (j == d) g[j] -= inv_n;
            }
            *reinterpret_cast<uint4*>(x + i) =
                make_uint4(pack2(g[0], g[1]), pack2(g[2], g[3]), pack2(g[4], g[5]), pack2(g[6], g[7]));
          }
          for (int64_t i = vf + ct; i < nv; i += kGfConsumers) {
            float gs = fast_exp2(fmaf(bf16_to_f32(x[i]), kLog2e, -lb));
            if (i == yl) gs -= inv_n;
            __nv_bfloat16 h = __float2bfloat16_rn(gs);
            out[e0 + i] = *reinterpret_cast<uint16_t*>(&h);
          }
          fence_proxy_async_shared();  // these writes, for the store warp's bulk copy
        });
    }
  }
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

bool goldfish_vocab_supported(int64_t vocab) { return vocab >= 1 && vocab <= kGoldfishMaxVocab; }

cudaError_t goldfish_launch(const GoldfishArgs& a, int sms, cudaStream_t stream) {
  const int64_t T = a.batch * a.seq;
  goldfish_mask_kernel<<<1, kMaskThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (T > 0) {
    RowParams p;
    p.a = a;
    const int64_t vpad = (a.vocab + 7) / 8 * 8;
    p.chunks = static_cast<int>((vpad + kGfChunk - 1) / kGfChunk);
    const int smem = static_cast<int>(kGfRing * kGfChunk * 2 + kGfZeroBytes + sizeof(GfTail));
    e = cudaFuncSetAttribute(goldfish_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // Persistent: one CTA per SM, at most one per row.
    const int64_t ctas = std::min<int64_t>(sms, T);
    goldfish_rows_kernel<<<static_cast<unsigned>(ctas), kGfThreads, smem, stream>>>(p);
    e = cudaGetLastError();
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
