// C ABI of the FC-layer GEMM library: argument checks, 3D-grid block
// resolution, TMA tensor-map encoding and kernel launches.  Declarations and
// the contract of every entry point are in include/axonn_fc.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cerrno>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <mutex>
#include <sstream>
#include <string>
#include <unordered_map>
#include <vector>

#include "axonn_fc.h"
#include "gemm_kernel.cuh"
#include "goldfish.h"
#include "kernel_launch.h"

namespace {

using axonn::GemmParams;
using axonn::ProblemDesc;

constexpr int kMaxProblems = 64;  // largest virtual grid Gx*Gy*Gz
// The kernel parameter block holds a tensor-map pair per problem, so a
// launch with few problems uses a smaller instantiation (less to copy per
// launch): 1 problem, up to kFewProblems, or up to kMaxProblems.
constexpr int kFewProblems = 8;

thread_local std::string t_last_error;
std::atomic<uint64_t> g_timeout_ns{4000000000ULL};
std::atomic<int> g_inject{0};
std::atomic<int> g_pdl{1};  // GEMMs launched as programmatic dependent launches
// L2 bytes a rasterisation group's kept operand panel may claim as
// evict-last lines (0: no L2 hints on the operand loads)
std::atomic<int64_t> g_l2_budget{int64_t{64} << 20};

axonn_status_t fail(axonn_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

axonn_status_t ok() {
  t_last_error.clear();
  return AXONN_OK;
}

// ------------------------------------------------------------------ driver
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Per-device facts and one-time kernel attributes.
struct DeviceState {
  int sms = 0;
  int max_pairs = 0;  // CTA pairs (clusters of 2) resident at once
  // Clusters of the reduction-split kernels resident at once, by tile
  // ([0] 128 x 128, [1] 128 x 64) and pieces ([1] 2, [2] 4, [3] 8).
  int split_clusters[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
  bool attrs_set = false;
};

// Per-device state lives in a fixed table so that pointers handed out stay
// valid while other threads initialise other devices.
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceState g_devs[kMaxDevices];

// Host threads that never touched the runtime have no current context, and
// the driver call that encodes tensor maps needs one: make the current
// device's primary context current, once per thread and device.
thread_local int t_context_device = -1;

axonn_status_t device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(AXONN_ERR_UNSUPPORTED, "device index %d", dev);
  if (t_context_device != dev) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "cudaSetDevice(%d): %s", dev, cudaGetErrorString(e));
    t_context_device = dev;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_devs[dev];
  if (!d.attrs_set) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(AXONN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    bool split_ok = true;
    const cudaError_t es[] = {axonn::kernels_init<1>(&split_ok),
                              axonn::kernels_init<kFewProblems>(&split_ok),
                              axonn::kernels_init<kMaxProblems>(&split_ok)};
    for (cudaError_t x : es)
      if (x != cudaSuccess)
        return fail(AXONN_ERR_CUDA, "kernel attributes: %s", cudaGetErrorString(x));
    if (!split_ok)
      return fail(AXONN_ERR_UNSUPPORTED,
                  "a 12-warp GEMM kernel was not built with %d registers per thread",
                  axonn::kRegsAtLaunch);
    int clusters = 0;
    if (axonn::pair_clusters_resident(d.sms, &clusters) != cudaSuccess || clusters <= 0) {
      (void)cudaGetLastError();
      clusters = d.sms / 2;
    }
    d.max_pairs = clusters;
    e = axonn::split_kernel_init();
    if (e != cudaSuccess)
      return fail(AXONN_ERR_CUDA, "split kernel attributes: %s", cudaGetErrorString(e));
    for (int t = 0; t < 2; ++t)
      for (int lg = 1; lg <= 3; ++lg) {
        int n = 0;
        if (axonn::split_clusters_resident(d.sms, 1 << lg, t == 0 ? 128 : 64, &n) != cudaSuccess ||
            n <= 0) {
          (void)cudaGetLastError();
          n = 0;  // this split is not offered on the device
        }
        d.split_clusters[t][lg] = n;
      }
    d.attrs_set = true;
  }
  *out = &d;
  return AXONN_OK;
}

// ------------------------------------------------------------------ grid
void split_range(int64_t D, int64_t G, int64_t b, int64_t* s, int64_t* e) {
  const int64_t units = (D + 7) / 8;
  const int64_t base = units / G, rem = units % G;
  const int64_t start = 8 * (b * base + (b < rem ? b : rem));
  const int64_t n = base + (b < rem ? 1 : 0);
  *s = start < D ? start : D;
  const int64_t stop = start + 8 * n;
  *e = stop < D ? stop : D;
}

struct Range {
  int64_t s = 0, e = 0;
  int64_t len() const { return e - s; }
};

// The op as C[M x N] = A[M x R] . B[R x N] over full logical matrices.
struct OpView {
  const char* A;
  int64_t lda;
  bool a_mn;  // A(i, r) at A + (r*lda + i) (M-contiguous) else A + (i*lda + r)
  const char* B;
  int64_t ldb;
  bool b_mn;  // B(r, j) at B + (r*ldb + j) (N-contiguous) else B + (j*ldb + r)
  char* C;
  int64_t ldc;
  int64_t M, N, R;
};

// Logical ranges of block (x,y,z): output rows, reduced range, output cols.
void block_ranges(int op, const axonn_fc_shape_t& s, int x, int y, int z, Range* rows, Range* red,
                  Range* cols) {
  Range Tz, Kx, Ny;
  split_range(s.T, s.gz, z, &Tz.s, &Tz.e);
  split_range(s.K, s.gx, x, &Kx.s, &Kx.e);
  split_range(s.N, s.gy, y, &Ny.s, &Ny.e);
  if (op == AXONN_OP_FWD) {  // Y[Tz,Ny] += X[Tz,Kx] W[Kx,Ny]
    *rows = Tz; *red = Kx; *cols = Ny;
  } else if (op == AXONN_OP_DGRAD) {  // dX[Tz,Kx] += dY[Tz,Ny] W[Kx,Ny]^T
    *rows = Tz; *red = Ny; *cols = Kx;
  } else {  // dW[Kx,Ny] += X[Tz,Kx]^T dY[Tz,Ny]
    *rows = Kx; *red = Tz; *cols = Ny;
  }
}

int reduce_extent(int op, const axonn_fc_shape_t& s) {
  return op == AXONN_OP_FWD ? s.gx : (op == AXONN_OP_DGRAD ? s.gy : s.gz);
}

int reduce_coord(int op, int x, int y, int z) {
  return op == AXONN_OP_FWD ? x : (op == AXONN_OP_DGRAD ? y : z);
}

void full_dims(int op, const axonn_fc_shape_t& s, int64_t* M, int64_t* N, int64_t* R) {
  if (op == AXONN_OP_FWD) { *M = s.T; *N = s.N; *R = s.K; }
  else if (op == AXONN_OP_DGRAD) { *M = s.T; *N = s.K; *R = s.N; }
  else { *M = s.K; *N = s.N; *R = s.T; }
}

constexpr uint32_t kKnownFlags = AXONN_A_T | AXONN_B_T | AXONN_ACCUM_F32 | AXONN_VGRID |
                                 AXONN_FULL_OPERANDS | AXONN_OUT_F32 | AXONN_ZSHARDED |
                                 AXONN_REDUCE_ADD | AXONN_VGRID_PARTIALS;

axonn_status_t check_shape(int op, const axonn_fc_shape_t* s, uint32_t flags) {
  if (op < AXONN_OP_FWD || op > AXONN_OP_WGRAD) return fail(AXONN_ERR_INVALID_ARG, "bad op %d", op);
  if (!s) return fail(AXONN_ERR_INVALID_ARG, "shape is NULL");
  if (flags & ~kKnownFlags) return fail(AXONN_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~kKnownFlags);
  if ((flags & AXONN_ACCUM_F32) && (flags & AXONN_OUT_F32))
    return fail(AXONN_ERR_INVALID_ARG, "AXONN_ACCUM_F32 and AXONN_OUT_F32 are exclusive");
  if ((flags & AXONN_REDUCE_ADD) && (flags & (AXONN_VGRID | AXONN_ACCUM_F32)) != (AXONN_VGRID | AXONN_ACCUM_F32))
    return fail(AXONN_ERR_INVALID_ARG, "AXONN_REDUCE_ADD needs AXONN_VGRID and AXONN_ACCUM_F32");
  if ((flags & AXONN_VGRID_PARTIALS) && !(flags & AXONN_VGRID))
    return fail(AXONN_ERR_INVALID_ARG, "AXONN_VGRID_PARTIALS needs AXONN_VGRID");
  if ((flags & AXONN_VGRID_PARTIALS) && (flags & AXONN_REDUCE_ADD))
    return fail(AXONN_ERR_INVALID_ARG, "AXONN_VGRID_PARTIALS and AXONN_REDUCE_ADD are exclusive");
  if (s->T < 0 || s->K < 0 || s->N < 0) return fail(AXONN_ERR_INVALID_ARG, "negative extent");
  const int64_t lim = (int64_t{1} << 31) - 256;
  if (s->T > lim || s->K > lim || s->N > lim) return fail(AXONN_ERR_UNSUPPORTED, "extent above 2^31");
  if (s->gx < 1 || s->gy < 1 || s->gz < 1) return fail(AXONN_ERR_INVALID_ARG, "grid extents must be >= 1");
  if (static_cast<int64_t>(s->gx) * s->gy * s->gz > kMaxProblems)
    return fail(AXONN_ERR_UNSUPPORTED, "grid %dx%dx%d has more than %d blocks", s->gx, s->gy, s->gz,
                kMaxProblems);
  if (!(flags & AXONN_VGRID)) {
    if (s->x < 0 || s->x >= s->gx || s->y < 0 || s->y >= s->gy || s->z < 0 || s->z >= s->gz)
      return fail(AXONN_ERR_INVALID_ARG, "block (%d,%d,%d) outside grid %dx%dx%d", s->x, s->y, s->z,
                  s->gx, s->gy, s->gz);
  }
  return AXONN_OK;
}

size_t vgrid_ws_bytes(int op, const axonn_fc_shape_t& s, uint32_t flags) {
  if (!(flags & AXONN_VGRID) || !(flags & AXONN_VGRID_PARTIALS)) return 0;
  const int G = reduce_extent(op, s);
  if (G <= 1) return 0;
  int64_t M, N, R;
  full_dims(op, s, &M, &N, &R);
  const int64_t ldp = (N + 7) / 8 * 8;
  // Partials 0..G-2 go to the workspace; the last block's epilogue adds
  // them to its own accumulator and writes the output.
  return static_cast<size_t>(G - 1) * static_cast<size_t>(M) * static_cast<size_t>(ldp) * 4u;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks one stored operand: pointer, leading dimension, alignment.
axonn_status_t check_operand(const char* name, const void* p, int64_t ld, int64_t rows,
                             int64_t cols) {
  if (rows == 0 || cols == 0) return AXONN_OK;
  if (!p) return fail(AXONN_ERR_INVALID_ARG, "%s is NULL", name);
  if (ld < cols) return fail(AXONN_ERR_INVALID_ARG, "%s: leading dimension %lld < row length %lld", name,
                             (long long)ld, (long long)cols);
  if (!aligned16(p)) return fail(AXONN_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  if (ld % 8 != 0) return fail(AXONN_ERR_ALIGNMENT, "%s: leading dimension %lld is not a multiple of 8", name,
                               (long long)ld);
  if (ld * 2 >= (int64_t{1} << 40)) return fail(AXONN_ERR_UNSUPPORTED, "%s: stride too large", name);
  return AXONN_OK;
}

axonn_status_t encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                         int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  // A box row of 128 B takes the 128-byte swizzle, one of 64 B the 64-byte.
  const CUtensorMapSwizzle swz =
      box_inner * 2 >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  auto fn = encode_fn();
  if (!fn) return fail(AXONN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(AXONN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return AXONN_OK;
}

// MN-major operand stored [R rows x MN] as a 3-D map {64, R, MN/64} (chunk
// stride 128 B): one box {64, bk, chunks} loads every 64-wide chunk of a
// tile.  Needs MN % 64 == 0 so that no chunk runs past the end of a row;
// chunks past the last one are zero-filled like any out-of-range box.
axonn_status_t encode_mn_3d(CUtensorMap* m, const void* base, uint64_t mn, uint64_t r, int64_t ld,
                            uint32_t bk, uint32_t chunks) {
  auto fn = encode_fn();
  if (!fn) return fail(AXONN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[3] = {64, r, mn / 64};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, 128};
  cuuint32_t box[3] = {64, bk, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rr = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rr != CUDA_SUCCESS)
    return fail(AXONN_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", static_cast<int>(rr));
  return AXONN_OK;
}

// tcgen05 instruction descriptor, kind::f16: bf16 A and B, fp32 D.
uint32_t make_idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// One block product to run: operand bases and extents, output and mode.
struct Block {
  const char* A;
  const char* B;
  char* C;
  int64_t ldc;
  int64_t M, N, R;
  int out_mode;
  // Chains: the head of a run of `chain` consecutive blocks (same output,
  // same M x N) whose products all add into one accumulator, in order; the
  // members after the head have chain = 0.  An ordinary block has chain = 1.
  int chain = 1;
  bool out_t = false;          // computes the transpose (operand roles swapped)
  int phase = 1;               // 0: writes an fp32 partial that a phase-1 block reads
  int red_count = 0;           // partials to add in the epilogue (last partial only)
  const float* red_src = nullptr;
  int64_t red_stride = 0, red_ld = 0;
};

// Kernel configurations the library can run.  A configuration fixes the
// output tile, whether a CTA pair shares each MMA, and the ring depth.
struct KernelConfig {
  const char* name;
  int bm, bn;   // output tile of one CTA (or CTA pair)
  int bk;       // reduction depth of one pipeline stage
  bool pair;    // cta_group::2 across a cluster of 2
  int mma_m;    // rows of one tcgen05.mma
};
constexpr KernelConfig kConfigs[] = {
    {"1cta_128x128", 128, 128, 64, false, 128},
    {"1cta_128x256", 128, 256, 64, false, 128},
    {"pair_256x256", 256, 256, 64, true, 256},
    {"1cta_256x256", 256, 256, 64, false, 128},
    {"1cta_128x192", 128, 192, 64, false, 128},
    {"1cta_256x192", 256, 192, 64, false, 128},
    {"pair_512x256", 512, 256, 64, true, 256},
    {"1cta_128x64", 128, 64, 64, false, 128},
};
// Throughput of each configuration relative to 1cta_128x256 on full waves
// (measured on GB300 over the 12 GEMMs of a GPT block, H = 6144; the
// 128x64 tile on an 8192 x 6144 x 6144 forward product).  The 128x64 tile
// reads 1.5x the operand bytes per FLOP of 128x128: it is for products with
// too few larger tiles to fill the GPU.
constexpr double kConfigSpeed[] = {0.68, 1.0, 0.92, 1.06, 0.92, 1.12, 1.2, 0.36};
constexpr int kNumConfigs = static_cast<int>(sizeof(kConfigs) / sizeof(kConfigs[0]));
static_assert(kNumConfigs == axonn::kKernelConfigs, "configuration table and kernel instantiations");
std::atomic<int> g_forced_config{-1};
thread_local int t_last_config = -1;

// Stream-K modes: off; on when the partial round is at most a quarter full
// (the default); on whenever the launch allows it.
enum StreamKMode : int { kStreamKOff = 0, kStreamKShortTail = 1, kStreamKAlways = 2 };

struct LaunchPlan {
  int config = 1;
  int group_m = 16;
  std::vector<Block> blocks;
  int streamk = kStreamKOff;
  int split = 1;       // pieces of the reduction split (cluster size), 1 = none
  void* ws = nullptr;  // workspace for the stream-K partials and counters
  size_t ws_bytes = 0;
};

// One way to run a call: kernel configuration, split of the reduction range
// into `split` pieces summed in fixed order inside a cluster (configuration
// 0 only), and the rasterisation group height.
struct TuneChoice {
  int config = -1;
  int split = 1;
  int group_m = 16;
  int streamk = 1;  // StreamKMode (see configure_streamk)
  int swap = 0;     // 1: run C^T = B^T . A^T (operand roles exchanged)
};
std::atomic<int> g_forced_streamk{-1};
std::atomic<int> g_forced_swap{-1};
thread_local TuneChoice t_last_choice;

struct TuneEntry {
  TuneChoice choice;
  double us = 0;
};
std::mutex g_tune_mu;
std::unordered_map<std::string, TuneEntry> g_tune;  // call signature -> fastest choice

constexpr int kMaxSplit = 8;
constexpr int64_t kSplitMinR = 128;

template <int MAXP>
axonn_status_t fill_params(GemmParams<MAXP>& P, const OpView& v, const std::vector<Block>& blocks,
                           const KernelConfig& c, int group_m) {
  static_assert(sizeof(GemmParams<MAXP>) < 32000, "kernel parameter space");
  memset(&P, 0, sizeof(P));
  // Rows of A and columns of B that one CTA loads per stage (A in boxes of
  // 128 rows, or one 3-D box of all its rows).
  const uint32_t a_rows = 128;
  const uint32_t cta_rows = c.pair ? c.bm / 2 : c.bm;
  const uint32_t b_cols = c.pair ? c.bn / 2 : c.bn;
  const uint32_t bk = static_cast<uint32_t>(c.bk);
  int64_t tiles = 0;
  int np = 0, nmaps = 0;
  for (size_t bi = 0; bi < blocks.size();) {
    const Block& b = blocks[bi];
    const size_t members = static_cast<size_t>(b.chain > 0 ? b.chain : 1);
    if (b.chain <= 0 || bi + members > blocks.size())
      return fail(AXONN_ERR_INVALID_ARG, "malformed chain of block products");
    const size_t next = bi + members;
    if (b.M == 0 || b.N == 0) {
      bi = next;
      continue;
    }
    if (np >= MAXP) return fail(AXONN_ERR_UNSUPPORTED, "too many block products");
    if (tiles + ((b.M + c.bm - 1) / c.bm) * ((b.N + c.bn - 1) / c.bn) > (int64_t{1} << 30))
      return fail(AXONN_ERR_UNSUPPORTED, "more than 2^30 output tiles in one launch");
    ProblemDesc& d = P.prob[np];
    d.C = b.C;
    d.ldc = b.ldc;
    d.M = static_cast<int32_t>(b.M);
    d.N = static_cast<int32_t>(b.N);
    d.tiles_m = static_cast<int32_t>((b.M + c.bm - 1) / c.bm);
    d.tiles_n = static_cast<int32_t>((b.N + c.bn - 1) / c.bn);
    d.tile_start = static_cast<int32_t>(tiles);
    d.a_mn = v.a_mn;
    d.b_mn = v.b_mn;
    d.idesc = make_idesc(c.mma_m, c.bn, v.a_mn, v.b_mn);
    d.out_mode = b.out_mode;
    d.red_count = b.red_count;
    d.red_src = b.red_src;
    d.red_stride = b.red_stride;
    d.red_ld = b.red_ld;
    d.out_t = b.out_t;
    d.fast_bf16 = !b.out_t && b.out_mode == axonn::kOutBF16 && b.red_count == 0 &&
                  reinterpret_cast<uintptr_t>(b.C) % 32 == 0 && b.ldc % 16 == 0;
    d.a_3d = v.a_mn && b.M % 64 == 0;
    d.b_3d = v.b_mn && b.N % 64 == 0;
    // One tensor-map pair per member with a non-empty reduction, each with
    // the member's own extents (loads past them read zeros).
    d.map0 = nmaps;
    d.chain = 0;
    int64_t steps = 0, red = 0;
    for (size_t g = bi; g < next; ++g) {
      const Block& m = blocks[g];
      if (m.M != b.M || m.N != b.N || m.out_t != b.out_t || (g > bi && m.chain != 0))
        return fail(AXONN_ERR_INVALID_ARG, "chain members differ in output extent");
      if (m.R == 0) continue;
      if (nmaps >= MAXP) return fail(AXONN_ERR_UNSUPPORTED, "too many block products");
      axonn_status_t s;
      CUtensorMap* ta = &P.tma[nmaps];
      CUtensorMap* tb = &P.tmb[nmaps];
      if (d.a_3d) s = encode_mn_3d(ta, m.A, m.M, m.R, v.lda, bk, cta_rows / 64);
      else if (v.a_mn) s = encode_2d(ta, m.A, m.M, m.R, v.lda, 64, bk);
      else s = encode_2d(ta, m.A, m.R, m.M, v.lda, bk, a_rows);
      if (s != AXONN_OK) return s;
      if (d.b_3d) s = encode_mn_3d(tb, m.B, m.N, m.R, v.ldb, bk, b_cols / 64);
      else if (v.b_mn) s = encode_2d(tb, m.B, m.N, m.R, v.ldb, 64, bk);
      else s = encode_2d(tb, m.B, m.R, m.N, v.ldb, bk, b_cols);
      if (s != AXONN_OK) return s;
      P.map_nk[nmaps] = static_cast<int32_t>((m.R + c.bk - 1) / c.bk);
      steps += P.map_nk[nmaps];
      red += m.R;
      ++d.chain;
      ++nmaps;
    }
    if (steps >= (int64_t{1} << 30)) return fail(AXONN_ERR_UNSUPPORTED, "reduction too long");
    if (d.chain == 0) {  // empty reduction: no loads, the epilogue writes zeros
      d.chain = 1;
      d.map0 = 0;
    }
    d.num_k = static_cast<int32_t>(steps);
    d.R = static_cast<int32_t>(std::min<int64_t>(red, INT32_MAX));
    // L2 priorities: the group's panel of the operand it walks along (A for
    // groups of tile rows, B for groups of tile columns) is kept, as much of
    // it as the budget allows.  Marking the other operand evict-first as
    // well was measured: the same step time and 23 % more DRAM traffic (the
    // wave's tiles drift apart in the reduction and re-read its panels).
    const int64_t budget = g_l2_budget.load();
    if (budget > 0 && group_m != 0) {
      const bool rows = group_m > 0;
      const int64_t g = std::min<int64_t>(rows ? group_m : -group_m, rows ? d.tiles_m : d.tiles_n);
      const int64_t panel = g * (rows ? c.bm : c.bn) * std::max<int64_t>(red, 1) * 2;
      d.l2_keep = rows ? 1 : 2;
      d.l2_keep_frac = panel <= budget ? 1.0f
                                       : std::max(1.0f / 64.0f, static_cast<float>(budget) / panel);
    }
    tiles += d.tiles_m * d.tiles_n;
    ++np;
    bi = next;
  }
  P.num_problems = np;
  P.num_maps = nmaps;
  P.total_tiles = static_cast<int32_t>(tiles);
  P.group_m = group_m;
  P.inject = g_inject.load();
  P.timeout_ns = g_timeout_ns.load();
  return AXONN_OK;
}

// Stream-K tail of a single-problem launch over `units` persistent CTAs (or
// CTA pairs): when the tiles do not fill a whole number of rounds, the last
// partial round and one full round (at least `units` tiles) are cut by
// reduction steps into equal consecutive ranges, one per unit, so every unit
// finishes at about the same time.  Units then start their ranges at
// different reduction offsets, so units working on neighbouring tiles no
// longer read the same operand panels at the same time.  When a unit's share
// is close to one tile (a partial round at most a quarter full) the offsets
// stay close and the tail is faster.  Otherwise the lost L2 reuse can cost
// more than the idle SMs it saves, so kStreamKShortTail applies it only in
// the first case.  A tile is cut into at most two pieces; whichever piece
// finishes second adds the other's fp32 partial to its own accumulator.
// Two fp32 terms sum alike in either order, so the result does not depend on
// which finishes second, and no piece waits for another (see epilogue_item).
// Workspace: a block of kStreamKFlagBytes for the counters (zeroed, in stream
// order, before the launch) followed by two tile-sized fp32 slots per unit.
constexpr size_t kStreamKFlagBytes = 16384;  // 16 counters per unit, up to 256 units
thread_local int t_last_sk_tiles = 0;
size_t streamk_ws_bytes(const KernelConfig& c, int units) {
  return kStreamKFlagBytes + 2 * static_cast<size_t>(units) * c.bm * c.bn * 4;
}

// Zeroes the stream-K counters.  A one-block kernel on the GEMM's own stream
// rather than cudaMemsetAsync: a memset can be carried out by a copy engine
// and then queues behind large host<->device copies running on other
// streams, which held each GEMM back in a copy-overlapped pipeline.
__global__ void zero_counters_kernel(uint32_t* p, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0u;
}

template <int MAXP>
axonn_status_t configure_streamk(GemmParams<MAXP>& P, const KernelConfig& c, int units,
                                 const LaunchPlan& plan, cudaStream_t stream) {
  const int T = P.total_tiles;
  t_last_sk_tiles = 0;
  if (plan.streamk == kStreamKOff || P.num_problems != 1 || units <= 0 || T <= units ||
      T % units == 0)
    return AXONN_OK;
  if (plan.streamk == kStreamKShortTail && 4 * (T % units) > units) return AXONN_OK;
  const int nk = P.prob[0].num_k;
  const int S = T >= 2 * units ? units + T % units : T;
  if (nk < 2 || static_cast<int64_t>(S) * nk >= (int64_t{1} << 31)) return AXONN_OK;
  const int counters = units * axonn::kSkCountersPerUnit;
  if (static_cast<size_t>(counters) * 4 > kStreamKFlagBytes || !plan.ws ||
      plan.ws_bytes < streamk_ws_bytes(c, units) || (reinterpret_cast<uintptr_t>(plan.ws) & 255u) != 0)
    return AXONN_OK;
  zero_counters_kernel<<<1, 256, 0, stream>>>(static_cast<uint32_t*>(plan.ws), counters);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "stream-K counters: %s", cudaGetErrorString(e));
  P.sk_tiles = S;
  t_last_sk_tiles = S;
  P.sk_slot_floats = c.bm * c.bn;
  P.sk_flags = static_cast<uint32_t*>(plan.ws);
  P.sk_partials = reinterpret_cast<float*>(static_cast<char*>(plan.ws) + kStreamKFlagBytes);
  return AXONN_OK;
}

// The reduction split runs on configurations 0 (128 x 128 tiles) and 7
// (128 x 64): the kernels that hold a split tile's staging rows and inbox
// beside their operand rings.  Index of the configuration's split kernel.
bool split_config(int c) { return c == 0 || c == 7; }
int split_index(int c) { return c == 7 ? 1 : 0; }
int split_lg(int split) { return split == 2 ? 1 : (split == 4 ? 2 : 3); }

// One launch of configuration `config` over the plan's blocks: the
// persistent grid is one unit (CTA, or CTA pair) per resident slot, or one
// per tile when there are fewer tiles.
template <int P1>
axonn_status_t launch_cfg(int config, const OpView& v, const LaunchPlan& plan,
                          const DeviceState& dev, cudaStream_t stream) {
  GemmParams<P1> P;
  axonn_status_t st = fill_params(P, v, plan.blocks, kConfigs[config], plan.group_m);
  if (st != AXONN_OK || P.num_problems == 0) return st;
  const int slots = kConfigs[config].pair ? dev.max_pairs : dev.sms;
  const int units = P.total_tiles < slots ? P.total_tiles : slots;
  if (plan.split > 1) {
    // The reduction split: clusters of plan.split CTAs, one tile per
    // cluster at a time, as many clusters as are resident at once.
    t_last_sk_tiles = 0;
    if constexpr (P1 == 1) {
      if (!split_config(config) || P.num_problems != 1 || (plan.split & (plan.split - 1)) ||
          plan.split > 8)
        return fail(AXONN_ERR_UNSUPPORTED, "reduction split of %d pieces not available here", plan.split);
      const int resident = dev.split_clusters[split_index(config)][split_lg(plan.split)];
      if (resident <= 0)
        return fail(AXONN_ERR_UNSUPPORTED, "reduction split of %d pieces not available here", plan.split);
      const int clusters = P.total_tiles < resident ? P.total_tiles : resident;
      const cudaError_t e = axonn::split_kernel_launch(P, plan.split, clusters, kConfigs[config].bn,
                                                       g_pdl.load() != 0, stream);
      if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "split GEMM launch: %s", cudaGetErrorString(e));
      return AXONN_OK;
    } else {
      return fail(AXONN_ERR_UNSUPPORTED, "reduction split of a multi-product launch");
    }
  }
  st = configure_streamk(P, kConfigs[config], units, plan, stream);
  if (st != AXONN_OK) return st;
  const cudaError_t e = axonn::kernels_launch<P1>(config, P, units, g_pdl.load() != 0, stream);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
  return AXONN_OK;
}

axonn_status_t run_blocks(const OpView& v, const LaunchPlan& plan, const DeviceState& dev,
                          cudaStream_t stream) {
  t_last_config = plan.config;
  const size_t n = plan.blocks.size();
  if (n <= 1) return launch_cfg<1>(plan.config, v, plan, dev, stream);
  if (n <= static_cast<size_t>(kFewProblems))
    return launch_cfg<kFewProblems>(plan.config, v, plan, dev, stream);
  return launch_cfg<kMaxProblems>(plan.config, v, plan, dev, stream);
}

// Operand bytes a CTA loads from L2 per multiply-add: its A rows and its
// share of B's columns per stage, over the stage's multiply-adds.
double operand_bytes_per_mac(const KernelConfig& c) {
  const double rows = c.pair ? c.bm / 2 : c.bm;
  const double cols = c.pair ? c.bn / 2 : c.bn;
  return 2.0 * (rows + cols) / (rows * c.bn);
}
// Products of at least this many FLOP run long enough (about 0.1 ms and
// more) for the power cap to set the clock; within kPowerTie of the fastest
// timed candidate, the tuner prefers the one that moves fewer operand bytes.
constexpr double kPowerBoundFlops = 2e11;
constexpr double kPowerTie = 0.02;

// Work units (tile slots) a configuration needs, counted in waves of the
// units the GPU runs at once; the rounding up is the wave-quantisation loss.
double config_cost(const std::vector<Block>& blocks, const KernelConfig& c, const DeviceState& dev) {
  int64_t tiles = 0;
  for (const Block& b : blocks)  // chain members after the head share its tiles
    if (b.chain > 0 && b.M > 0 && b.N > 0) tiles += ((b.M + c.bm - 1) / c.bm) * ((b.N + c.bn - 1) / c.bn);
  const int64_t slots = c.pair ? dev.max_pairs : dev.sms;
  const int64_t waves = (tiles + slots - 1) / slots;
  // One wave costs the tile's area over the configuration's speed.
  return static_cast<double>(waves) * c.bm * c.bn / kConfigSpeed[&c - kConfigs];
}

int choose_config(const std::vector<Block>& blocks, const DeviceState& dev) {
  const int forced = g_forced_config.load();
  if (forced >= 0 && forced < kNumConfigs) return forced;
  int best = 1;
  double best_cost = 0;
  for (int i = 0; i < kNumConfigs; ++i) {
    const double c = config_cost(blocks, kConfigs[i], dev);
    if (i == 0 || c < best_cost) {
      best = i;
      best_cost = c;
    }
  }
  return best;
}

// Products that leave most SMs idle: fewer 128x256 tiles than two waves.
// The split of the reduction range is offered to those with a reduction of
// at least 512 as well.  Slices are whole 64-deep stages.
bool underfilled(int64_t M, int64_t N, const DeviceState& dev) {
  const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
  return tiles < 2 * dev.sms;
}

bool split_eligible(int64_t M, int64_t N, int64_t R, const DeviceState& dev) {
  return underfilled(M, N, dev) && R >= 4 * kSplitMinR;
}

// The split actually run for a request of `want` pieces over nk reduction
// steps: a power of two (the tile's 128 rows are dealt out in equal bands),
// at most kMaxSplit and at most nk (no empty piece), or 1 for none.
int split_pieces(int want, int64_t nk) {
  int sp = 1;
  while (sp * 2 <= want && sp * 2 <= kMaxSplit && sp * 2 <= nk) sp *= 2;
  return sp;
}

// Default split (no tuning entry): only for reductions of at least
// kSplitMinSteps 64-deep stages, where the pieces' shorter mainloops repay
// the exchange of fp32 partials inside the cluster (measured on GB300: the
// 256x512x2048 data gradient, 32 stages over 8 tiles, gains 16 % split in
// 8; products of 8 to 16 stages lose).  Then the largest power of two up to
// kMaxSplit that keeps at least 4 stages a piece and one CTA per SM.
constexpr int64_t kSplitMinSteps = 32;
int choose_split(int64_t M, int64_t N, int64_t R, const DeviceState& dev) {
  const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
  const int64_t nk = (R + 63) / 64;
  if (nk < kSplitMinSteps) return 1;
  int split = 1;
  while (split < kMaxSplit && tiles * split * 2 <= dev.sms && nk / (split * 2) >= 4) split *= 2;
  return split;
}

std::string tune_key(int op, const axonn_fc_shape_t& s, uint32_t flags, int sms) {
  char buf[256];
  snprintf(buf, sizeof(buf), "op%d_T%lld_K%lld_N%lld_g%dx%dx%d_at%d.%d.%d_f%x_sm%d", op,
           (long long)s.T, (long long)s.K, (long long)s.N, s.gx, s.gy, s.gz, s.x, s.y, s.z, flags,
           sms);
  return buf;
}

// Shared body of the three entry points.  P and Q are the op's first and
// second stored operands, C its output.  `force` (tuning) fixes the choice.
axonn_status_t fc_op(int op, const void* P, const void* Q, void* C, int64_t ldp, int64_t ldq,
                     int64_t ldc, const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                     size_t ws_bytes, cudaStream_t stream, const TuneChoice* force = nullptr) {
  axonn_status_t st = check_shape(op, shape, flags);
  if (st != AXONN_OK) return st;
  if (flags & AXONN_ZSHARDED)
    return fail(AXONN_ERR_INVALID_ARG, "AXONN_ZSHARDED is for axonn_fc_workspace_size only");
  const axonn_fc_shape_t& s = *shape;
  const bool vgrid = (flags & AXONN_VGRID) != 0;
  const bool single = s.gx * s.gy * s.gz == 1;
  const bool full_ops = vgrid || single || (flags & AXONN_FULL_OPERANDS);
  const bool a_t = (flags & AXONN_A_T) != 0, b_t = (flags & AXONN_B_T) != 0;
  const bool out_f32 = (flags & (AXONN_ACCUM_F32 | AXONN_OUT_F32)) != 0;
  const int user_mode = (flags & AXONN_ACCUM_F32) ? axonn::kOutF32Accum
                        : (flags & AXONN_OUT_F32) ? axonn::kOutF32
                                                  : axonn::kOutBF16;

  // Logical extents the caller's buffers hold.
  int64_t M, N, R;
  full_dims(op, s, &M, &N, &R);
  Range rows{0, M}, red{0, R}, cols{0, N};
  if (!vgrid && !single) block_ranges(op, s, s.x, s.y, s.z, &rows, &red, &cols);
  const int64_t hM = full_ops ? M : rows.len();
  const int64_t hR = full_ops ? R : red.len();
  const int64_t hN = full_ops ? N : cols.len();

  // Map the op onto C = A . B with operand major-ness (see OpView).
  OpView v;
  v.A = static_cast<const char*>(P);
  v.lda = ldp;
  v.B = static_cast<const char*>(Q);
  v.ldb = ldq;
  v.C = static_cast<char*>(C);
  v.ldc = ldc;
  v.M = hM; v.N = hN; v.R = hR;
  if (op == AXONN_OP_FWD) {         // A = X, B = W
    v.a_mn = a_t;                   // X stored [K x T]
    v.b_mn = !b_t;                  // W stored [K x N] is N-contiguous
  } else if (op == AXONN_OP_DGRAD) {  // A = dY, B = W^T
    v.a_mn = a_t;                   // dY stored [N x T]
    v.b_mn = b_t;                   // W^T(n, k): W stored [N x K] is K(=cols)-contiguous
  } else {                          // A = X^T, B = dY
    v.a_mn = !a_t;                  // X stored [T x K] is K(=rows)-contiguous
    v.b_mn = !b_t;                  // dY stored [T x N] is N-contiguous
  }

  // Validate the stored operands as the caller laid them out.
  const char* pn = op == AXONN_OP_DGRAD ? "dY" : "X";
  const char* qn = op == AXONN_OP_WGRAD ? "dY" : "W";
  st = v.a_mn ? check_operand(pn, P, ldp, hR, hM) : check_operand(pn, P, ldp, hM, hR);
  if (st != AXONN_OK) return st;
  st = v.b_mn ? check_operand(qn, Q, ldq, hR, hN) : check_operand(qn, Q, ldq, hN, hR);
  if (st != AXONN_OK) return st;
  if (hM > 0 && hN > 0) {
    if (!C) return fail(AXONN_ERR_INVALID_ARG, "output is NULL");
    if (ldc < hN) return fail(AXONN_ERR_INVALID_ARG, "output leading dimension %lld < %lld", (long long)ldc,
                              (long long)hN);
    if (!aligned16(C)) return fail(AXONN_ERR_ALIGNMENT, "output is not 16-byte aligned");
    if (ldc % (out_f32 ? 4 : 8) != 0)
      return fail(AXONN_ERR_ALIGNMENT, "output leading dimension %lld misaligned", (long long)ldc);
  }
  if (hM == 0 || hN == 0) return ok();

  // The virtual grid's sum over the reduced axis, three ways:
  //  - chained (default): the G block products of each output tile run one
  //    after another into one TMEM accumulator (fixed order g = 0..G-1),
  //    one launch, no workspace;
  //  - AXONN_VGRID_PARTIALS: blocks 0..G-2 write fp32 partials to the
  //    workspace and the last block's epilogue adds them in order;
  //  - AXONN_REDUCE_ADD: every block adds its product into the fp32 output
  //    with reduction adds, in one launch, in no fixed order.
  const bool red_add = (flags & AXONN_REDUCE_ADD) != 0;
  const int G = reduce_extent(op, s);
  const bool partials = vgrid && G > 1 && (flags & AXONN_VGRID_PARTIALS);
  const bool chained = vgrid && G > 1 && !partials && !red_add;
  int64_t ldpart = 0;
  if (partials) {
    const size_t need = vgrid_ws_bytes(op, s, flags);
    if (!ws || ws_bytes < need)
      return fail(AXONN_ERR_WORKSPACE, "virtual grid needs %zu workspace bytes, got %zu", need, ws_bytes);
    if (!aligned16(ws)) return fail(AXONN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
    ldpart = (N + 7) / 8 * 8;
  }

  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != AXONN_OK) return st;

  auto a_at = [&](int64_t i, int64_t r) {
    return v.A + 2 * (v.a_mn ? r * v.lda + i : i * v.lda + r);
  };
  auto b_at = [&](int64_t r, int64_t j) {
    return v.B + 2 * (v.b_mn ? r * v.ldb + j : j * v.ldb + r);
  };
  const size_t celt = out_f32 ? 4 : 2;

  LaunchPlan plan;
  if (chained) {
    // Output blocks (o1, o2) in turn, each followed by its G block products
    // in order along the reduced axis.
    const int n1 = op == AXONN_OP_WGRAD ? s.gx : s.gz;
    const int n2 = op == AXONN_OP_DGRAD ? s.gx : s.gy;
    for (int o1 = 0; o1 < n1; ++o1)
      for (int o2 = 0; o2 < n2; ++o2)
        for (int g = 0; g < G; ++g) {
          const int x = op == AXONN_OP_FWD ? g : (op == AXONN_OP_DGRAD ? o2 : o1);
          const int y = op == AXONN_OP_DGRAD ? g : o2;
          const int z = op == AXONN_OP_WGRAD ? g : o1;
          Range br, bred, bc;
          block_ranges(op, s, x, y, z, &br, &bred, &bc);
          Block b;
          b.A = a_at(br.s, bred.s);
          b.B = b_at(bred.s, bc.s);
          b.M = br.len(); b.N = bc.len(); b.R = bred.len();
          b.C = v.C + celt * (br.s * ldc + bc.s);
          b.ldc = ldc;
          b.out_mode = user_mode;
          b.chain = g == 0 ? G : 0;
          plan.blocks.push_back(b);
        }
  } else if (vgrid) {
    for (int x = 0; x < s.gx; ++x)
      for (int y = 0; y < s.gy; ++y)
        for (int z = 0; z < s.gz; ++z) {
          Range br, bred, bc;
          block_ranges(op, s, x, y, z, &br, &bred, &bc);
          Block b;
          b.A = a_at(br.s, bred.s);
          b.B = b_at(bred.s, bc.s);
          b.M = br.len(); b.N = bc.len(); b.R = bred.len();
          const int g = reduce_coord(op, x, y, z);
          if (partials && g < G - 1) {
            // partial g of the reduced axis, fp32, at its place in slot g
            b.C = static_cast<char*>(ws) + 4 * (static_cast<int64_t>(g) * M * ldpart + br.s * ldpart + bc.s);
            b.ldc = ldpart;
            b.out_mode = axonn::kOutF32;
            b.phase = 0;
          } else if (partials) {
            // the last partial sums slots 0..G-2 and itself into the output
            b.C = v.C + celt * (br.s * ldc + bc.s);
            b.ldc = ldc;
            b.out_mode = user_mode;
            b.red_count = G - 1;
            b.red_src = reinterpret_cast<const float*>(ws) + (br.s * ldpart + bc.s);
            b.red_stride = M * ldpart;
            b.red_ld = ldpart;
          } else {
            b.C = v.C + celt * (br.s * ldc + bc.s);
            b.ldc = ldc;
            b.out_mode = red_add ? axonn::kOutF32Red : user_mode;
          }
          plan.blocks.push_back(b);
        }
  } else {
    Block b;
    const bool offs = full_ops && !single;
    b.A = offs ? a_at(rows.s, red.s) : v.A;
    b.B = offs ? b_at(red.s, cols.s) : v.B;
    b.C = offs ? v.C + celt * (rows.s * ldc + cols.s) : v.C;
    b.ldc = ldc;
    b.M = rows.len(); b.N = cols.len(); b.R = red.len();
    b.out_mode = user_mode;
    plan.blocks.push_back(b);
  }

  // How to run it: forced (tuning), tuned earlier, or the default choice.
  TuneChoice ch;
  if (force) {
    ch = *force;
  } else {
    bool found = false;
    {
      std::lock_guard<std::mutex> lk(g_tune_mu);
      auto it = g_tune.find(tune_key(op, s, flags, dev->sms));
      if (it != g_tune.end()) {
        ch = it->second.choice;
        found = true;
      }
    }
    if (!found) {
      const Block& b0 = plan.blocks[0];
      ch.split = (!vgrid && split_eligible(b0.M, b0.N, b0.R, *dev))
                     ? choose_split(b0.M, b0.N, b0.R, *dev) : 1;
      ch.config = ch.split > 1 ? 0 : choose_config(plan.blocks, *dev);
      ch.group_m = 16;
    }
    const int forced_cfg = g_forced_config.load();
    if (forced_cfg >= 0) ch.config = forced_cfg;
  }
  const int forced_sw = g_forced_swap.load();
  if (forced_sw >= 0) ch.swap = forced_sw;
  const int forced_sk = g_forced_streamk.load();
  if (forced_sk >= 0) ch.streamk = forced_sk == 0 ? kStreamKOff : kStreamKAlways;
  if (ch.config < 0 || ch.config >= kNumConfigs) ch.config = choose_config(plan.blocks, *dev);
  if (ch.group_m == 0) ch.group_m = 16;

  // Split of the reduction range into S pieces of whole stages, computed
  // by the S CTAs of a cluster and summed in order inside it (the kernel's
  // kSplit form): one launch, no workspace.  Single products only.
  if (ch.split > 1) {
    const Block& b0 = plan.blocks[0];
    const bool able = !vgrid && plan.blocks.size() == 1 && split_config(ch.config);
    ch.split = able ? split_pieces(ch.split, (b0.R + 63) / 64) : 1;
    if (ch.split > 1 && dev->split_clusters[split_index(ch.config)][split_lg(ch.split)] <= 0)
      ch.split = 1;
  }
  // Exchanged operand roles: C^T[N x M] = B^T . A^T, the same operands read
  // through each other's tensor-map role, written back transposed by the
  // epilogue.  Not with the two-launch grid sum, whose fp32 partials are
  // laid out in the caller's orientation.
  OpView lv = v;
  if (ch.swap && partials) ch.swap = 0;
  if (ch.swap) {
    lv.A = v.B; lv.lda = v.ldb; lv.a_mn = v.b_mn;
    lv.B = v.A; lv.ldb = v.lda; lv.b_mn = v.a_mn;
    lv.M = v.N; lv.N = v.M;
    for (Block& b : plan.blocks) {
      std::swap(b.A, b.B);
      std::swap(b.M, b.N);
      b.out_t = true;
    }
  }
  plan.config = ch.config;
  plan.group_m = ch.group_m;
  plan.split = ch.split;
  if (!vgrid) {
    if (ch.split == 1) plan.streamk = ch.streamk;
    plan.ws = ws;
    plan.ws_bytes = ws_bytes;
  }
  t_last_choice = ch;
  // Products whose epilogue sums earlier partials run in a second launch,
  // after every partial they read has been written by the first.
  LaunchPlan first = plan, last = plan;
  first.blocks.clear();
  last.blocks.clear();
  for (const Block& b : plan.blocks) (b.phase == 0 ? first : last).blocks.push_back(b);
  if (!first.blocks.empty()) {
    st = run_blocks(lv, first, *dev, stream);
    if (st != AXONN_OK) return st;
  }
  if (!last.blocks.empty()) {
    st = run_blocks(lv, last, *dev, stream);
    if (st != AXONN_OK) return st;
  }

  return ok();
}

// ----------------------------------------------------------------------
// Z-sharded weights.  Inside the 3D grid the weight block W_{x,y} (and its
// gradient) is kept as G_z row shards, shard z on rank (x, y, z): an
// all-gather over the Z group rebuilds the block before it is used and a
// reduce-scatter over the Z group turns the G_z weight-gradient partials into
// the shards of their sum.  Row shards follow the grid's split rule (units of
// 8 rows, leading shards take the extra unit).
// ----------------------------------------------------------------------
__global__ void __launch_bounds__(256) copy_rows_kernel(const char* __restrict__ src,
                                                        int64_t src_ld, char* __restrict__ dst,
                                                        int64_t dst_ld, int64_t rows,
                                                        int64_t chunks_per_row) {
  const int64_t total = rows * chunks_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks_per_row, c = i - r * chunks_per_row;
    *reinterpret_cast<uint4*>(dst + r * dst_ld + 16 * c) =
        *reinterpret_cast<const uint4*>(src + r * src_ld + 16 * c);
  }
}

size_t zsharded_ws_bytes(const axonn_fc_shape_t& s) {
  if (s.gz <= 1) return 0;
  Range Kx, Ny;
  split_range(s.K, s.gx, s.x, &Kx.s, &Kx.e);
  split_range(s.N, s.gy, s.y, &Ny.s, &Ny.e);
  return static_cast<size_t>(s.gz - 1) * static_cast<size_t>(Kx.len()) *
         static_cast<size_t>((Ny.len() + 7) / 8 * 8) * 4u;
}

// ----------------------------------------------------------------------
// Fixed scratch for callers that cannot allocate device memory.
//
// The virtual-grid path needs an fp32 buffer for the partial products of
// the reduced grid axis.  Normally the caller passes it as a workspace.  A
// caller that may not call cudaMalloc -- code running where device memory is
// handed out by someone else, or under a policy that forbids allocation
// after start-up -- can use axonn_fc_vgrid_static instead, which takes its
// scratch from this array.  The array is part of the library image: every
// GPU that loads the library holds these bytes until the process exits.
// ----------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t{64} << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
std::vector<void*> g_static_addr;  // per device; set on the first call there

// Device address of g_static_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked
// for once per device (with that device current) and cached.
axonn_status_t static_scratch_addr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (static_cast<int>(g_static_addr.size()) <= dev) g_static_addr.resize(dev + 1, nullptr);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(AXONN_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return AXONN_OK;
}

}  // namespace

extern "C" {

axonn_status_t axonn_fc_vgrid_static(int op, const void* P, const void* Q, void* C, int64_t ldp,
                                     int64_t ldq, int64_t ldc, const axonn_fc_shape_t* shape,
                                     uint32_t flags, cudaStream_t stream) {
  const uint32_t f = flags | AXONN_VGRID;
  axonn_status_t st = check_shape(op, shape, f);
  if (st != AXONN_OK) return st;
  const size_t need = vgrid_ws_bytes(op, *shape, f);
  if (need > kStaticScratchBytes)
    return fail(AXONN_ERR_WORKSPACE,
                "this product needs %zu bytes of partial-sum scratch; the built-in scratch holds %zu "
                "(use the entry point with a caller workspace)",
                need, kStaticScratchBytes);
  void* ws = nullptr;
  if (need > 0) {
    st = static_scratch_addr(&ws);
    if (st != AXONN_OK) return st;
  }
  return fc_op(op, P, Q, C, ldp, ldq, ldc, shape, f, ws, need > 0 ? kStaticScratchBytes : 0, stream);
}

axonn_status_t axonn_fc_fwd(const void* X, const void* W, void* Y, int64_t ldx, int64_t ldw, int64_t ldy,
                            const axonn_fc_shape_t* shape, uint32_t flags, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  return fc_op(AXONN_OP_FWD, X, W, Y, ldx, ldw, ldy, shape, flags, ws, ws_bytes, stream);
}

axonn_status_t axonn_fc_dgrad(const void* dY, const void* W, void* dX, int64_t lddy, int64_t ldw,
                              int64_t lddx, const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  return fc_op(AXONN_OP_DGRAD, dY, W, dX, lddy, ldw, lddx, shape, flags, ws, ws_bytes, stream);
}

axonn_status_t axonn_fc_wgrad(const void* X, const void* dY, void* dW, int64_t ldx, int64_t lddy,
                              int64_t lddw, const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  return fc_op(AXONN_OP_WGRAD, X, dY, dW, ldx, lddy, lddw, shape, flags, ws, ws_bytes, stream);
}

axonn_status_t axonn_shards_gather(const void* const* shards, int32_t g, int64_t rows, int64_t cols,
                                   int64_t ld_shard, void* out, int64_t ld_out, cudaStream_t stream) {
  if (g < 1 || g > kMaxProblems) return fail(AXONN_ERR_INVALID_ARG, "shard count %d not in [1, %d]", g, kMaxProblems);
  if (rows < 0 || cols < 0) return fail(AXONN_ERR_INVALID_ARG, "negative extent");
  if (rows == 0 || cols == 0) return ok();
  if (!shards || !out) return fail(AXONN_ERR_INVALID_ARG, "NULL shard table or output");
  if (cols % 8 != 0) return fail(AXONN_ERR_ALIGNMENT, "row length %lld is not a multiple of 8", (long long)cols);
  if (ld_shard < cols || ld_out < cols) return fail(AXONN_ERR_INVALID_ARG, "leading dimension below row length");
  if (ld_shard % 8 != 0 || ld_out % 8 != 0 || !aligned16(out))
    return fail(AXONN_ERR_ALIGNMENT, "leading dimensions must be multiples of 8, pointers 16-byte aligned");
  for (int z = 0; z < g; ++z) {
    int64_t s0, s1;
    split_range(rows, g, z, &s0, &s1);
    if (s1 > s0 && (!shards[z] || !aligned16(shards[z])))
      return fail(AXONN_ERR_ALIGNMENT, "shard %d is NULL or not 16-byte aligned", z);
  }
  DeviceState* dev = nullptr;
  axonn_status_t st = device_state(&dev);
  if (st != AXONN_OK) return st;
  const int64_t chunks = cols * 2 / 16;
  for (int z = 0; z < g; ++z) {
    int64_t s0, s1;
    split_range(rows, g, z, &s0, &s1);
    if (s1 <= s0) continue;
    const int64_t total = (s1 - s0) * chunks;
    int64_t blocks = (total + 255) / 256;
    if (blocks > static_cast<int64_t>(dev->sms) * 16) blocks = static_cast<int64_t>(dev->sms) * 16;
    copy_rows_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const char*>(shards[z]), ld_shard * 2, static_cast<char*>(out) + s0 * ld_out * 2,
        ld_out * 2, s1 - s0, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "gather launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

axonn_status_t axonn_fc_wgrad_zsharded(const void* X, const void* dY, void* const* dW_shards,
                                       int64_t ldx, int64_t lddy, int64_t ld_shard,
                                       const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                                       size_t ws_bytes, cudaStream_t stream) {
  if (!shape) return fail(AXONN_ERR_INVALID_ARG, "shape is NULL");
  if (flags & (AXONN_VGRID | AXONN_FULL_OPERANDS | AXONN_ZSHARDED))
    return fail(AXONN_ERR_INVALID_ARG, "grid-mode flags are implied by this entry point");
  axonn_fc_shape_t s = *shape;
  s.z = 0;
  axonn_status_t st = check_shape(AXONN_OP_WGRAD, &s, flags);
  if (st != AXONN_OK) return st;
  const bool out_f32 = (flags & (AXONN_ACCUM_F32 | AXONN_OUT_F32)) != 0;
  const int user_mode = (flags & AXONN_ACCUM_F32) ? axonn::kOutF32Accum
                        : (flags & AXONN_OUT_F32) ? axonn::kOutF32
                                                  : axonn::kOutBF16;
  // Full operands: X [T x K], dY [T x N] (transposed storage by flags).
  OpView v;
  v.A = static_cast<const char*>(X);
  v.lda = ldx;
  v.B = static_cast<const char*>(dY);
  v.ldb = lddy;
  v.C = nullptr;
  v.ldc = ld_shard;
  v.M = s.K; v.N = s.N; v.R = s.T;
  v.a_mn = !(flags & AXONN_A_T);
  v.b_mn = !(flags & AXONN_B_T);
  st = v.a_mn ? check_operand("X", X, ldx, s.T, s.K) : check_operand("X", X, ldx, s.K, s.T);
  if (st != AXONN_OK) return st;
  st = v.b_mn ? check_operand("dY", dY, lddy, s.T, s.N) : check_operand("dY", dY, lddy, s.N, s.T);
  if (st != AXONN_OK) return st;
  Range Kx, Ny;
  split_range(s.K, s.gx, s.x, &Kx.s, &Kx.e);
  split_range(s.N, s.gy, s.y, &Ny.s, &Ny.e);
  const int64_t Mb = Kx.len(), Nb = Ny.len();
  if (Mb == 0 || Nb == 0) return ok();
  if (!dW_shards) return fail(AXONN_ERR_INVALID_ARG, "shard table is NULL");
  if (ld_shard < Nb) return fail(AXONN_ERR_INVALID_ARG, "shard leading dimension %lld < %lld",
                                 (long long)ld_shard, (long long)Nb);
  if (ld_shard % (out_f32 ? 4 : 8) != 0) return fail(AXONN_ERR_ALIGNMENT, "shard leading dimension misaligned");
  for (int z = 0; z < s.gz; ++z) {
    int64_t r0, r1;
    split_range(Mb, s.gz, z, &r0, &r1);
    if (r1 > r0 && (!dW_shards[z] || !aligned16(dW_shards[z])))
      return fail(AXONN_ERR_ALIGNMENT, "shard %d is NULL or not 16-byte aligned", z);
  }
  const size_t need = zsharded_ws_bytes(s);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(AXONN_ERR_WORKSPACE, "Z-sharded weight gradient needs %zu workspace bytes, got %zu", need,
                ws_bytes);
  if (need > 0 && !aligned16(ws)) return fail(AXONN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != AXONN_OK) return st;

  auto a_at = [&](int64_t i, int64_t r) { return v.A + 2 * (v.a_mn ? r * v.lda + i : i * v.lda + r); };
  auto b_at = [&](int64_t r, int64_t j) { return v.B + 2 * (v.b_mn ? r * v.ldb + j : j * v.ldb + r); };
  const int64_t ldp = (Nb + 7) / 8 * 8;
  float* part = static_cast<float*>(ws);
  LaunchPlan first, last;
  for (int z = 0; z < s.gz; ++z) {
    Range Tz;
    split_range(s.T, s.gz, z, &Tz.s, &Tz.e);
    if (z < s.gz - 1) {  // partial z of the Z group, fp32, into workspace slot z
      Block b;
      b.A = a_at(Kx.s, Tz.s);
      b.B = b_at(Tz.s, Ny.s);
      b.C = reinterpret_cast<char*>(part + static_cast<int64_t>(z) * Mb * ldp);
      b.ldc = ldp;
      b.M = Mb; b.N = Nb; b.R = Tz.len();
      b.out_mode = axonn::kOutF32;
      b.phase = 0;
      first.blocks.push_back(b);
    } else {  // the last partial, cut at the shard rows, sums the others into each shard
      for (int zz = 0; zz < s.gz; ++zz) {
        int64_t r0, r1;
        split_range(Mb, s.gz, zz, &r0, &r1);
        if (r1 <= r0) continue;
        Block b;
        b.A = a_at(Kx.s + r0, Tz.s);
        b.B = b_at(Tz.s, Ny.s);
        b.C = static_cast<char*>(dW_shards[zz]);
        b.ldc = ld_shard;
        b.M = r1 - r0; b.N = Nb; b.R = Tz.len();
        b.out_mode = user_mode;
        if (s.gz > 1) {
          b.red_count = s.gz - 1;
          b.red_src = part + r0 * ldp;
          b.red_stride = Mb * ldp;
          b.red_ld = ldp;
        }
        last.blocks.push_back(b);
      }
    }
  }
  std::vector<Block> all = first.blocks;
  all.insert(all.end(), last.blocks.begin(), last.blocks.end());
  const int forced = g_forced_config.load();
  first.config = last.config = (forced >= 0) ? forced : choose_config(all, *dev);
  t_last_choice = TuneChoice{first.config, 1, first.group_m};
  if (!first.blocks.empty()) {
    st = run_blocks(v, first, *dev, stream);
    if (st != AXONN_OK) return st;
  }
  st = run_blocks(v, last, *dev, stream);
  if (st != AXONN_OK) return st;
  return ok();
}

axonn_status_t axonn_fc_tune(int op, const void* P, const void* Q, void* C, int64_t ldp, int64_t ldq,
                             int64_t ldc, const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                             size_t ws_bytes, cudaStream_t stream, int* best_config, int* best_split,
                             int* best_group_m, float* best_us) {
  axonn_status_t st = check_shape(op, shape, flags);
  if (st != AXONN_OK) return st;
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != AXONN_OK) return st;
  const axonn_fc_shape_t& s = *shape;
  // Tuning runs the product many times: an accumulating call is timed as an
  // overwriting one (the caller's output is overwritten either way), except
  // with AXONN_REDUCE_ADD, whose atomic epilogue only adds: those runs add
  // into the output again and again.
  const uint32_t run_flags =
      (flags & AXONN_ACCUM_F32) && !(flags & AXONN_REDUCE_ADD)
          ? ((flags & ~AXONN_ACCUM_F32) | AXONN_OUT_F32) : flags;
  int64_t M, N, R;
  full_dims(op, s, &M, &N, &R);
  Range rows{0, M}, red{0, R}, cols{0, N};
  if (s.gx * s.gy * s.gz > 1 && !(flags & AXONN_VGRID))
    block_ranges(op, s, s.x, s.y, s.z, &rows, &red, &cols);

  // Candidates.  Products that fill the GPU many times over only try the
  // configurations that ever win there (128x256, 256-row and 512-row tiles);
  // under-filled products try everything, reduction splits included.
  // Products that leave SMs idle (fewer 128x256 tiles than two waves) try
  // every configuration; those with a long enough reduction also try the
  // reduction split.
  const bool small = underfilled(rows.len(), cols.len(), *dev);
  const bool splittable = split_eligible(rows.len(), cols.len(), red.len(), *dev);
  std::vector<TuneChoice> cands;
  for (int c = 0; c < kNumConfigs; ++c) {
    if (!small && !(c == 1 || c == 3 || c == 5 || c == 6)) continue;
    for (int gm : {8, 16, -8, -16}) cands.push_back(TuneChoice{c, 1, gm});
  }
  if (!(flags & AXONN_VGRID) && splittable)
    for (int sp = 2; sp <= kMaxSplit; sp *= 2)
      if (red.len() / sp >= kSplitMinR)
        for (int c : {0, 7})
          for (int gm : {16, -16}) cands.push_back(TuneChoice{c, sp, gm});

  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    return fail(AXONN_ERR_CUDA, "cudaEventCreate failed");
  }
  // Two rounds over all candidates, each candidate timed over kReps runs
  // per round; a candidate's time is its best round, so slow drifts of the
  // clock (power capping) do not favour the candidates measured first.
  // Each candidate's kReps runs are captured into a CUDA graph and the graph
  // is timed, so small products are measured on the device timeline rather
  // than through host launch overhead.  Streams that cannot be captured
  // (the legacy default stream) are timed with eager launches instead.
  constexpr int kRounds = 2;
  // Calls per timed graph: 3, or 20 for products of a few microseconds,
  // whose differences between candidates would otherwise be within the
  // jitter of one graph launch.
  const double flops = 2.0 * static_cast<double>(rows.len()) * static_cast<double>(cols.len()) *
                       static_cast<double>(red.len());
  const int kReps = flops < 2e10 ? 20 : 3;
  std::vector<double> cand_us(cands.size(), -1.0);
  auto time_candidate = [&](const TuneChoice& c, double* us) -> bool {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    bool ok_run = true;
    if (cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
      for (int r = 0; r < kReps && ok_run; ++r)
        ok_run = fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &c) == AXONN_OK;
      const cudaError_t ec = cudaStreamEndCapture(stream, &graph);
      if (ec != cudaSuccess || !ok_run || !graph ||
          cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        (void)cudaGetLastError();
        return false;
      }
      bool good = cudaGraphLaunch(exec, stream) == cudaSuccess;  // warm
      good = good && cudaEventRecord(e0, stream) == cudaSuccess;
      good = good && cudaGraphLaunch(exec, stream) == cudaSuccess;
      good = good && cudaEventRecord(e1, stream) == cudaSuccess;
      good = good && cudaEventSynchronize(e1) == cudaSuccess;
      cudaGraphExecDestroy(exec);
      cudaGraphDestroy(graph);
      if (!good) return false;
    } else {
      (void)cudaGetLastError();
      cudaEventRecord(e0, stream);
      for (int r = 0; r < kReps && ok_run; ++r)
        ok_run = fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &c) == AXONN_OK;
      cudaEventRecord(e1, stream);
      if (cudaEventSynchronize(e1) != cudaSuccess || !ok_run) return false;
    }
    float ms = 0;
    cudaEventElapsedTime(&ms, e0, e1);
    *us = 1e3 * ms / kReps;
    return true;
  };
  // Under a power cap the SM clock drifts while candidates run, so every
  // candidate is timed between two runs of a reference (the default choice)
  // and scored by its time over theirs; a candidate's score is its best
  // round.
  TuneChoice ref;
  {
    std::vector<Block> probe(1);
    probe[0].M = rows.len(); probe[0].N = cols.len(); probe[0].R = red.len();
    ref.config = choose_config(probe, *dev);
  }
  std::vector<double> cand_ratio(cands.size(), -1.0);
  double ref_us = 0;
  bool ref_ok = fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &ref) == AXONN_OK &&
                time_candidate(ref, &ref_us);
  for (int round = 0; round < kRounds && ref_ok; ++round) {
    for (size_t i = 0; i < cands.size(); ++i) {
      const TuneChoice& c = cands[i];
      if (round > 0 && cand_us[i] < 0) continue;  // failed in the first round
      if (fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &c) != AXONN_OK)
        continue;
      if (t_last_choice.split != c.split) continue;  // the split could not be applied
      double us = 0, ref_next = 0;
      if (!time_candidate(c, &us)) continue;
      if (!time_candidate(ref, &ref_next)) ref_next = ref_us;
      const double ratio = us / (0.5 * (ref_us + ref_next));
      ref_us = ref_next;
      if (cand_ratio[i] < 0 || ratio < cand_ratio[i]) {
        cand_ratio[i] = ratio;
        cand_us[i] = us;
      }
    }
  }
  TuneEntry best;
  best.us = -1;
  double best_ratio = 0;
  for (size_t i = 0; i < cands.size(); ++i)
    if (cand_ratio[i] >= 0 && (best.us < 0 || cand_ratio[i] < best_ratio)) {
      best_ratio = cand_ratio[i];
      best.us = cand_us[i];
      best.choice = cands[i];
    }
  // Products long enough for the power cap to set the clock: a candidate
  // within kPowerTie of the fastest that moves fewer operand bytes from L2
  // per multiply-add is taken instead.  The timing runs above are too short
  // for the cap to act, and L2-to-SM traffic costs clock in a long step
  // (measured: loading every A tile twice cost 3 % of SM clock).
  if (best.us >= 0 && flops >= kPowerBoundFlops) {
    const double limit = best_ratio * (1.0 + kPowerTie);
    size_t pick = cands.size();
    double pick_bytes = operand_bytes_per_mac(kConfigs[best.choice.config]);
    for (size_t i = 0; i < cands.size(); ++i) {
      if (cand_ratio[i] < 0 || cand_ratio[i] > limit) continue;
      const double b = operand_bytes_per_mac(kConfigs[cands[i].config]);
      if (b < pick_bytes * 0.99 ||
          (pick < cands.size() && b <= pick_bytes * 1.01 && cand_ratio[i] < cand_ratio[pick])) {
        pick = i;
        pick_bytes = b;
      }
    }
    if (pick < cands.size()) {
      best_ratio = cand_ratio[pick];
      best.us = cand_us[pick];
      best.choice = cands[pick];
    }
  }
  // Exchanged operand roles (C^T = B^T . A^T): the two best candidates are
  // timed again with the roles swapped, each between reference runs like
  // the others, and a swapped one is kept where it scores better.
  if (best.us >= 0 && g_forced_swap.load() < 0) {
    size_t order[2] = {cands.size(), cands.size()};
    for (size_t i = 0; i < cands.size(); ++i) {
      if (cand_ratio[i] < 0) continue;
      if (order[0] == cands.size() || cand_ratio[i] < cand_ratio[order[0]]) {
        order[1] = order[0];
        order[0] = i;
      } else if (order[1] == cands.size() || cand_ratio[i] < cand_ratio[order[1]]) {
        order[1] = i;
      }
    }
    for (size_t i : order) {
      if (i == cands.size()) continue;
      TuneChoice c = cands[i];
      c.swap = 1;
      if (fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &c) != AXONN_OK ||
          t_last_choice.swap != 1)
        continue;  // the swap does not apply to this call
      double us = 0, ref_next = 0;
      if (!time_candidate(c, &us)) continue;
      if (!time_candidate(ref, &ref_next)) ref_next = ref_us;
      const double ratio = us / (0.5 * (ref_us + ref_next));
      ref_us = ref_next;
      if (ratio < best_ratio) {
        best_ratio = ratio;
        best.us = us;
        best.choice = c;
      }
    }
  }
  // The candidates ran with the default stream-K mode.  Time the best one
  // in all three modes back to back (so they see the same clock) and keep
  // the fastest; the modes are the same launch where no tail applies.
  if (best.us >= 0 && g_forced_streamk.load() < 0) {
    double mode_us[3] = {-1, -1, -1};
    for (int m : {kStreamKOff, kStreamKShortTail, kStreamKAlways}) {
      TuneChoice c = best.choice;
      c.streamk = m;
      if (fc_op(op, P, Q, C, ldp, ldq, ldc, shape, run_flags, ws, ws_bytes, stream, &c) != AXONN_OK ||
          !time_candidate(c, &mode_us[m]))
        mode_us[m] = -1;
    }
    int pick = best.choice.streamk;
    for (int m : {kStreamKOff, kStreamKShortTail, kStreamKAlways})
      if (mode_us[m] >= 0 && (mode_us[pick] < 0 || mode_us[m] < mode_us[pick])) pick = m;
    if (mode_us[pick] >= 0) {
      best.choice.streamk = pick;
      best.us = mode_us[pick];
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (best.us < 0) return fail(AXONN_ERR_CUDA, "no candidate configuration ran");
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tune[tune_key(op, s, flags, dev->sms)] = best;
  }
  if (best_config) *best_config = best.choice.config;
  if (best_split) *best_split = best.choice.split;
  if (best_group_m) *best_group_m = best.choice.group_m;
  if (best_us) *best_us = static_cast<float>(best.us);
  return ok();
}

axonn_status_t axonn_tune_cache_save(const char* path) {
  if (!path) return fail(AXONN_ERR_INVALID_ARG, "path is NULL");
  std::ofstream f(path);
  if (!f) return fail(AXONN_ERR_INVALID_ARG, "cannot write %s", path);
  std::lock_guard<std::mutex> lk(g_tune_mu);
  for (const auto& kv : g_tune) {
    char line[512];
    snprintf(line, sizeof(line),
             "{\"key\": \"%s\", \"config\": \"%s\", \"split\": %d, \"group_m\": %d, "
             "\"streamk\": %d, \"swap\": %d, \"us\": %.3f}\n",
             kv.first.c_str(), kConfigs[kv.second.choice.config].name, kv.second.choice.split,
             kv.second.choice.group_m, kv.second.choice.streamk, kv.second.choice.swap,
             kv.second.us);
    f << line;
  }
  return f ? ok() : fail(AXONN_ERR_INVALID_ARG, "write to %s failed", path);
}

namespace {
// Value of "name" in one line written by axonn_tune_cache_save.
bool json_field(const std::string& line, const char* name, std::string* out) {
  const std::string tag = std::string("\"") + name + "\": ";
  const size_t p = line.find(tag);
  if (p == std::string::npos) return false;
  size_t b = p + tag.size(), e;
  if (b < line.size() && line[b] == '"') {
    e = line.find('"', b + 1);
    if (e == std::string::npos) return false;
    *out = line.substr(b + 1, e - b - 1);
  } else {
    e = line.find_first_of(",}", b);
    if (e == std::string::npos) return false;
    *out = line.substr(b, e - b);
  }
  return true;
}
}  // namespace

}  // extern "C"

namespace {
// A whole decimal integer in [lo, hi] (no trailing characters).
bool parse_int(const std::string& text, long lo, long hi, int* out) {
  if (text.empty()) return false;
  char* end = nullptr;
  errno = 0;
  const long v = strtol(text.c_str(), &end, 10);
  if (errno != 0 || end == text.c_str() || *end != '\0' || v < lo || v > hi) return false;
  *out = static_cast<int>(v);
  return true;
}
// Rasterisation groups the kernels take: at most 64 tile rows or columns
// (the tuner writes 8 and 16); larger values would overflow the tile walk.
constexpr long kMaxGroup = 64;
}  // namespace

extern "C" {

axonn_status_t axonn_tune_cache_load(const char* path) {
  if (!path) return fail(AXONN_ERR_INVALID_ARG, "path is NULL");
  std::ifstream f(path);
  if (!f) return fail(AXONN_ERR_INVALID_ARG, "cannot read %s", path);
  std::string line;
  std::unordered_map<std::string, TuneEntry> loaded;
  int lineno = 0;
  while (std::getline(f, line)) {
    ++lineno;
    if (line.find_first_not_of(" \t\r") == std::string::npos) continue;
    std::string key, cfg, split, gm, us;
    if (!json_field(line, "key", &key) || !json_field(line, "config", &cfg) ||
        !json_field(line, "split", &split) || !json_field(line, "group_m", &gm) ||
        !json_field(line, "us", &us))
      return fail(AXONN_ERR_INVALID_ARG, "%s:%d: malformed tuning entry", path, lineno);
    TuneEntry e;
    e.choice.config = -1;
    for (int c = 0; c < kNumConfigs; ++c)
      if (cfg == kConfigs[c].name) e.choice.config = c;
    std::string sk, sw;
    const bool has_sk = json_field(line, "streamk", &sk);
    const bool has_sw = json_field(line, "swap", &sw);
    if (e.choice.config < 0 || !parse_int(split, 1, kMaxSplit, &e.choice.split) ||
        !parse_int(gm, -kMaxGroup, kMaxGroup, &e.choice.group_m) || e.choice.group_m == 0 ||
        (has_sk && !parse_int(sk, kStreamKOff, kStreamKAlways, &e.choice.streamk)) ||
        (has_sw && !parse_int(sw, 0, 1, &e.choice.swap)))
      return fail(AXONN_ERR_INVALID_ARG, "%s:%d: unknown configuration", path, lineno);
    e.us = atof(us.c_str());
    loaded[key] = e;
  }
  std::lock_guard<std::mutex> lk(g_tune_mu);
  for (auto& kv : loaded) g_tune[kv.first] = kv.second;
  return ok();
}

void axonn_tune_cache_clear(void) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.clear();
}

int axonn_tune_cache_size(void) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return static_cast<int>(g_tune.size());
}

axonn_status_t axonn_tune_lookup(int op, const axonn_fc_shape_t* shape, uint32_t flags,
                                 int* found) {
  if (!found) return fail(AXONN_ERR_INVALID_ARG, "found is NULL");
  *found = 0;
  axonn_status_t st = check_shape(op, shape, flags);
  if (st != AXONN_OK) return st;
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != AXONN_OK) return st;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  *found = g_tune.count(tune_key(op, *shape, flags, dev->sms)) ? 1 : 0;
  return ok();
}

void axonn_last_choice(int* config, int* split, int* group_m) {
  if (config) *config = t_last_choice.config;
  if (split) *split = t_last_choice.split;
  if (group_m) *group_m = t_last_choice.group_m;
}

axonn_status_t axonn_fc_workspace_size(int op, const axonn_fc_shape_t* shape, uint32_t flags,
                                       size_t* bytes) {
  if (!bytes) return fail(AXONN_ERR_INVALID_ARG, "bytes is NULL");
  axonn_status_t st = check_shape(op, shape, flags);
  if (st != AXONN_OK) return st;
  if (flags & AXONN_ZSHARDED) {
    if (op != AXONN_OP_WGRAD) return fail(AXONN_ERR_INVALID_ARG, "AXONN_ZSHARDED applies to the weight gradient");
    *bytes = zsharded_ws_bytes(*shape);
    return ok();
  }
  *bytes = vgrid_ws_bytes(op, *shape, flags);
  if (!(flags & AXONN_VGRID)) {
    // The reduction split needs none; products of more than one wave of
    // tiles may run a stream-K tail.
    DeviceState* dev = nullptr;
    if (device_state(&dev) == AXONN_OK) {
      const axonn_fc_shape_t& s = *shape;
      int64_t M, N, R;
      full_dims(op, s, &M, &N, &R);
      Range rows{0, M}, red{0, R}, cols{0, N};
      if (s.gx * s.gy * s.gz > 1) block_ranges(op, s, s.x, s.y, s.z, &rows, &red, &cols);
      const int64_t tiles128 = ((rows.len() + 127) / 128) * ((cols.len() + 127) / 128);
      if (tiles128 > dev->sms)
        for (const KernelConfig& c : kConfigs)
          *bytes = std::max(*bytes, streamk_ws_bytes(c, c.pair ? dev->max_pairs : dev->sms));
    }
  }
  return ok();
}

axonn_status_t axonn_block_range(int64_t D, int32_t G, int32_t b, int64_t* start, int64_t* stop) {
  if (!start || !stop) return fail(AXONN_ERR_INVALID_ARG, "NULL output");
  if (D < 0 || G < 1 || b < 0 || b >= G) return fail(AXONN_ERR_INVALID_ARG, "bad D/G/b");
  split_range(D, G, b, start, stop);
  return ok();
}

axonn_status_t axonn_goldfish_ce(const void* logits, int64_t ld_logits, const int32_t* input_ids,
                                 const int32_t* labels, int64_t batch, int64_t seq, int64_t vocab,
                                 int32_t k, int32_t h, uint8_t* keep, float* token_loss,
                                 float* loss, int32_t* kept, void* dlogits, int64_t ld_dlogits,
                                 cudaStream_t stream) {
  if (batch < 0 || seq < 0) return fail(AXONN_ERR_INVALID_ARG, "negative batch or sequence length");
  if (vocab < 1 || vocab > INT32_MAX) return fail(AXONN_ERR_INVALID_ARG, "vocabulary size %lld", (long long)vocab);
  if (k < 0) return fail(AXONN_ERR_INVALID_ARG, "k = %d", k);
  if (h < 1 || h > 4096) return fail(AXONN_ERR_INVALID_ARG, "h = %d not in [1, 4096]", h);
  if (seq > 0 && batch > (int64_t{1} << 31) / seq)
    return fail(AXONN_ERR_UNSUPPORTED, "more than 2^31 positions");
  const int64_t T = batch * seq;
  if (!loss || !kept) return fail(AXONN_ERR_INVALID_ARG, "loss or kept is NULL");
  if (T > 0 && (!logits || !input_ids || !labels || !keep || !token_loss))
    return fail(AXONN_ERR_INVALID_ARG, "NULL input or output");
  if (ld_logits < vocab) return fail(AXONN_ERR_INVALID_ARG, "logits leading dimension below the vocabulary");
  if (ld_logits % 8 != 0 || !aligned16(logits))
    return fail(AXONN_ERR_ALIGNMENT, "logits: 16-byte aligned base and leading dimension a multiple of 8");
  if (dlogits) {
    if (ld_dlogits < vocab) return fail(AXONN_ERR_INVALID_ARG, "dlogits leading dimension below the vocabulary");
    if (ld_dlogits % 8 != 0 || !aligned16(dlogits))
      return fail(AXONN_ERR_ALIGNMENT, "dlogits: 16-byte aligned base and leading dimension a multiple of 8");
  }
  if (!axonn::goldfish_vocab_supported(vocab))
    return fail(AXONN_ERR_UNSUPPORTED, "vocabulary %lld above %lld", (long long)vocab,
                (long long)axonn::kGoldfishMaxVocab);
  DeviceState* dev = nullptr;
  axonn_status_t st = device_state(&dev);
  if (st != AXONN_OK) return st;
  axonn::GoldfishArgs a;
  a.logits = static_cast<const uint16_t*>(logits);
  a.ld_logits = ld_logits;
  a.input_ids = input_ids;
  a.labels = labels;
  a.batch = batch;
  a.seq = seq;
  a.vocab = vocab;
  a.k = k;
  a.h = h;
  a.keep = keep;
  a.token_loss = token_loss;
  a.loss = loss;
  a.kept = kept;
  a.dlogits = static_cast<uint16_t*>(dlogits);
  a.ld_dlogits = ld_dlogits;
  a.timeout_ns = g_timeout_ns.load();
  a.inject = g_inject.load();
  const cudaError_t e = axonn::goldfish_launch(a, dev->sms, stream);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "Goldfish loss launch: %s", cudaGetErrorString(e));
  return ok();
}

axonn_status_t axonn_fc_block_extents(int op, const axonn_fc_shape_t* shape, int64_t* rows,
                                      int64_t* red, int64_t* cols) {
  if (!rows || !red || !cols) return fail(AXONN_ERR_INVALID_ARG, "NULL output");
  axonn_status_t st = check_shape(op, shape, 0);
  if (st != AXONN_OK) return st;
  Range r, k, c;
  block_ranges(op, *shape, shape->x, shape->y, shape->z, &r, &k, &c);
  rows[0] = r.s; rows[1] = r.e;
  red[0] = k.s; red[1] = k.e;
  cols[0] = c.s; cols[1] = c.e;
  return ok();
}

axonn_status_t axonn_sync_status(cudaStream_t stream, uint64_t* detail) {
  if (detail) *detail = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  // One error word per kernel translation unit; report the first set.
  unsigned long long word = 0, w1 = 0, w8 = 0, w64 = 0;
  unsigned long long wg = 0;
  e = axonn::kernels_take_status<1>(&w1, stream);
  if (e == cudaSuccess) e = axonn::kernels_take_status<kFewProblems>(&w8, stream);
  if (e == cudaSuccess) e = axonn::kernels_take_status<kMaxProblems>(&w64, stream);
  if (e == cudaSuccess) e = axonn::goldfish_take_status(&wg, stream);
  if (e != cudaSuccess) return fail(AXONN_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  word = w1 ? w1 : (w8 ? w8 : (w64 ? w64 : wg));
  if (word == 0) return ok();
  if (detail) *detail = word;
  return fail(AXONN_ERR_TIMEOUT, "device wait expired: CTA %llu, site %llu", (word >> 8) & 0xFFFFFFull,
              word & 0xFFull);
}

void axonn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void axonn_debug_set_inject(int mode) { g_inject.store(mode); }

axonn_status_t axonn_set_kernel_config(int config) {
  if (config < -1 || config >= kNumConfigs)
    return fail(AXONN_ERR_INVALID_ARG, "kernel configuration %d not in [-1, %d)", config, kNumConfigs);
  g_forced_config.store(config);
  return ok();
}

int axonn_num_kernel_configs(void) { return kNumConfigs; }

axonn_status_t axonn_set_streamk(int mode) {
  if (mode < -1 || mode > 1) return fail(AXONN_ERR_INVALID_ARG, "stream-K mode %d not in {-1, 0, 1}", mode);
  g_forced_streamk.store(mode);
  return ok();
}

axonn_status_t axonn_set_l2_budget(int64_t bytes) {
  if (bytes < 0) return fail(AXONN_ERR_INVALID_ARG, "L2 budget must be >= 0");
  g_l2_budget.store(bytes);
  return ok();
}

int64_t axonn_l2_budget(void) { return g_l2_budget.load(); }

axonn_status_t axonn_set_pdl(int on) {
  if (on != 0 && on != 1) return fail(AXONN_ERR_INVALID_ARG, "PDL switch %d not 0 or 1", on);
  g_pdl.store(on);
  return ok();
}

axonn_status_t axonn_set_swap(int mode) {
  if (mode < -1 || mode > 1) return fail(AXONN_ERR_INVALID_ARG, "swap mode %d not in {-1, 0, 1}", mode);
  g_forced_swap.store(mode);
  return ok();
}

int axonn_last_swap(void) { return t_last_choice.swap; }

axonn_status_t axonn_device_info(int* sms, int* max_pairs) {
  DeviceState* d = nullptr;
  axonn_status_t st = device_state(&d);
  if (st != AXONN_OK) return st;
  if (sms) *sms = d->sms;
  if (max_pairs) *max_pairs = d->max_pairs;
  return ok();
}

const char* axonn_kernel_config_name(int config) {
  return (config >= 0 && config < kNumConfigs) ? kConfigs[config].name : "";
}

int axonn_last_kernel_config(void) { return t_last_config; }

int axonn_last_streamk_tiles(void) { return t_last_sk_tiles; }

const char* axonn_last_error(void) { return t_last_error.c_str(); }

const char* axonn_version(void) { return "axonn_fc 0.1 (sm_103a tcgen05)"; }

}  // extern "C"
