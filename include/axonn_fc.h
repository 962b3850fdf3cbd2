/*
 * axonn_fc.h -- C ABI of the GB300 FC-layer GEMM library (libaxonn_fc.so).
 *
 * What it computes.  The three matrix products of a fully-connected layer's
 * training step, either on the whole layer or on one local block of
 * Agarwal's 3D parallel matrix multiplication.  Figure 1 of "Democratizing
 * AI: Open-source Scalable LLM Training on GPU-based Supercomputers" shows
 * one FC layer's matmul split this way over a virtual grid whose three
 * extents are G_x, G_y and G_z; the pith.science review of arXiv
 * 2502.08145 ("What carries the argument") places that grid inside a 4D
 * one, G_data x G_x x G_y x G_z, joined by collectives:
 *
 *   forward          Y[T x N]  = X[T x K] . W[K x N]
 *   data gradient    dX[T x K] = dY[T x N] . W^T
 *   weight gradient  dW[K x N] = X^T . dY
 *
 * Inputs and outputs are bf16; products accumulate in fp32 on the tensor
 * cores and are rounded once, to nearest even, when written as bf16.
 *
 * 3D grid.  T is split by G_z, K by G_x and N by G_y.  Block (x, y, z) owns
 * X[Tz, Kx], W[Kx, Ny] and dY[Tz, Ny] and computes
 *   fwd    Y^(x)_{z,y}  = X[Tz,Kx] . W[Kx,Ny]      (partials summed over x)
 *   dgrad  dX^(y)_{z,x} = dY[Tz,Ny] . W[Kx,Ny]^T   (summed over y)
 *   wgrad  dW^(z)_{x,y} = X[Tz,Kx]^T . dY[Tz,Ny]   (summed over z)
 * A dimension D is cut into units of 8 elements: with U = ceil(D/8), block b
 * of G gets floor(U/G) units plus one if b < U mod G, blocks are contiguous
 * in order, and the last block is clipped at D (see axonn_block_range).
 *
 * Virtual grid (AXONN_VGRID).  All G_x*G_y*G_z block products run on this
 * GPU, and an on-device sum over the reduced axis (G = G_x for fwd, G_y for
 * dgrad, G_z for wgrad) stands in for the grid's all-reduce /
 * reduce-scatter.  Three forms:
 *  - default (chained): each output tile runs the G block products of its
 *    output block one after another, in order g = 0..G-1, into one fp32
 *    accumulator on the tensor cores, each block product read from its own
 *    block (its own tensor maps, zero-filled at the block's edges).  One
 *    launch, no workspace, no partial in memory; results are the same on
 *    every run.
 *  - AXONN_VGRID_PARTIALS: one launch writes the partials 0..G-2 in fp32 to
 *    the caller's workspace, and a second computes partial G-1, whose
 *    epilogue adds partials 0..G-1 in that order and writes the output
 *    (the partials as the grid's ranks would hold them); results are the
 *    same on every run, and may differ from the chained form in the last
 *    bits (another summation order).
 *  - AXONN_REDUCE_ADD (fp32 accumulating output only): all blocks run in
 *    one launch and each adds its tile into the output with fp32 reduction
 *    adds (PTX red.global.add: rounded to nearest even, subnormal inputs
 *    and results flushed to zero): no workspace, and a summation order that
 *    can change from run to run (every order stays within the same error
 *    bound; integer-valued sums below 2^24 are exact in any order).
 *
 * Conventions for every entry point below.
 *  - Pointers are DEVICE pointers; the caller owns every buffer and the
 *    stream.  The library never allocates device memory on a call; scratch
 *    comes from the caller's workspace (axonn_fc_workspace_size).
 *  - Layout: matrices are row-major with a leading dimension (row stride) in
 *    elements.  Flag AXONN_A_T says the op's first operand (X for fwd and
 *    wgrad, dY for dgrad) is stored transposed, i.e. as [K x T] / [N x T];
 *    AXONN_B_T says the second operand (W for fwd and dgrad, dY for wgrad) is
 *    stored transposed ([N x K] for W -- PyTorch's Linear layout -- or
 *    [N x T] for dY).  Outputs are always row-major in their logical shape.
 *  - Alignment: every base pointer 16-byte aligned; bf16 leading dimensions
 *    multiples of 8, fp32 ones multiples of 4.  Otherwise AXONN_ERR_ALIGNMENT.
 *  - Calls are asynchronous on `stream`.  A device-side timeout (a bounded
 *    wait inside a kernel that expired) is reported by axonn_sync_status.
 *  - Errors are status codes; axonn_last_error() gives a thread-local message.
 *    No C++ exception crosses this boundary.
 *  - Threads: every entry point may be called from several host threads at
 *    once (on different streams); the tuning table and per-device set-up are
 *    guarded by locks.  The kernel-configuration override and the wait
 *    timeout are process-wide.
 *  - Empty outputs (an extent of 0) return AXONN_OK and touch nothing; an
 *    empty reduction range writes zeros (leaves C bit for bit unchanged
 *    with AXONN_ACCUM_F32).
 */
#ifndef AXONN_FC_H_
#define AXONN_FC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  AXONN_OK = 0,
  AXONN_ERR_INVALID_ARG = 1,  /* bad size, grid, coordinate, flag or pointer */
  AXONN_ERR_ALIGNMENT = 2,    /* pointer or leading dimension misaligned */
  AXONN_ERR_UNSUPPORTED = 3,  /* valid request the library cannot run */
  AXONN_ERR_WORKSPACE = 4,    /* workspace missing or too small */
  AXONN_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  AXONN_ERR_TIMEOUT = 6       /* a bounded device-side wait expired */
} axonn_status_t;

typedef enum { AXONN_OP_FWD = 0, AXONN_OP_DGRAD = 1, AXONN_OP_WGRAD = 2 } axonn_op_t;

/* Layer sizes, grid and block coordinate.  A full-layer product is the grid
 * 1x1x1 at (0,0,0).  gx, gy, gz >= 1; 0 <= x < gx etc. */
typedef struct {
  int64_t T, K, N;
  int32_t gx, gy, gz;
  int32_t x, y, z;
} axonn_fc_shape_t;

/* Flags (bitwise or). */
#define AXONN_A_T 0x1u            /* first operand stored transposed */
#define AXONN_B_T 0x2u            /* second operand stored transposed */
#define AXONN_ACCUM_F32 0x4u      /* output is fp32 and the result is added (one fp32
                                     reduction add per element: round to nearest even,
                                     subnormals flushed to zero) */
#define AXONN_VGRID 0x8u          /* all blocks + on-device partial sum */
#define AXONN_FULL_OPERANDS 0x10u /* block mode: pointers are full matrices */
#define AXONN_OUT_F32 0x20u       /* output is fp32, overwritten */
#define AXONN_ZSHARDED 0x40u      /* axonn_fc_workspace_size of axonn_fc_wgrad_zsharded */
#define AXONN_REDUCE_ADD 0x80u    /* with AXONN_VGRID | AXONN_ACCUM_F32: every block added
                                     into the output by fp32 reduction adds, in no fixed
                                     order; one launch, no workspace */
#define AXONN_VGRID_PARTIALS 0x100u /* with AXONN_VGRID: the two-launch form, fp32 partials
                                     of blocks 0..G-2 in the workspace, summed in order in
                                     the last block's epilogue */

/*
 * Forward product Y = X . W of the layer, of block (x,y,z), or of the whole
 * virtual grid.
 *   X   first operand, [T x K] (or [K x T] with AXONN_A_T), leading dim ldx
 *   W   second operand, [K x N] (or [N x K] with AXONN_B_T), leading dim ldw
 *   Y   output [T x N], leading dim ldy; bf16 unless AXONN_ACCUM_F32 /
 *       AXONN_OUT_F32 make it fp32
 *   Block mode (no AXONN_VGRID, grid larger than 1): without
 *   AXONN_FULL_OPERANDS the pointers address the block's own shards
 *   (X_blk [Tz x Kx], W_blk [Kx x Ny], Y_blk [Tz x Ny], each with its ld);
 *   with it they address the full matrices and the block is located by its
 *   offsets, its partial written at Y[Tz, Ny].
 *   ws / ws_bytes: device workspace, needed with AXONN_VGRID |
 *   AXONN_VGRID_PARTIALS when G_x > 1 (size from
 *   axonn_fc_workspace_size).  Otherwise optional: a full-size one enables
 *   the stream-K tail of large products; NULL / 0 runs without it.
 *   Reduction split: a single product (no AXONN_VGRID) whose tiles leave
 *   SMs idle may have its reduction range cut into S = 2, 4 or 8 pieces of
 *   whole 64-deep stages, computed by the S CTAs of a thread-block cluster
 *   and added in fixed order (pieces 0, 1, ..., S-1) inside it, with no
 *   workspace and no extra launch.  Without a tuning entry it is chosen
 *   for reductions of 32 stages or more; the tuner times S = 2, 4, 8.
 */
axonn_status_t axonn_fc_fwd(const void* X, const void* W, void* Y, int64_t ldx, int64_t ldw,
                            int64_t ldy, const axonn_fc_shape_t* shape, uint32_t flags,
                            void* ws, size_t ws_bytes, cudaStream_t stream);

/* Data gradient dX = dY . W^T.  dY [T x N] (AXONN_A_T: [N x T]), W [K x N]
 * (AXONN_B_T: [N x K]), dX [T x K].  Block (x,y,z) yields dX^(y)_{z,x};
 * the virtual grid sums over y.  Other arguments as for axonn_fc_fwd. */
axonn_status_t axonn_fc_dgrad(const void* dY, const void* W, void* dX, int64_t lddy,
                              int64_t ldw, int64_t lddx, const axonn_fc_shape_t* shape,
                              uint32_t flags, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Weight gradient dW = X^T . dY.  X [T x K] (AXONN_A_T: [K x T]), dY
 * [T x N] (AXONN_B_T: [N x T]), dW [K x N].  Block (x,y,z) yields
 * dW^(z)_{x,y}; the virtual grid sums over z.  AXONN_ACCUM_F32 gives the
 * fp32 main-gradient update dW += X^T . dY. */
axonn_status_t axonn_fc_wgrad(const void* X, const void* dY, void* dW, int64_t ldx,
                              int64_t lddy, int64_t lddw, const axonn_fc_shape_t* shape,
                              uint32_t flags, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Z-sharded weights of the 3D grid.  Each rank (x, y, z) keeps only shard z
 * of its weight block W_{x,y}; the grid all-gathers the block over the Z
 * group before using it and reduce-scatters the weight-gradient partials
 * over the Z group into shards (the review of arXiv 2502.08145, "What
 * carries the argument", has the weights split over the Z axis and data
 * moved by all-gather, reduce-scatter and all-reduce).  Shards are row
 * blocks of W_{x,y} cut by the grid's split rule (units of 8 rows, leading
 * shards take the extra unit; see axonn_block_range).
 *
 * axonn_shards_gather -- the all-gather, on one GPU: copies g bf16 row
 * shards, shard z = rows [split(rows, g, z)) stored row-major with leading
 * dimension ld_shard at shards[z] (a HOST array of g DEVICE pointers), into
 * `out` [rows x cols] (leading dimension ld_out).  cols, ld_shard and ld_out
 * must be multiples of 8 and every pointer 16-byte aligned
 * (AXONN_ERR_ALIGNMENT); 1 <= g <= 64.
 *
 * axonn_fc_wgrad_zsharded -- the Z-group weight gradient with its
 * reduce-scatter, on one GPU: for block (shape->x, shape->y) it computes
 * every partial dW^(z)_{x,y} = X[Tz,Kx]^T . dY[Tz,Ny], z = 0..G_z-1, sums
 * them in fixed order z = 0..G_z-1 and writes row shard z' of the sum to
 * dW_shards[z'] (a HOST array of G_z DEVICE pointers; each [rows of shard z'
 * x Ny], leading dimension ld_shard; bf16, or fp32 with AXONN_OUT_F32 /
 * AXONN_ACCUM_F32).  X and dY are the full [T x K] and [T x N] matrices (or
 * transposed with AXONN_A_T / AXONN_B_T); shape->z is ignored.  Partials
 * 0..G_z-2 go to `ws`: axonn_fc_workspace_size(AXONN_OP_WGRAD, shape,
 * AXONN_ZSHARDED) bytes.
 */
axonn_status_t axonn_shards_gather(const void* const* shards, int32_t g, int64_t rows, int64_t cols,
                                   int64_t ld_shard, void* out, int64_t ld_out, cudaStream_t stream);
axonn_status_t axonn_fc_wgrad_zsharded(const void* X, const void* dY, void* const* dW_shards,
                                       int64_t ldx, int64_t lddy, int64_t ld_shard,
                                       const axonn_fc_shape_t* shape, uint32_t flags, void* ws,
                                       size_t ws_bytes, cudaStream_t stream);

/*
 * Virtual-grid product (as the entry points above with AXONN_VGRID) that
 * allocates nothing and needs no workspace argument.  The pages have no
 * counterpart: this exists for callers that cannot call cudaMalloc, such as
 * code that runs inside a host framework that owns all device memory, or
 * code that must not allocate once it is running.
 *   op        axonn_op_t; P, Q, C and ld* as for that op's entry point
 *   flags     as for the entry points; AXONN_VGRID is implied
 * The fp32 partials of the two-launch form (AXONN_VGRID_PARTIALS) live in
 * a fixed 64 MiB scratch array inside the library, which every GPU that
 * loads the library holds until the process exits.  A product whose
 * partials need more ((G-1) * M * ceil8(N) * 4 bytes, G the reduced grid
 * extent, M x N the output) returns AXONN_ERR_WORKSPACE with a message.
 * The default chained form, AXONN_REDUCE_ADD and products whose reduced
 * axis has one block need no scratch.  The first call
 * on each device looks up the scratch's device address (once, with that
 * device current); make that first call before any stream capture.  Every
 * call uses the same scratch and the kernels overwrite every partial they
 * later read, so no clearing is needed -- but calls that overlap on the GPU
 * (on different streams, or from different threads) race on it and must be
 * serialised by the caller.
 */
axonn_status_t axonn_fc_vgrid_static(int op, const void* P, const void* Q, void* C, int64_t ldp,
                                     int64_t ldq, int64_t ldc, const axonn_fc_shape_t* shape,
                                     uint32_t flags, cudaStream_t stream);

/*
 * Goldfish-loss masked cross-entropy over bf16 logits, with its gradient.
 * Against memorisation the paper trains with Goldfish Loss, which leaves
 * tokens out of the cross-entropy at random (pith.science review of arXiv
 * 2502.08145, "What carries the argument"), with mask parameters k = 2 and
 * h = 13 ("Assumptions & free parameters").  The rule, read from the
 * method's own paper that the pages cite (Hans et al., arXiv 2406.10209):
 *   label (b, t) is dropped when FNV-1a-64 of input_ids[b, t-h+1 .. t] (each
 *   id as 4 little-endian bytes, oldest first) is 0 mod k; labels with
 *   fewer than h tokens before them in their row are kept; k = 0 keeps all;
 *   labels outside [0, vocab) are padding (neither kept nor counted).
 *   CE_t = logsumexp(z_t) - z_t[y_t] (natural log, fp32 arithmetic)
 *   loss = sum over kept t of CE_t / n, n = number kept (0 when n = 0)
 *   dlogits_t = G_t (softmax(z_t) - e_{y_t}) / n  (zero rows where dropped)
 * Arguments (DEVICE pointers, caller-owned; T = batch * seq positions in
 * row-major (b, t) order):
 *   logits      bf16 [T x vocab], leading dimension ld_logits (multiple of
 *               8, 16-byte aligned base); rows of dropped labels are not read
 *   input_ids   int32 [batch x seq], the tokens the windows are hashed from
 *   labels      int32 [batch x seq], the token each position predicts
 *   keep        out, uint8 [T]: 1 where the label counts
 *   token_loss  out, fp32 [T]: CE_t where kept, 0 elsewhere
 *   loss        out, fp32 [1]: the mean over kept labels (a fixed-order sum);
 *               during the call its word is the kernels' row counter
 *   kept        out, int32 [1]: n
 *   dlogits     out, bf16 [T x vocab] with ld_dlogits (same alignment), or
 *               NULL for the loss alone
 * 1 <= h <= 4096, k >= 0, vocab up to 8 x 49152.  Three kernel launches on
 * `stream`, no workspace, no allocation.  A wait that expires is reported
 * by axonn_sync_status.  AXONN_ERR_INVALID_ARG / _ALIGNMENT / _UNSUPPORTED
 * as for the products.
 */
axonn_status_t axonn_goldfish_ce(const void* logits, int64_t ld_logits, const int32_t* input_ids,
                                 const int32_t* labels, int64_t batch, int64_t seq, int64_t vocab,
                                 int32_t k, int32_t h, uint8_t* keep, float* token_loss,
                                 float* loss, int32_t* kept, void* dlogits, int64_t ld_dlogits,
                                 cudaStream_t stream);

/*
 * Per-shape tuning -- the GB300 counterpart of the automatic tuning of BLAS
 * kernels that the pages credit (TL;DR of the sciencestack.ai page; "The
 * reading", review of arXiv 2502.08145).  Runs this call once per candidate -- kernel
 * configuration x rasterisation group {8, 16 tile rows; 8, 16 tile columns,
 * written -8, -16}, every configuration for products that leave SMs idle
 * (with reduction splits {2, 4, 8} of the 128x128 and 128x64
 * configurations, each piece
 * at least 128 deep), the 128x256 and 256-row configurations otherwise,
 * and the two best of them again with the
 * operand roles exchanged (see axonn_set_swap) -- and times each (through a captured
 * CUDA graph of 3 calls, 20 for products under 2e10 FLOP, where the stream
 * allows it) relative to the default choice run just before and after it,
 * so clock drift under the power cap cancels.  For products of 2e11 FLOP or
 * more, a candidate within 2 % of the fastest that loads fewer operand
 * bytes from L2 per multiply-add is kept instead (under the power cap those
 * bytes cost clock in a long run, which short timings do not show).  The
 * call synchronises `stream`.  It
 * records the fastest for later calls with the same op, sizes, grid, block
 * and flags on a GPU with the same SM count.  Arguments are those of the
 * op's entry point (op is an axonn_op_t); the caller's output is
 * overwritten (with AXONN_ACCUM_F32 the runs overwrite instead of adding;
 * with AXONN_REDUCE_ADD as well they add, once per run: tune on a scratch
 * output).  Not for use during stream capture.  Any
 * of the result pointers may be NULL.
 */
axonn_status_t axonn_fc_tune(int op, const void* P, const void* Q, void* C, int64_t ldp,
                             int64_t ldq, int64_t ldc, const axonn_fc_shape_t* shape,
                             uint32_t flags, void* ws, size_t ws_bytes, cudaStream_t stream,
                             int* best_config, int* best_split, int* best_group_m,
                             float* best_us);

/* The tuning table as text, one JSON object per line:
 *   {"key": "...", "config": "<name>", "split": S, "group_m": G,
 *    "streamk": 0 | 1 | 2, "swap": 0 | 1, "us": t}
 * (S a whole number 1..8, run as the largest power of two not above it
 * or the product's stage count, and only on the 128x128 and 128x64
 * configurations;
 * G a whole number in -64..-1 or 1..64, tile rows
 * per rasterisation group, negative for tile columns; streamk: off, on for
 * a partial round at most a quarter full, on wherever it applies; a line
 * without it loads as 1; swap: operand roles exchanged, see axonn_set_swap;
 * a line without it loads as 0).
 * save writes every entry; load merges a file's entries into the table
 * (AXONN_ERR_INVALID_ARG on an unreadable file or a malformed line, leaving
 * the table unchanged).  Host-only. */
axonn_status_t axonn_tune_cache_save(const char* path);
axonn_status_t axonn_tune_cache_load(const char* path);
void axonn_tune_cache_clear(void);
int axonn_tune_cache_size(void);

/* Whether the tuning table holds an entry that a call of op `op` (an
 * axonn_op_t) with this shape and these flags would run on the current
 * device (same SM count): *found = 1, else 0 (the call runs the default
 * choice).  AXONN_ERR_INVALID_ARG for a bad shape or flag or a NULL
 * `found`; AXONN_ERR_CUDA without a usable device.  Launches nothing. */
axonn_status_t axonn_tune_lookup(int op, const axonn_fc_shape_t* shape, uint32_t flags,
                                 int* found);

/* How the last call on this thread ran: kernel configuration, reduction
 * split and rasterisation group. */
void axonn_last_choice(int* config, int* split, int* group_m);

/* Workspace bytes an op needs with these flags (0 when none).  `op` is an
 * axonn_op_t.  With AXONN_VGRID | AXONN_VGRID_PARTIALS it is the fp32
 * partials 0..G-2 of the reduced grid axis ((G-1) * M * ceil8(N) * 4); the
 * other virtual-grid forms need none.  Without AXONN_VGRID it is nonzero
 * for products of more than one wave of 128x128 tiles, which may run a
 * stream-K tail (see axonn_set_streamk; up to about 80 MB on a 152-SM GPU);
 * the reduction split needs none.  Passing less workspace just disables
 * the tail.
 * Returns AXONN_ERR_INVALID_ARG for a bad shape or flag. */
axonn_status_t axonn_fc_workspace_size(int op, const axonn_fc_shape_t* shape, uint32_t flags,
                                       size_t* bytes);

/* Rows [*start, *stop) of block b when a dimension D is cut into G blocks by
 * the 8-element-unit rule above.  Host-only, no GPU needed. */
axonn_status_t axonn_block_range(int64_t D, int32_t G, int32_t b, int64_t* start, int64_t* stop);

/* Logical ranges of block (shape->x, shape->y, shape->z) of op `op` (an
 * axonn_op_t), as the product entry points resolve them: rows[2] = its
 * output rows, red[2] = its reduced range, cols[2] = its output columns,
 * each [start, stop) in the full matrices (forward: Tz, Kx, Ny; data
 * gradient: Tz, Ny, Kx; weight gradient: Kx, Tz, Ny -- the block products
 * of Figure 1 of the sciencestack.ai page under the reading T by G_z, K by
 * G_x, N by G_y).  AXONN_ERR_INVALID_ARG for a bad op, shape or
 * coordinate or a NULL output.  Host-only, no GPU needed. */
axonn_status_t axonn_fc_block_extents(int op, const axonn_fc_shape_t* shape, int64_t* rows,
                                      int64_t* red, int64_t* cols);

/* Waits for `stream`, then reports (and clears) a device-side timeout
 * recorded by any kernel of this library on the current device since the
 * last call: AXONN_ERR_TIMEOUT, AXONN_ERR_CUDA if the stream failed, else
 * AXONN_OK.  *detail (may be NULL) receives the raw error word. */
axonn_status_t axonn_sync_status(cudaStream_t stream, uint64_t* detail);

/* Upper bound, in nanoseconds, on any single wait inside the kernels
 * (default 4e9).  Process-wide; applies to launches made afterwards. */
void axonn_set_wait_timeout_ns(uint64_t ns);

/* Test hook: 1 makes the next launches' producer withhold all operand
 * loads (the GEMM kernels' tiles, the Goldfish loss's kept rows), so the
 * bounded waits expire and AXONN_ERR_TIMEOUT is reported; 0 restores normal
 * operation.  Never needed in production. */
void axonn_debug_set_inject(int mode);

/* Kernel configurations.  The library chooses one per call from the
 * problem's tile counts (the pages' automatic BLAS kernel tuning: review of
 * arXiv 2502.08145, "The reading"); these calls expose the choice.
 *   0  1cta_128x128      one CTA per 128x128 output tile, 64-deep stages
 *   1  1cta_128x256      one CTA per 128x256 output tile, 64-deep stages
 *   2  pair_256x256      a CTA pair (cluster of 2, cta_group::2 MMA) per
 *                        256x256 output tile, 64-deep stages
 *   3  1cta_256x256      one CTA per 256x256 output tile (two M=128 MMAs
 *                        per B slice), 3 stages, single-buffered TMEM
 *   4  1cta_128x192      one CTA per 128x192 output tile, 5 stages
 *   5  1cta_256x192      one CTA per 256x192 output tile, 4 stages
 *   6  pair_512x256      a CTA pair per 512x256 output tile (each CTA two
 *                        M=128 halves of 256 columns), 4 stages, 12 warps
 *   7  1cta_128x64       one CTA per 128x64 output tile, 8 stages (for
 *                        products with too few larger tiles)
 * (the N=192 tiles trade a little operand reuse for fewer idle SMs in the
 * last wave on shapes such as 8192 x 6144; configurations 0 and 7 also run
 * the reduction split inside a cluster)
 * axonn_set_kernel_config(c) forces configuration c for all later calls in
 * the process (-1 restores automatic choice); AXONN_ERR_INVALID_ARG if c is
 * out of range.  axonn_last_kernel_config() is the configuration the last
 * GEMM launch on this thread used (-1 before any). */
axonn_status_t axonn_set_kernel_config(int config);
/* SM count of the current device and how many CTA pairs (clusters of 2
 * running configuration 2) it keeps resident at once. */
axonn_status_t axonn_device_info(int* sms, int* max_pairs);
int axonn_num_kernel_configs(void);

/* Stream-K tail for later calls in this process: -1 = as tuned, 0 = off,
 * 1 = on wherever it applies.  It applies to a single-product call that is
 * given the workspace axonn_fc_workspace_size reports and whose output
 * tiles do not fill a whole number of rounds of the persistent grid: the
 * last partial round plus one full round are cut into equal ranges of
 * 64-deep reduction steps, one per CTA (or CTA pair).  Untuned calls use it
 * only when the partial round is at most a quarter full; the tuner times
 * off, that default and always-on, and keeps the fastest.  Each such tile
 * is computed in at most two pieces; the second to finish adds the other's
 * fp32 partial (two terms, the same sum in either order), so results are
 * deterministic for a given shape and GPU but may differ in the last bit
 * from a call with it off.  No CTA waits for another, so concurrent
 * launches cannot stall each other.
 * Not part of the source pages: it removes the idle SMs of the last wave.
 * AXONN_ERR_INVALID_ARG for another mode.  Host-only. */
axonn_status_t axonn_set_streamk(int mode);

/* Operand roles for later calls in this process: -1 = as tuned (default
 * off), 0 = never exchanged, 1 = exchanged wherever it applies.  Exchanged,
 * a call computes the transpose of its product, C^T = B^T . A^T: the second
 * operand is read in the first operand's role (output rows) and the first
 * in the second's, and the epilogue writes each tile back transposed, so
 * the caller's output is the same matrix.  The tuner times the swap for the
 * two best configurations of each call, the row-major BLAS counterpart of
 * choosing among NN, NT and TN operand orders (the pages' automatic BLAS
 * kernel tuning: TL;DR of the sciencestack.ai page; review of arXiv
 * 2502.08145, "The reading").  It does not apply with AXONN_VGRID_PARTIALS.
 * Results may differ from the unswapped call in the
 * last bit (another tile order of the same fp32 sums).  Host-only;
 * AXONN_ERR_INVALID_ARG for another mode. */
axonn_status_t axonn_set_swap(int mode);

/* Programmatic dependent launch of the GEMM kernels (1, the default): each
 * launch may start while the previous kernel in the stream finishes, so its
 * barrier set-up, TMEM allocation and tensor-map prefetch overlap that
 * kernel's last tiles; it reads and writes global memory only after the
 * previous kernel has completed (griddepcontrol.wait), so stream order is
 * kept.  0 launches them plainly.  Process-wide, host-only;
 * AXONN_ERR_INVALID_ARG for another value. */
axonn_status_t axonn_set_pdl(int on);

/* L2 priorities of the GEMM operand loads.  A rasterisation group walks its
 * tile rows (or columns) across the whole product, so each later wave of
 * the group reads the group's panel of that operand again, while the other
 * operand's panels pass through once.  With a budget of `bytes` > 0 the
 * kept operand's loads mark their lines evict-last (the fraction
 * min(1, bytes / panel bytes) of them, panel = group x tile edge x
 * reduction x 2; createpolicy and the .L2::cache_hint form of the tensor
 * copies); the other operand's keep the default priority.  0 issues all
 * loads with the default priority.  Default 64 MiB.  Results are unchanged
 * either way.
 * Process-wide, host-only; AXONN_ERR_INVALID_ARG for a negative value. */
axonn_status_t axonn_set_l2_budget(int64_t bytes);
int64_t axonn_l2_budget(void);

/* 1 if the last call on this thread ran with exchanged operand roles. */
int axonn_last_swap(void);

/* Output tiles the last GEMM launch on this thread computed as stream-K
 * pieces (0: none).  Host-only. */
int axonn_last_streamk_tiles(void);
const char* axonn_kernel_config_name(int config);
int axonn_last_kernel_config(void);

/* Thread-local description of the last error returned on this thread. */
const char* axonn_last_error(void);

/* Library version string. */
const char* axonn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AXONN_FC_H_ */
