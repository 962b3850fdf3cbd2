"""fp64 CPU oracle for the FC-layer GEMMs of a 3D-parallel-matmul grid.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may load it.  It shares no code with the CUDA path; the only
thing both sides share is the seeded input generator in ``fc_inputs``.

What it follows
---------------
* The operation: Figure 1 of "Democratizing AI: Open-source Scalable LLM
  Training on GPU-based Supercomputers" (sciencestack.ai page) splits the
  matmul of one FC layer over eight GPUs in a 2x2x2 grid, by Agarwal's 3D
  parallel matrix multiplication.  An FC layer's training step is three products:
  forward Y = X.W, data gradient dX = dY.W^T, weight gradient dW = X^T.dY.
* The grid: GPUs form G_data x G_x x G_y x G_z; inside a data-parallel group
  the 3D scheme shards the matmul and moves data with all-gather,
  reduce-scatter and all-reduce -- "What carries the argument", pith.science
  review of arXiv 2502.08145.  The pages give no index formulas, so this
  oracle takes the plainest reading that the block shapes of the workloads
  fix: T (tokens) is split by G_z, K (layer input) by G_x and N (layer
  output) by G_y.  Block (x, y, z) computes
      fwd   Y^(x)_{z,y}  = X[Tz, Kx] . W[Kx, Ny]     summed over x
      dgrad dX^(y)_{z,x} = dY[Tz, Ny] . W[Kx, Ny]^T  summed over y
      wgrad dW^(z)_{x,y} = X[Tz, Kx]^T . dY[Tz, Ny]  summed over z
  and the collective's sum of partials is taken here in fp64, in fixed
  order 0..G-1 along the reduced axis.
* Uneven splits (the pages are silent): a dimension D is cut into units of
  8 elements, U = ceil(D / 8); block b of G gets floor(U/G) units plus one
  more if b < U mod G; blocks are contiguous in order and the last one is
  clipped at D.

Pins (tests/test_oracle.py): exact-rational brute force on tiny sizes, hand
worked examples (tests/golden/), identity and rank-1 closed forms, the
non-negative case S == C, the block-sum invariant, torch's bf16 rounding as a
library special case for ``bf16_rne``.  No function here is unpinned.

Storage convention: operands are numpy uint16 arrays of bf16 bits in their
stored shape; a flag ``*_t`` says the array holds the logical matrix
transposed (X logical [T x K], W [K x N], dY [T x N]).  Views with a row
stride larger than the row length are allowed (leading dimension = stride).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

OPS = ("fwd", "dgrad", "wgrad")


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` (gcc, OpenMP) into an in-tree shared library."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp",
                           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_gemm_f64.argtypes = [vp, i64, ci, vp, i64, ci, i64, i64,
                                            i64, vp, vp]
            lib.oracle_gemm_entries_f64.argtypes = [vp, i64, ci, vp, i64, ci,
                                                    i64, vp, vp, i64, vp, vp]
            lib.oracle_bf16_to_f64.argtypes = [vp, i64, vp]
            lib.oracle_f64_to_bf16.argtypes = [vp, i64, vp]
            for f in (lib.oracle_gemm_f64, lib.oracle_gemm_entries_f64,
                      lib.oracle_bf16_to_f64, lib.oracle_f64_to_bf16):
                f.restype = None
            lib.oracle_max_threads.restype = ci
            lib.oracle_set_threads.argtypes = [ci]
            lib.oracle_set_threads.restype = ci
            _lib = lib
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle's loops use."""
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> int:
    """Use `n` OpenMP threads in the oracle's loops from now on (calling
    thread); returns the count in effect."""
    return int(_load().oracle_set_threads(int(n)))


# --------------------------------------------------------------------------
# bf16 helpers
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    if b.size:
        _load().oracle_bf16_to_f64(b.ctypes.data, b.size, out.ctypes.data)
    return out


def bf16_rne(values: np.ndarray) -> np.ndarray:
    """Round doubles to bf16 bits, ties to even (IEEE 754 definition)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    if v.size:
        _load().oracle_f64_to_bf16(v.ctypes.data, v.size, out.ctypes.data)
    return out


# --------------------------------------------------------------------------
# the plain product
# --------------------------------------------------------------------------
def _ld(view: np.ndarray) -> int:
    assert view.dtype == np.uint16 and view.ndim == 2
    assert view.strides[1] == 2 or view.shape[1] <= 1, "rows must be contiguous"
    return view.strides[0] // 2 if view.shape[0] > 1 else max(view.shape[1], 1)


def _logical(view: np.ndarray, t: bool):
    """Logical (rows, cols) of a stored operand."""
    return (view.shape[1], view.shape[0]) if t else (view.shape[0], view.shape[1])


def gemm(A: np.ndarray, a_t: bool, B: np.ndarray, b_t: bool):
    """C = A . B and S = |A| . |B| in fp64 for bf16-bit operands.

    A holds logical A[M x R] (transposed if ``a_t``), B logical B[R x N]."""
    M, R = _logical(A, a_t)
    R2, N = _logical(B, b_t)
    assert R == R2, f"reduction dims differ: {R} vs {R2}"
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    if M and N and R:
        _load().oracle_gemm_f64(A.ctypes.data, _ld(A), int(a_t), B.ctypes.data,
                                _ld(B), int(b_t), M, N, R, C.ctypes.data,
                                S.ctypes.data)
    return C, S


def gemm_entries(A, a_t, B, b_t, I, J):
    """Entries (I[e], J[e]) of A . B and |A| . |B|, each a dot product."""
    M, R = _logical(A, a_t)
    R2, N = _logical(B, b_t)
    assert R == R2
    I = np.ascontiguousarray(I, dtype=np.int64)
    J = np.ascontiguousarray(J, dtype=np.int64)
    assert I.shape == J.shape
    if I.size:
        assert I.min() >= 0 and I.max() < M and J.min() >= 0 and J.max() < N
    C = np.zeros(I.shape, dtype=np.float64)
    S = np.zeros(I.shape, dtype=np.float64)
    if I.size and R:
        _load().oracle_gemm_entries_f64(A.ctypes.data, _ld(A), int(a_t),
                                        B.ctypes.data, _ld(B), int(b_t), R,
                                        I.ctypes.data, J.ctypes.data, I.size,
                                        C.ctypes.data, S.ctypes.data)
    return C, S


# --------------------------------------------------------------------------
# the three FC-layer products
# --------------------------------------------------------------------------
def _sub(view: np.ndarray, t: bool, rows, cols) -> np.ndarray:
    """Stored view of logical rows x cols of an operand."""
    (r0, r1), (c0, c1) = rows, cols
    return view[c0:c1, r0:r1] if t else view[r0:r1, c0:c1]


def operands(op: str, P, Q, p_t: bool, q_t: bool):
    """(A, a_t, B, b_t) of C = A . B for an FC op.

    fwd:   P = X, Q = W  -> Y  = X . W       A = X,   B = W
    dgrad: P = dY, Q = W -> dX = dY . W^T    A = dY,  B = W^T
    wgrad: P = X, Q = dY -> dW = X^T . dY    A = X^T, B = dY
    Reading a stored operand transposed flips its flag; no data is copied."""
    if op == "fwd":
        return P, p_t, Q, q_t
    if op == "dgrad":
        return P, p_t, Q, not q_t
    if op == "wgrad":
        return P, not p_t, Q, q_t
    raise ValueError(op)


def fc(op: str, P, Q, p_t=False, q_t=False):
    """Full-layer product for ``op`` -> (C, S)."""
    A, a_t, B, b_t = operands(op, P, Q, p_t, q_t)
    return gemm(A, a_t, B, b_t)


def fc_entries(op: str, P, Q, p_t, q_t, I, J):
    A, a_t, B, b_t = operands(op, P, Q, p_t, q_t)
    return gemm_entries(A, a_t, B, b_t, I, J)


def fc_fwd(X, W, x_t=False, w_t=False):
    return fc("fwd", X, W, x_t, w_t)


def fc_dgrad(dY, W, dy_t=False, w_t=False):
    return fc("dgrad", dY, W, dy_t, w_t)


def fc_wgrad(X, dY, x_t=False, dy_t=False):
    return fc("wgrad", X, dY, x_t, dy_t)


# --------------------------------------------------------------------------
# Agarwal 3D grid: blocks, partials and their sum
# --------------------------------------------------------------------------
def split_range(D: int, G: int, b: int):
    """Rows [start, stop) of block b when a dimension D is cut into G blocks
    (units of 8 elements, leading blocks take the extra unit)."""
    assert G >= 1 and 0 <= b < G and D >= 0
    U = (D + 7) // 8
    base, rem = divmod(U, G)
    start = 8 * (b * base + min(b, rem))
    units = base + (1 if b < rem else 0)
    return min(start, D), min(start + 8 * units, D)


def reduce_axis(op: str) -> str:
    """Grid axis whose partials sum to the op's output."""
    return {"fwd": "x", "dgrad": "y", "wgrad": "z"}[op]


def block_extents(op, T, K, N, grid, coords):
    """Logical ranges of one block product.

    Returns (a_rows, red, b_cols) -- the rows of A, the reduced range and the
    columns of B -- which are also the output rows/cols in the full result."""
    gx, gy, gz = grid
    x, y, z = coords
    Tz, Kx, Ny = split_range(T, gz, z), split_range(K, gx, x), split_range(N, gy, y)
    if op == "fwd":      # Y[Tz, Ny] += X[Tz, Kx] W[Kx, Ny]
        return Tz, Kx, Ny
    if op == "dgrad":    # dX[Tz, Kx] += dY[Tz, Ny] W[Kx, Ny]^T
        return Tz, Ny, Kx
    if op == "wgrad":    # dW[Kx, Ny] += X[Tz, Kx]^T dY[Tz, Ny]
        return Kx, Tz, Ny
    raise ValueError(op)


def fc_block(op, P, Q, p_t, q_t, T, K, N, grid, coords):
    """One block product of the grid -> (C_blk, S_blk, out_rows, out_cols)."""
    rows, red, cols = block_extents(op, T, K, N, grid, coords)
    A, a_t, B, b_t = operands(op, P, Q, p_t, q_t)
    Ab = _sub(A, a_t, rows, red)
    Bb = _sub(B, b_t, red, cols)
    C, S = gemm(Ab, a_t, Bb, b_t)
    return C, S, rows, cols


def out_shape(op, T, K, N):
    return {"fwd": (T, N), "dgrad": (T, K), "wgrad": (K, N)}[op]


def fc_vgrid(op, P, Q, p_t, q_t, T, K, N, grid):
    """All Gx*Gy*Gz block products, partials summed over the op's reduced axis
    in fixed order (0..G-1), assembled into the full output -> (C, S).  The
    blocks only regroup a sum of exact products, so C equals ``fc`` up to
    fp64 reassociation."""
    gx, gy, gz = grid
    M, Nn = out_shape(op, T, K, N)
    C = np.zeros((M, Nn), dtype=np.float64)
    S = np.zeros((M, Nn), dtype=np.float64)
    axis = reduce_axis(op)
    G = {"x": gx, "y": gy, "z": gz}[axis]
    for g in range(G):  # fixed order along the reduced axis
        for x in range(gx):
            for y in range(gy):
                for z in range(gz):
                    if {"x": x, "y": y, "z": z}[axis] != g:
                        continue
                    Cb, Sb, rows, cols = fc_block(op, P, Q, p_t, q_t, T, K, N,
                                                  grid, (x, y, z))
                    C[rows[0]:rows[1], cols[0]:cols[1]] += Cb
                    S[rows[0]:rows[1], cols[0]:cols[1]] += Sb
    return C, S


# --------------------------------------------------------------------------
# Z-sharded weights: all-gather and reduce-scatter over the Z group
# --------------------------------------------------------------------------
def shard_rows(Wblk: np.ndarray, G: int):
    """Row shards of a weight block: shard z = rows split_range(rows, G, z)."""
    return [Wblk[slice(*split_range(Wblk.shape[0], G, z))] for z in range(G)]


def gather_shards(shards):
    """The all-gather over the Z group: the shards stacked back in order."""
    return np.concatenate(list(shards), axis=0)


def wgrad_zsharded(X, dY, x_t, dy_t, T, K, N, grid, xy):
    """Weight gradient of block (x, y): the Z-group partials dW^(z)_{x,y} summed
    in order z = 0..Gz-1 (fp64), then cut into the Gz row shards that the
    reduce-scatter leaves on the ranks -> (list of C shards, list of S shards)."""
    gx, gy, gz = grid
    x, y = xy
    Kx, Ny = split_range(K, gx, x), split_range(N, gy, y)
    C = np.zeros((Kx[1] - Kx[0], Ny[1] - Ny[0]))
    S = np.zeros_like(C)
    for z in range(gz):
        Cb, Sb, _, _ = fc_block("wgrad", X, dY, x_t, dy_t, T, K, N, grid, (x, y, z))
        C += Cb
        S += Sb
    return shard_rows(C, gz), shard_rows(S, gz)


# --------------------------------------------------------------------------
# acceptance bound
# --------------------------------------------------------------------------
def error_ratio(c_test: np.ndarray, C: np.ndarray, S: np.ndarray,
                rel: float = 1e-2, abs_: float = 1e-5) -> np.ndarray:
    """|c_test - C| / (rel * S + abs); every entry must be <= 1."""
    return np.abs(np.asarray(c_test, np.float64) - C) / (rel * S + abs_)
