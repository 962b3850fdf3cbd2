"""Communication performance model of the 4D grid -- a CPU planning tool.

Purpose: rank grid configurations G_data x G_x x G_y x G_z for a set of FC
layers before running them, as the pages' performance model does.  The
pith.science review of arXiv 2502.08145 (its circularity check, and the
Figure 2 caption) says that model takes ring-collective formulas and
separately measured bandwidths to predict communication time, and that it
put 9 of the 10 fastest configurations in the right places.  The
pages state its assumptions but not its equations, so this module writes the
plainest model those assumptions fix; its parity with the pages' Equations
1-7 cannot be checked (parity unpinned):

* Assumption 1: every all-gather, reduce-scatter and all-reduce is a ring.
  A ring all-gather or reduce-scatter of a tensor of S bytes over p ranks
  moves (p-1)/p * S bytes through each rank's link; a ring all-reduce (a
  reduce-scatter followed by an all-gather) moves 2 (p-1)/p * S.
* Assumption 3: message start-up is negligible, so time = bytes / bandwidth.
* Assumption 5: one inter-node bandwidth for every pair of nodes.
* Intra-node bandwidths are measured per process-group size and looked up.

Rank layout (not given on the pages; the plainest reading): ranks are
numbered with x fastest, then y, then z, then the data-parallel index.  A
group along an axis uses the intra-node bandwidth when every group along
that axis lies inside one node (for power-of-two grids: when stride x size
divides the GPUs per node).

Per FC layer [K -> N] with T tokens per data-parallel group, block (x,y,z)
holds X[T/Gz x K/Gx], W[K/Gx x N/Gy], dY[T/Gz x N/Gy]:

  forward  all-gather W_{x,y} over Z;  all-reduce Y^(x)_{z,y} over X
  dgrad    all-gather W_{x,y} over Z;  all-reduce dX^(y)_{z,x} over Y
  wgrad    reduce-scatter dW_{x,y} over Z
  data     all-reduce the weight-gradient shard over G_data

The compute term is the layer's FLOPs per GPU over a sustained per-GPU GEMM
rate (the rate this library measures on one GB300 by default).  Overlap of
communication with compute is not modelled.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from itertools import product

BYTES_BF16 = 2


@dataclass
class Machine:
    """Bandwidths (GB/s per GPU through its ring link) and the per-GPU GEMM rate."""
    gpus_per_node: int
    inter_node_gbs: float
    intra_node_gbs: dict = field(default_factory=dict)   # group size -> GB/s
    gpu_tflops: float = 1650.0

    def intra(self, size: int) -> float:
        if size in self.intra_node_gbs:
            return float(self.intra_node_gbs[size])
        if not self.intra_node_gbs:
            return float(self.inter_node_gbs)
        # nearest profiled group size not smaller, else the largest profiled
        larger = [s for s in self.intra_node_gbs if s >= size]
        key = min(larger) if larger else max(self.intra_node_gbs)
        return float(self.intra_node_gbs[key])


def ring_time(kind: str, nbytes: float, p: int, gbs: float) -> float:
    """Seconds for a ring collective over p ranks on a tensor of nbytes."""
    if p <= 1 or nbytes <= 0:
        return 0.0
    factor = {"all_gather": 1.0, "reduce_scatter": 1.0, "all_reduce": 2.0}[kind]
    return factor * (p - 1) / p * nbytes / (gbs * 1e9)


def axis_stride(grid, axis: str) -> int:
    """Rank stride of a process group along `axis` of grid (Gd, Gx, Gy, Gz)."""
    gd, gx, gy, gz = grid
    return {"x": 1, "y": gx, "z": gx * gy, "data": gx * gy * gz}[axis]


def axis_size(grid, axis: str) -> int:
    gd, gx, gy, gz = grid
    return {"x": gx, "y": gy, "z": gz, "data": gd}[axis]


def groups_within_nodes(grid, axis: str, gpus_per_node: int) -> bool:
    """Whether every process group along `axis` lies inside one node.  The
    group of first rank b holds b, b + s, ..., b + (g-1) s (stride s, size g),
    and its first ranks are i + s g j with i < s.  b mod P (P = GPUs per
    node) repeats with period at most P in both i and j, so P x P candidates
    decide it."""
    size, stride = axis_size(grid, axis), axis_stride(grid, axis)
    if size == 1:
        return True
    n = grid[0] * grid[1] * grid[2] * grid[3]
    block = stride * size
    P = gpus_per_node
    for j in range(min(n // block, P)):
        for i in range(min(stride, P)):
            if (i + block * j) % P + (size - 1) * stride >= P:
                return False
    return True


def group_bandwidth(grid, axis: str, m: Machine) -> float:
    if groups_within_nodes(grid, axis, m.gpus_per_node):
        return m.intra(axis_size(grid, axis))
    return float(m.inter_node_gbs)


def layer_comm(T: int, K: int, N: int, grid, m: Machine) -> dict:
    """Seconds of each collective of one FC layer's training step."""
    gd, gx, gy, gz = grid
    w_blk = BYTES_BF16 * (K / gx) * (N / gy)
    y_blk = BYTES_BF16 * (T / gz) * (N / gy)
    dx_blk = BYTES_BF16 * (T / gz) * (K / gx)
    bw = {a: group_bandwidth(grid, a, m) for a in ("x", "y", "z", "data")}
    return {
        "fwd_allgather_w_z": ring_time("all_gather", w_blk, gz, bw["z"]),
        "fwd_allreduce_y_x": ring_time("all_reduce", y_blk, gx, bw["x"]),
        "dgrad_allgather_w_z": ring_time("all_gather", w_blk, gz, bw["z"]),
        "dgrad_allreduce_dx_y": ring_time("all_reduce", dx_blk, gy, bw["y"]),
        "wgrad_reducescatter_dw_z": ring_time("reduce_scatter", w_blk, gz, bw["z"]),
        "data_allreduce_dw": ring_time("all_reduce", w_blk / gz, gd, bw["data"]),
    }


def step_time(layers, tokens: int, grid, m: Machine) -> dict:
    """Predicted seconds of one training step of the FC layers.

    layers: iterable of (K, N); tokens: global batch tokens (split over
    G_data, then over G_z inside each group)."""
    gd, gx, gy, gz = grid
    T = tokens / gd
    comm = 0.0
    flops = 0.0
    for K, N in layers:
        comm += sum(layer_comm(T, K, N, grid, m).values())
        flops += 3 * 2.0 * T * K * N / (gx * gy * gz)     # fwd + dgrad + wgrad per GPU
    compute = flops / (m.gpu_tflops * 1e12)
    return {"comm": comm, "compute": compute, "total": comm + compute}


def factorizations(n: int):
    """Every (Gd, Gx, Gy, Gz) of positive integers with product n."""
    divs = [d for d in range(1, n + 1) if n % d == 0]
    for gx, gy, gz in product(divs, repeat=3):
        if n % (gx * gy * gz) == 0:
            yield (n // (gx * gy * gz), gx, gy, gz)


def rank_configs(layers, tokens: int, n_gpus: int, m: Machine):
    """All grid configurations of n_gpus, fastest predicted first."""
    out = [(step_time(layers, tokens, g, m)["total"], g) for g in factorizations(n_gpus)]
    out.sort(key=lambda t: (t[0], t[1]))
    return out
