"""Multi-process checks on CPU (gloo, world size 2).

* The 3D grid across ranks: each rank owns the blocks whose coordinate on
  the op's reduced axis equals its rank, computes their partial products
  (fp64 oracle), and an all-reduce over the group sums them -- the
  collective that the virtual grid replaces on one GPU.  The sum must equal
  the full product exactly for integer-valued operands.
* Z-sharded weights across ranks: rank z of a Z group holds row shard z of
  the weight block; an all-gather over the group rebuilds the block, and the
  weight-gradient partials are reduce-scattered into the shards.  Both must
  match the oracle's sharded forms exactly for integer-valued operands.
* The benchmark's cross-rank timing: the reported time is the slowest
  rank's.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grid_worker(rank, world, port, op, grid, out_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import fc_inputs
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, K, N = 72, 40, 56
        X = fc_inputs.small_int_bf16((T, K), 5, 1, h=2)
        W = fc_inputs.small_int_bf16((K, N), 5, 2, h=2)
        dY = fc_inputs.small_int_bf16((T, N), 5, 3, h=2)
        P, Q = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (X, dY)}[op]
        axis = oracle.reduce_axis(op)
        gx, gy, gz = grid
        local = np.zeros(oracle.out_shape(op, T, K, N), dtype=np.float64)
        for x in range(gx):
            for y in range(gy):
                for z in range(gz):
                    if {"x": x, "y": y, "z": z}[axis] % world != rank:
                        continue
                    Cb, _, rows, cols = oracle.fc_block(op, P, Q, False, False, T, K, N, grid,
                                                        (x, y, z))
                    local[rows[0]:rows[1], cols[0]:cols[1]] += Cb
        t = torch.from_numpy(local)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            full, _ = oracle.fc(op, P, Q)
            out_q.put(bool(np.array_equal(t.numpy(), full)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("op,grid", [("fwd", (2, 1, 1)), ("dgrad", (1, 2, 1)),
                                     ("wgrad", (1, 1, 2)), ("fwd", (2, 2, 2)),
                                     ("wgrad", (1, 4, 4))])
def test_grid_partials_allreduce_to_full_product(op, grid):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_grid_worker, args=(r, 2, port, op, grid, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) is True


def _zshard_worker(rank, world, port, grid, xy, out_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import fc_inputs
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, K, N = 72, 40, 56
        gx, gy, gz = grid
        x, y = xy
        z = rank                                   # this rank's place in the Z group
        X = fc_inputs.small_int_bf16((T, K), 6, 1, h=2)
        W = fc_inputs.small_int_bf16((K, N), 6, 2, h=2)
        dY = fc_inputs.small_int_bf16((T, N), 6, 3, h=2)
        Kx, Ny = oracle.split_range(K, gx, x), oracle.split_range(N, gy, y)
        Wblk = W[Kx[0]:Kx[1], Ny[0]:Ny[1]]
        shards = oracle.shard_rows(Wblk, gz)
        # all-gather (gloo wants equal sizes: pad each shard to the largest)
        rows = max(sh.shape[0] for sh in shards)
        mine = np.zeros((rows, Wblk.shape[1]), dtype=np.int32)
        mine[:shards[z].shape[0]] = shards[z].astype(np.int32)
        parts = [torch.zeros_like(torch.from_numpy(mine)) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(mine))
        got = np.concatenate([parts[r].numpy()[:shards[r].shape[0]] for r in range(world)])
        gather_ok = np.array_equal(got.astype(np.uint16), oracle.gather_shards(shards))
        # weight gradient: this rank's partial, then the reduce-scatter (gloo
        # has no reduce-scatter: an all-reduce and keeping one's own shard
        # gives the same shard)
        Cb, _, _, _ = oracle.fc_block("wgrad", X, dY, False, False, T, K, N, grid, (x, y, z))
        t = torch.from_numpy(np.ascontiguousarray(Cb))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        r0, r1 = oracle.split_range(Cb.shape[0], gz, z)
        want, _ = oracle.wgrad_zsharded(X, dY, False, False, T, K, N, grid, xy)
        rs_ok = np.array_equal(t.numpy()[r0:r1], want[z])
        out_q.put((rank, bool(gather_ok), bool(rs_ok)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("grid,xy", [((1, 1, 2), (0, 0)), ((2, 2, 2), (1, 0)),
                                     ((2, 3, 2), (0, 2))])
def test_zsharded_gather_and_reduce_scatter_across_ranks(grid, xy):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_zshard_worker, args=(r, 2, port, grid, xy, q))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, True, True), (1, True, True)]


def _timing_worker(rank, world, port, out_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out_q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")))
    finally:
        dist.destroy_process_group()


def test_bench_reports_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_timing_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_group():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
