"""Z-sharded weights on the GPU: the all-gather of row shards and the Z-group
weight gradient written as reduce-scattered shards, against the oracle."""
import numpy as np
import pytest

import fc_inputs
import oracle
from fc_cases import assert_within_bound, host_bits, host_f64, make_operand, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,G", [(1, 8, 1), (300, 520, 2), (3072, 9216, 2), (1000, 64, 4),
                                         (17, 16, 3)])
def test_shards_gather_exact(cuda_lib, rows, cols, G):
    import torch
    Wb = fc_inputs.normal_bf16((rows, cols), seed=201, tid=G)
    shards = [to_device(np.ascontiguousarray(s)) for s in oracle.shard_rows(Wb, G)]
    out = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    cuda_lib.axonn_shards_gather(shards, out, rows, cols, ld_shard=cols)
    cuda_lib.axonn_sync_status()
    assert np.array_equal(host_bits(out), oracle.gather_shards(oracle.shard_rows(Wb, G)))


def _zsharded(fc, X, dY, T, K, N, grid, xy, flags=0, f32=False):
    import torch
    Kx = oracle.split_range(K, grid[0], xy[0])
    Ny = oracle.split_range(N, grid[1], xy[1])
    Mb, Nb = Kx[1] - Kx[0], Ny[1] - Ny[0]
    ld = ((Nb + 7) // 8) * 8
    dt = torch.float32 if f32 else torch.bfloat16
    shards = []
    for z in range(grid[2]):
        r0, r1 = oracle.split_range(Mb, grid[2], z)
        shards.append(torch.full((max(r1 - r0, 1), ld), 5.0, dtype=dt, device="cuda")[: r1 - r0])
    shape = fc.Shape(T, K, N, grid, (xy[0], xy[1], 0))
    nbytes = fc.axonn_fc_workspace_size("wgrad", shape, fc.ZSHARDED)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    fc.axonn_fc_wgrad_zsharded(to_device(X), to_device(dY), shards, shape, flags, ws, ld_shard=ld)
    fc.axonn_sync_status()
    return shards


@pytest.mark.parametrize("grid,xy", [((2, 2, 2), (1, 0)), ((1, 4, 4), (0, 3)), ((3, 1, 2), (2, 0)),
                                     ((2, 3, 1), (1, 2)), ((1, 1, 3), (0, 0))])
@pytest.mark.parametrize("cfg", [-1, 1, 5])
def test_wgrad_zsharded_integer_exact(cuda_lib, grid, xy, cfg):
    T, K, N = 300, 200, 520
    X = make_operand("X", T, K, N, False, seed=203, kind="int")
    dY = make_operand("dY", T, K, N, False, seed=203, kind="int")
    cuda_lib.axonn_set_kernel_config(cfg)
    try:
        shards = _zsharded(cuda_lib, X, dY, T, K, N, grid, xy)
    finally:
        cuda_lib.axonn_set_kernel_config(-1)
    Cs, _ = oracle.wgrad_zsharded(X, dY, False, False, T, K, N, grid, xy)
    assert len(shards) == len(Cs)
    for got, want in zip(shards, Cs):
        assert np.array_equal(host_bits(got), oracle.bf16_rne(want))


def test_wgrad_zsharded_random_and_accumulate(cuda_lib):
    T, K, N = 1024, 768, 1536
    grid, xy = (2, 2, 2), (1, 1)
    X = make_operand("X", T, K, N, False, seed=205)
    dY = make_operand("dY", T, K, N, False, seed=205)
    Cs, Ss = oracle.wgrad_zsharded(X, dY, False, False, T, K, N, grid, xy)
    shards = _zsharded(cuda_lib, X, dY, T, K, N, grid, xy)
    for got, C, S in zip(shards, Cs, Ss):
        assert_within_bound(host_f64(got), C, S, "zsharded wgrad")
    # fp32 main-gradient update of the shards: shard += partial sum
    acc = _zsharded(cuda_lib, X, dY, T, K, N, grid, xy, flags=cuda_lib.ACCUM_F32, f32=True)
    for got, C, S in zip(acc, Cs, Ss):
        assert_within_bound(host_f64(got), C + 5.0, S, "zsharded wgrad accumulate")
