"""GPU parity: the tcgen05 path through the C ABI against the fp64 oracle.

Exact-arithmetic cases (small-integer operands) must match bit for bit:
fp32 sums of integers below 2^24 are exact, and both sides round the same
integer to bf16 with ties to even.  Random cases must satisfy, element by
element, |C_gpu - C| <= 1e-2 * (|A|.|B|) + 1e-5.
"""
import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_bits, host_f64, make_operand, operand_names,
                      run_gpu)

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]
CONFIGS = [0, 1, 2, 3, 4, 5, 6, 7]   # every kernel configuration of the library


@pytest.fixture
def forced(cuda_lib, request):
    """Force one kernel configuration for the test, restore automatic after."""
    cfg = request.param
    cuda_lib.axonn_set_kernel_config(cfg)
    yield cfg
    cuda_lib.axonn_set_kernel_config(-1)


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", LAYOUTS)
@pytest.mark.parametrize("T,K,N", [(128, 64, 256), (300, 200, 520), (129, 1000, 257),
                                   (520, 136, 776), (384, 200, 448), (320, 448, 200)])
def test_integer_exact_layouts_and_tails(cuda_lib, forced, op, p_t, q_t, T, K, N):
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=21, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=21, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, p_t, q_t, T, K, N)
    assert cuda_lib.axonn_last_kernel_config() == forced
    C, _ = oracle.fc(op, P, Q, p_t, q_t)
    want = oracle.bf16_rne(C)
    got = host_bits(out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_config1_single_layer_random(cuda_lib, forced, op):
    """X[256x512] ~N(0,1), W[512x2048] ~N(0,0.02), dY[256x2048] ~N(0,1)."""
    T, K, N = 256, 512, 2048
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1001)
    Q = make_operand(qn, T, K, N, False, seed=1001)
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N)
    C, S = oracle.fc(op, P, Q)
    assert_within_bound(host_f64(out), C, S, f"config1 {op}")


# The virtual grid's two fixed-order sums: the G block products of a tile
# chained into one accumulator (default), or fp32 partials in the workspace
# summed in the last block's epilogue (AXONN_VGRID_PARTIALS).
FORMS = ["chained", "partials"]


def _vgrid_flags(fc, form):
    return fc.VGRID | (fc.VGRID_PARTIALS if form == "partials" else 0)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("grid", [(2, 2, 2), (1, 4, 4), (3, 1, 2), (2, 3, 1)])
def test_vgrid_integer_exact(cuda_lib, forced, op, grid, form):
    T, K, N = 300, 200, 520
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=31, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=31, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N, grid=grid,
                  extra=_vgrid_flags(cuda_lib, form))
    C, _ = oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


@pytest.mark.parametrize("forced", [1, 2, 5, 6], indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", LAYOUTS)
@pytest.mark.parametrize("grid,TKN", [((2, 2, 2), (520, 384, 776)), ((3, 1, 2), (300, 1000, 257)),
                                      ((1, 4, 4), (1024, 200, 640)), ((4, 2, 1), (129, 1000, 520))])
def test_vgrid_chain_layouts_and_ragged_blocks(cuda_lib, forced, op, p_t, q_t, grid, TKN):
    """Chained block products in every storage layout, with block extents
    that are not tile multiples (so every member's tensor maps zero-fill at
    its own edges) and members of unequal reduction length: bitwise."""
    T, K, N = TKN
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=33, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=33, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, p_t, q_t, T, K, N, grid=grid, extra=cuda_lib.VGRID)
    assert cuda_lib.axonn_last_kernel_config() == forced
    C, _ = oracle.fc_vgrid(op, P, Q, p_t, q_t, T, K, N, grid)
    bad = np.argwhere(host_bits(out) != oracle.bf16_rne(C))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def test_vgrid_chained_needs_no_workspace(cuda_lib):
    """The chained sum keeps the partials in TMEM: no workspace is asked for
    or passed, and the result is exact."""
    fc = cuda_lib
    T, K, N = 300, 200, 520
    for op in ("fwd", "dgrad", "wgrad"):
        assert fc.axonn_fc_workspace_size(op, fc.Shape(T, K, N, (2, 2, 2)), fc.VGRID) == 0
        assert fc.axonn_fc_workspace_size(op, fc.Shape(T, K, N, (2, 2, 2)),
                                          fc.VGRID | fc.VGRID_PARTIALS) > 0
    X = make_operand("X", T, K, N, False, seed=35, kind="int")
    W = make_operand("W", T, K, N, False, seed=35, kind="int")
    import torch
    from fc_cases import to_device
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    fc.axonn_fc_fwd(to_device(X), to_device(W), out, fc.Shape(T, K, N, (4, 1, 1)), fc.VGRID, None)
    fc.axonn_sync_status()
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_vgrid_random_config3_shape_scaled(cuda_lib, op, form):
    """2x2x2 grid on an H=768, T=1024 layer (config-3 structure, scaled)."""
    T, K, N = 1024, 768, 3072
    grid = (2, 2, 2)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1003)
    Q = make_operand(qn, T, K, N, False, seed=1003)
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N, grid=grid,
                  extra=_vgrid_flags(cuda_lib, form))
    C, S = oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)
    assert_within_bound(host_f64(out), C, S, f"vgrid {op} {form}")


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("coords", [(0, 0, 0), (1, 0, 1), (1, 1, 1)])
def test_block_full_operands(cuda_lib, forced, op, coords):
    """One block product addressed inside the full matrices; fp32 partial."""
    T, K, N = 300, 200, 520
    grid = (2, 2, 2)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=41, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=41, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N, grid=grid, coords=coords,
                  extra=cuda_lib.FULL_OPERANDS | cuda_lib.OUT_F32)
    Cb, _, rows, cols = oracle.fc_block(op, P, Q, False, False, T, K, N, grid, coords)
    got = host_f64(out)
    assert np.array_equal(got[rows[0]:rows[1], cols[0]:cols[1]], Cb)
    # nothing outside the block was written
    mask = np.ones(got.shape, bool)
    mask[rows[0]:rows[1], cols[0]:cols[1]] = False
    assert not np.any(got[mask])


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_block_local_shards(cuda_lib, op):
    """Pointers address the block's own shards (what one rank holds)."""
    T, K, N = 300, 200, 520
    grid, coords = (2, 2, 2), (1, 0, 1)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=43)
    Q = make_operand(qn, T, K, N, False, seed=43)
    Tz = oracle.split_range(T, grid[2], coords[2])
    Kx = oracle.split_range(K, grid[0], coords[0])
    Ny = oracle.split_range(N, grid[1], coords[1])
    rng = {"X": (Tz, Kx), "W": (Kx, Ny), "dY": (Tz, Ny)}
    Pl = np.ascontiguousarray(P[slice(*rng[pn][0]), slice(*rng[pn][1])])
    Ql = np.ascontiguousarray(Q[slice(*rng[qn][0]), slice(*rng[qn][1])])
    Cb, Sb, rows, cols = oracle.fc_block(op, P, Q, False, False, T, K, N, grid, coords)
    out = run_gpu(cuda_lib, op, Pl, Ql, False, False, T, K, N, grid=grid, coords=coords,
                  local_shape=Cb.shape)
    assert_within_bound(host_f64(out), Cb, Sb, f"local block {op}")


def test_wgrad_accumulate_f32(cuda_lib):
    import torch
    T, K, N = 256, 192, 320
    X = make_operand("X", T, K, N, False, seed=51, kind="int")
    dY = make_operand("dY", T, K, N, False, seed=51, kind="int")
    C0 = torch.arange(K * N, dtype=torch.float32, device="cuda").reshape(K, N) * 0.5
    out = C0.clone()
    run_gpu(cuda_lib, "wgrad", X, dY, False, False, T, K, N, extra=cuda_lib.ACCUM_F32, out=out)
    C, _ = oracle.fc_wgrad(X, dY)
    assert np.array_equal(host_f64(out), host_f64(C0) + C)


@pytest.mark.parametrize("form", FORMS)
def test_vgrid_accumulate_f32(cuda_lib, form):
    import torch
    T, K, N = 300, 200, 520
    X = make_operand("X", T, K, N, False, seed=53, kind="int")
    W = make_operand("W", T, K, N, False, seed=53, kind="int")
    out = torch.full((T, N), 3.0, dtype=torch.float32, device="cuda")
    run_gpu(cuda_lib, "fwd", X, W, False, False, T, K, N, grid=(2, 2, 2),
            extra=_vgrid_flags(cuda_lib, form) | cuda_lib.ACCUM_F32, out=out)
    C, _ = oracle.fc_fwd(X, W)
    assert np.array_equal(host_f64(out), C + 3.0)


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("T,K,N", [(1, 1, 1), (7, 9, 5), (1, 300, 1), (513, 8, 3)])
def test_degenerate_small_shapes(cuda_lib, forced, T, K, N):
    for op in ("fwd", "dgrad", "wgrad"):
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=61, kind="int", pad=True)
        Q = make_operand(qn, T, K, N, False, seed=61, kind="int", pad=True)
        out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N)
        C, _ = oracle.fc(op, P, Q)
        assert np.array_equal(host_bits(out), oracle.bf16_rne(C)), op


def test_empty_reduction_writes_zeros(cuda_lib):
    import torch
    T, N = 64, 40
    out = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    Xd = torch.empty((T, 8), dtype=torch.bfloat16, device="cuda")
    Wd = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")[:0]
    cuda_lib.axonn_fc_fwd(Xd, Wd, out, cuda_lib.Shape(T, 0, N), 0, ldx=8, ldw=40)
    cuda_lib.axonn_sync_status()
    assert torch.count_nonzero(out).item() == 0


def test_empty_reduction_leaves_accumulated_output_unchanged(cuda_lib):
    """K = 0 with an accumulating fp32 output adds nothing: every bit stays,
    a subnormal and a negative zero included."""
    import torch
    T, N = 64, 40
    out = torch.randn((T, N), generator=torch.Generator().manual_seed(9)).cuda()
    out[0, 0] = 1e-40            # subnormal in fp32
    out[1, 1] = -0.0
    before = out.clone()
    Xd = torch.empty((T, 8), dtype=torch.bfloat16, device="cuda")
    Wd = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")[:0]
    cuda_lib.axonn_fc_fwd(Xd, Wd, out, cuda_lib.Shape(T, 0, N), cuda_lib.ACCUM_F32, ldx=8, ldw=40)
    cuda_lib.axonn_sync_status()
    assert torch.equal(out.view(torch.int32), before.view(torch.int32))


def test_empty_output_is_noop(cuda_lib):
    import torch
    out = torch.full((4, 8), 5.0, dtype=torch.bfloat16, device="cuda")
    X = torch.ones((0, 16), dtype=torch.bfloat16, device="cuda")
    W = torch.ones((16, 8), dtype=torch.bfloat16, device="cuda")
    cuda_lib.axonn_fc_fwd(X, W, out, cuda_lib.Shape(0, 16, 8), 0, ldx=16, ldw=8, ldy=8)
    cuda_lib.axonn_sync_status()
    assert torch.all(out == 5.0)


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
def test_bounded_wait_timeout_reports_and_recovers(cuda_lib, forced):
    """A producer that withholds its loads makes every bounded wait expire;
    the library reports AXONN_ERR_TIMEOUT and the context stays usable."""
    T, K, N = 128, 64, 256
    X = make_operand("X", T, K, N, False, seed=71, kind="int")
    W = make_operand("W", T, K, N, False, seed=71, kind="int")
    try:
        cuda_lib.axonn_set_wait_timeout_ns(20_000_000)
        cuda_lib.axonn_debug_set_inject(1)
        with pytest.raises(cuda_lib.AxonnError) as ei:
            run_gpu(cuda_lib, "fwd", X, W, False, False, T, K, N)
        assert ei.value.status == cuda_lib.ERR_TIMEOUT
    finally:
        cuda_lib.axonn_debug_set_inject(0)
        cuda_lib.axonn_set_wait_timeout_ns(4_000_000_000)
    out = run_gpu(cuda_lib, "fwd", X, W, False, False, T, K, N)
    C, _ = oracle.fc_fwd(X, W)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))
