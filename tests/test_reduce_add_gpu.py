"""GPU parity of the order-free virtual grid (AXONN_REDUCE_ADD).

Every block product adds its tile into the fp32 output with atomic adds, in
one launch, so the order in which the G partials of the reduced axis reach
an element changes from run to run.  What stays fixed, and is checked here:

  * integer-valued operands and an integer-valued starting output keep every
    partial sum an integer below 2^24, exact in fp32 whatever the order, so
    the result must equal C0 + (the oracle's product) bit for bit;
  * random operands must satisfy, element by element,
    |C_gpu - (C0 + C)| <= 1e-2 * (S + |C0|) + 1e-5;
  * no workspace is needed, also for products whose fixed-order partials
    would not fit the library's built-in scratch.
"""
import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_f64, make_operand, operand_names, run_gpu,
                      sample_indices, to_device)

pytestmark = pytest.mark.gpu

CONFIGS = [0, 1, 2, 3, 4, 5, 6, 7]
GRIDS = [(2, 2, 2), (1, 4, 4), (3, 1, 2), (2, 3, 1)]


@pytest.fixture
def forced(cuda_lib, request):
    cfg = request.param
    cuda_lib.axonn_set_kernel_config(cfg)
    yield cfg
    cuda_lib.axonn_set_kernel_config(-1)


def _int_base(M, N, ld=None):
    """Integer-valued fp32 starting output in [-3, 3], row stride `ld`."""
    import torch
    ld = ld or ((N + 3) // 4) * 4
    base = (torch.arange(M * ld, dtype=torch.int64).reshape(M, ld) % 7 - 3).to(torch.float32)
    return base.cuda()[:, :N]


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("grid", GRIDS)
def test_reduce_add_integer_exact(cuda_lib, forced, op, grid):
    fc = cuda_lib
    T, K, N = 300, 200, 520
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=71, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=71, kind="int")
    M, Nn = fc.out_shape(op, T, K, N)
    out = _int_base(M, Nn)
    want = host_f64(out) + oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)[0]
    flags = fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD
    assert fc.axonn_fc_workspace_size(op, fc.Shape(T, K, N, grid), flags) == 0
    run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid, extra=flags, out=out)
    assert fc.axonn_last_kernel_config() == forced
    got = host_f64(out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("forced", [5, 6], indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", [(False, True), (True, False), (True, True)])
def test_reduce_add_layouts_integer_exact(cuda_lib, forced, op, p_t, q_t):
    """Transposed storage, and an output row stride wider than the row."""
    import torch
    fc = cuda_lib
    T, K, N = 520, 136, 776
    grid = (2, 2, 2)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=72, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=72, kind="int")
    M, Nn = fc.out_shape(op, T, K, N)
    ld = ((Nn + 3) // 4) * 4 + 12
    out = _int_base(M, Nn, ld)
    guard = out.as_strided((M, ld - Nn), (ld, 1), Nn)    # the columns past the row
    guard.fill_(7.0)
    want = host_f64(out) + oracle.fc(op, P, Q, p_t, q_t)[0]
    run_gpu(fc, op, P, Q, p_t, q_t, T, K, N, grid=grid,
            extra=fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD, out=out)
    assert np.array_equal(host_f64(out), want)
    assert bool(torch.all(guard == 7.0))


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_reduce_add_random_config3_shape_scaled(cuda_lib, op):
    """2x2x2 grid on an H=768, T=1024 layer, random operands and output."""
    import torch
    fc = cuda_lib
    T, K, N = 1024, 768, 3072
    grid = (2, 2, 2)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1073)
    Q = make_operand(qn, T, K, N, False, seed=1073)
    M, Nn = fc.out_shape(op, T, K, N)
    g = torch.Generator().manual_seed(73)
    base = torch.randn((M, Nn), generator=g, dtype=torch.float32)
    C, S = oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)
    b64 = base.double().numpy()
    for red in (True, False):       # order-free, then the fixed-order sum
        out = base.cuda()
        extra = fc.VGRID | fc.ACCUM_F32 | (fc.REDUCE_ADD if red else fc.VGRID_PARTIALS)
        run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid, extra=extra, out=out)
        assert_within_bound(host_f64(out), C + b64, S + np.abs(b64),
                            f"{op} {'order-free' if red else 'fixed order'}")


def test_reduce_add_repeat_and_graph(cuda_lib):
    """One launch per call and no scratch: repeated calls and graph replays
    keep adding, C = C0 + k * product, exact on integer operands."""
    import torch
    fc = cuda_lib
    T, K, N = 300, 200, 520
    grid = (1, 4, 4)
    X = make_operand("X", T, K, N, False, seed=74, kind="int")
    dY = make_operand("dY", T, K, N, False, seed=74, kind="int")
    C, _ = oracle.fc_wgrad(X, dY)
    out = _int_base(K, N)
    c0 = host_f64(out)
    Xd, dYd = to_device(X), to_device(dY)
    shape = fc.Shape(T, K, N, grid)
    flags = fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD
    for _ in range(3):
        fc.call("wgrad", Xd, dYd, out, shape, flags, None)
    fc.axonn_sync_status()
    assert np.array_equal(host_f64(out), c0 + 3 * C)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            fc.call("wgrad", Xd, dYd, out, shape, flags, None, stream=s)
        for _ in range(4):
            gr.replay()
    torch.cuda.synchronize()
    fc.axonn_sync_status(s)
    # 3 calls and 4 replays; the capture itself runs nothing
    assert np.array_equal(host_f64(out), c0 + 7 * C)


def test_reduce_add_static_entry_point_needs_no_scratch(cuda_lib):
    """A product whose fixed-order partial (one slot of 4096 x 8192 fp32 =
    128 MiB on a 2x1x1 grid) exceeds the built-in 64 MiB scratch: refused in
    the two-launch form (AXONN_VGRID_PARTIALS), exact with AXONN_REDUCE_ADD
    and in the chained form, which need no scratch."""
    import torch
    fc = cuda_lib
    T, K, N = 4096, 64, 8192
    grid = (2, 1, 1)
    X = make_operand("X", T, K, N, False, seed=75, kind="int")
    W = make_operand("W", T, K, N, False, seed=75, kind="int")
    Xd, Wd = to_device(X), to_device(W)
    out = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    shape = fc.Shape(T, K, N, grid)
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_fc_vgrid_static("fwd", Xd, Wd, out, shape, fc.ACCUM_F32 | fc.VGRID_PARTIALS)
    assert ei.value.status == fc.ERR_WORKSPACE
    fc.axonn_fc_vgrid_static("fwd", Xd, Wd, out, shape, fc.ACCUM_F32 | fc.REDUCE_ADD)
    fc.axonn_sync_status()
    I, J = sample_indices(T, N, 75)
    got = host_f64(out[torch.from_numpy(I).cuda(), torch.from_numpy(J).cuda()])
    C, _ = oracle.fc_entries("fwd", X, W, False, False, I, J)
    assert np.array_equal(got, C)
    fc.axonn_fc_vgrid_static("fwd", Xd, Wd, out, shape, fc.ACCUM_F32)   # chained: adds again
    fc.axonn_sync_status()
    got = host_f64(out[torch.from_numpy(I).cuda(), torch.from_numpy(J).cuda()])
    assert np.array_equal(got, 2 * C)


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_reduce_add_gpt_block_up_2x2x2_full_size(cuda_lib, op):
    """The MLP-up layer of the H=6144, T=8192 block as a 2x2x2 grid at full
    size, in the library's own kernel choice; sampled entries against the
    oracle, starting output zero."""
    import torch
    import fc_inputs
    fc = cuda_lib
    T, K, N = 8192, 6144, 24576
    grid = (2, 2, 2)
    X = fc_inputs.normal_bf16((T, K), 1002, 48 + 1, sigma=1.0)
    W = fc_inputs.normal_bf16((K, N), 1002, 48 + 2, sigma=0.02)
    dY = fc_inputs.normal_bf16((T, N), 1002, 48 + 3, sigma=1.0)
    P, Q = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (X, dY)}[op]
    Pd, Qd = fc_inputs.as_torch_bf16(P, "cuda"), fc_inputs.as_torch_bf16(Q, "cuda")
    M, Nn = fc.out_shape(op, T, K, N)
    out = torch.zeros((M, Nn), dtype=torch.float32, device="cuda")
    fc.call(op, Pd, Qd, out, fc.Shape(T, K, N, grid),
            fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD, None)
    fc.axonn_sync_status()
    del Pd, Qd
    I, J = sample_indices(M, Nn, 76, n_random=32768)
    got = host_f64(out[torch.from_numpy(I).cuda(), torch.from_numpy(J).cuda()])
    del out
    torch.cuda.empty_cache()
    C, S = oracle.fc_entries(op, P, Q, False, False, I, J)
    assert_within_bound(got, C, S, f"order-free 2x2x2 up {op}")


def test_reduce_add_tune_then_call(cuda_lib):
    """The tuner times the order-free call as it runs (adding into a scratch
    output); the tuned choice is then used and stays exact."""
    import torch
    fc = cuda_lib
    T, K, N = 300, 200, 520
    grid = (2, 2, 2)
    X = make_operand("X", T, K, N, False, seed=77, kind="int")
    W = make_operand("W", T, K, N, False, seed=77, kind="int")
    Xd, Wd = to_device(X), to_device(W)
    shape = fc.Shape(T, K, N, grid)
    flags = fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD
    scratch = torch.zeros((T, N), dtype=torch.float32, device="cuda")
    try:
        cfg, _, _, us = fc.axonn_fc_tune("fwd", Xd, Wd, scratch, shape, flags, None)
        assert 0 <= cfg < fc.axonn_num_kernel_configs() and us > 0
        out = _int_base(T, N)
        want = host_f64(out) + oracle.fc_fwd(X, W)[0]
        fc.call("fwd", Xd, Wd, out, shape, flags, None)
        fc.axonn_sync_status()
        assert fc.axonn_last_kernel_config() == cfg
        assert np.array_equal(host_f64(out), want)
    finally:
        fc.axonn_tune_cache_clear()
