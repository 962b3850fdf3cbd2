"""GPU parity of the exchanged operand roles (C^T = B^T . A^T with a
transposing epilogue) against the fp64 oracle: bit for bit on integer
inputs in every storage layout, kernel configuration, output mode, virtual
grid form and with the stream-K tail; within the bound on random inputs;
and the tuner's swap candidates."""
import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_bits, host_f64, make_operand, operand_names,
                      run_gpu)

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]


@pytest.fixture
def swapped(cuda_lib):
    cuda_lib.axonn_set_swap(1)
    yield
    cuda_lib.axonn_set_swap(-1)
    cuda_lib.axonn_set_kernel_config(-1)
    cuda_lib.axonn_set_streamk(-1)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", LAYOUTS)
@pytest.mark.parametrize("T,K,N", [(300, 200, 520), (129, 1000, 257), (520, 136, 776)])
def test_swap_integer_exact(cuda_lib, swapped, cfg, op, p_t, q_t, T, K, N):
    cuda_lib.axonn_set_kernel_config(cfg)
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=501, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=501, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, p_t, q_t, T, K, N, workspace=False)
    assert cuda_lib.axonn_last_swap() == 1
    C, _ = oracle.fc(op, P, Q, p_t, q_t)
    bad = np.argwhere(host_bits(out) != oracle.bf16_rne(C))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("cfg", [1, 5, 6])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("grid", [(2, 2, 2), (3, 1, 2), (1, 4, 4)])
def test_swap_chained_vgrid_exact(cuda_lib, swapped, cfg, op, grid):
    cuda_lib.axonn_set_kernel_config(cfg)
    T, K, N = 520, 384, 776
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=503, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=503, kind="int")
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N, grid=grid, extra=cuda_lib.VGRID)
    assert cuda_lib.axonn_last_swap() == 1
    C, _ = oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


@pytest.mark.parametrize("mode", ["out_f32", "accum_f32", "block", "reduce_add"])
def test_swap_output_modes_exact(cuda_lib, swapped, mode):
    import torch
    fc = cuda_lib
    T, K, N = 300, 200, 520
    X = make_operand("X", T, K, N, False, seed=505, kind="int")
    W = make_operand("W", T, K, N, False, seed=505, kind="int")
    C, _ = oracle.fc_fwd(X, W)
    if mode == "out_f32":
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, extra=fc.OUT_F32, workspace=False)
        assert np.array_equal(host_f64(out), C)
    elif mode == "accum_f32":
        base = torch.full((T, N), 2.0, dtype=torch.float32, device="cuda")
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, extra=fc.ACCUM_F32, out=base,
                      workspace=False)
        assert np.array_equal(host_f64(out), C + 2.0)
    elif mode == "block":
        grid, coords = (2, 2, 2), (1, 1, 0)
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, grid=grid, coords=coords,
                      extra=fc.FULL_OPERANDS | fc.OUT_F32, workspace=False)
        Cb, _, rows, cols = oracle.fc_block("fwd", X, W, False, False, T, K, N, grid, coords)
        got = host_f64(out)
        assert np.array_equal(got[rows[0]:rows[1], cols[0]:cols[1]], Cb)
        mask = np.ones(got.shape, bool)
        mask[rows[0]:rows[1], cols[0]:cols[1]] = False
        assert not np.any(got[mask])
    else:
        base = torch.zeros((T, N), dtype=torch.float32, device="cuda")
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, grid=(2, 2, 2),
                      extra=fc.VGRID | fc.ACCUM_F32 | fc.REDUCE_ADD, out=base)
        assert np.array_equal(host_f64(out), C)
    assert fc.axonn_last_swap() == 1


@pytest.mark.parametrize("cfg", [1, 5, 6])
@pytest.mark.parametrize("op", ["fwd", "wgrad"])
def test_swap_with_streamk_tail_exact(cuda_lib, swapped, cfg, op):
    """Enough tiles for more than one round of the persistent grid, with the
    tail forced on: the pieces' partial slots stay in the problem's own
    orientation and only the final store is transposed."""
    fc = cuda_lib
    fc.axonn_set_kernel_config(cfg)
    fc.axonn_set_streamk(1)
    T, K, N = 2600, 2600, 4200   # more tiles than one round in every configuration
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=507, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=507, kind="int")
    out = run_gpu(fc, op, P, Q, False, False, T, K, N)
    assert fc.axonn_last_swap() == 1 and fc.axonn_last_streamk_tiles() > 0
    C, _ = oracle.fc(op, P, Q)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


def test_swap_not_applied_to_partials_but_to_split(cuda_lib, swapped):
    fc = cuda_lib
    T, K, N = 300, 200, 520
    X = make_operand("X", T, K, N, False, seed=509, kind="int")
    W = make_operand("W", T, K, N, False, seed=509, kind="int")
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, grid=(2, 2, 2),
                  extra=fc.VGRID | fc.VGRID_PARTIALS)
    assert fc.axonn_last_swap() == 0
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
    # a small product whose reduction (33 stages) the default choice splits:
    # the split's epilogue stores the transposed band
    N = 2100
    dY = make_operand("dY", T, K, N, False, seed=509, kind="int")
    W = make_operand("W", T, K, N, False, seed=509, kind="int")
    out = run_gpu(fc, "dgrad", dY, W, False, False, T, K, N)
    assert fc.axonn_last_choice()[1] > 1 and fc.axonn_last_swap() == 1
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_dgrad(dY, W)[0]))


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_swap_random_within_bound(cuda_lib, swapped, op):
    T, K, N = 1000, 1000, 5000
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1005, scale=0.05)
    Q = make_operand(qn, T, K, N, False, seed=1005, scale=0.05)
    out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N, workspace=False)
    assert cuda_lib.axonn_last_swap() == 1
    C, S = oracle.fc(op, P, Q)
    assert_within_bound(host_f64(out), C, S, f"swapped {op}")


def test_tuner_times_the_swap_and_keeps_parity(cuda_lib):
    """The tuner's choice (swapped or not) is recorded, saved with the swap
    field, reloaded, and the tuned call stays exact."""
    import json
    import os
    import tempfile

    import torch
    from fc_cases import to_device
    fc = cuda_lib
    fc.axonn_tune_cache_clear()
    T, K, N = 512, 5000, 1000
    X = make_operand("X", T, K, N, False, seed=511, kind="int")
    W = make_operand("W", T, K, N, False, seed=511, kind="int")
    Xd, Wd = to_device(X), to_device(W)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    shape = fc.Shape(T, K, N)
    nbytes = fc.axonn_fc_workspace_size("fwd", shape, 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    try:
        fc.axonn_fc_tune("fwd", Xd, Wd, out, shape, 0, ws)
        path = os.path.join(tempfile.mkdtemp(), "tune.jsonl")
        fc.axonn_tune_cache_save(path)
        entry = json.loads(open(path).read().splitlines()[0])
        assert entry["swap"] in (0, 1)
        fc.axonn_tune_cache_clear()
        fc.axonn_tune_cache_load(path)
        out.zero_()
        fc.axonn_fc_fwd(Xd, Wd, out, shape, 0, ws)
        fc.axonn_sync_status()
        assert fc.axonn_last_swap() == entry["swap"]
        assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
    finally:
        fc.axonn_tune_cache_clear()
