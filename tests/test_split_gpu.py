"""GPU parity of the reduction split: a tile's reduction cut into S pieces
(S = 2, 4, 8) computed by the S CTAs of one thread-block cluster and added
in fixed order inside it, each CTA finishing a band of 128/S rows, on
128 x 128 tiles (configuration 0) and 128 x 64 tiles (configuration 7).  Bit for
bit on integer inputs for every split, storage layout, output mode, ragged
shape, block of the grid and with the operand roles exchanged; several
tiles per cluster (the inbox reused); within the bound on random inputs.
The split needs no workspace: these calls pass none.  It is forced through
a tuning-table entry for the exact call."""
import json

import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_bits, host_f64, make_operand, operand_names,
                      run_gpu)

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]


@pytest.fixture
def force_split(cuda_lib, tmp_path):
    """Loads a tuning entry that runs (op, shape, flags) on configuration 0
    split into `split` pieces; clears the table afterwards."""
    fc = cuda_lib

    def force(op, T, K, N, flags, split, group_m=16, grid=(1, 1, 1), coords=(0, 0, 0), swap=0,
              config="1cta_128x128"):
        sms, _ = fc.axonn_device_info()
        g = "x".join(str(v) for v in grid)
        at = ".".join(str(v) for v in coords)
        key = f"op{fc.OPS[op]}_T{T}_K{K}_N{N}_g{g}_at{at}_f{flags:x}_sm{sms}"
        path = tmp_path / "split.jsonl"
        path.write_text(json.dumps({"key": key, "config": config, "split": split,
                                    "group_m": group_m, "streamk": 1, "swap": swap,
                                    "us": 1.0}) + "\n")
        fc.axonn_tune_cache_load(str(path))

    yield force
    fc.axonn_tune_cache_clear()
    fc.axonn_set_swap(-1)


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", LAYOUTS)
def test_split_integer_exact(cuda_lib, force_split, split, op, p_t, q_t):
    fc = cuda_lib
    T, K, N = 300, 1000, 520   # ragged in every dimension, 9 to 16 reduction stages
    if op == "wgrad":
        T, K, N = 1000, 300, 520
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=701, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=701, kind="int")
    flags = (fc.A_T if p_t else 0) | (fc.B_T if q_t else 0)
    force_split(op, T, K, N, flags, split)
    out = run_gpu(fc, op, P, Q, p_t, q_t, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[:2] == (0, split)
    C, _ = oracle.fc(op, P, Q, p_t, q_t)
    bad = np.argwhere(host_bits(out) != oracle.bf16_rne(C))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("group_m", [16, -8])
def test_split_many_tiles_per_cluster(cuda_lib, force_split, split, group_m):
    """256 tiles: more than the clusters resident at once for every split,
    so each cluster finishes several tiles through the same inbox."""
    fc = cuda_lib
    T, K, N = 2048, 1024, 2040
    X = make_operand("X", T, K, N, False, seed=711, kind="int")
    W = make_operand("W", T, K, N, False, seed=711, kind="int")
    force_split("fwd", T, K, N, 0, split, group_m=group_m)
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice() == (0, split, group_m)
    bad = np.argwhere(host_bits(out) != oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("mode", ["out_f32", "accum_f32"])
@pytest.mark.parametrize("split", [2, 8])
def test_split_fp32_outputs_exact(cuda_lib, force_split, mode, split):
    import torch
    fc = cuda_lib
    T, K, N = 256, 2048, 512
    dY = make_operand("dY", T, K, N, False, seed=703, kind="int")
    W = make_operand("W", T, K, N, False, seed=703, kind="int")
    C, _ = oracle.fc_dgrad(dY, W)
    if mode == "out_f32":
        force_split("dgrad", T, K, N, fc.OUT_F32, split)
        out = run_gpu(fc, "dgrad", dY, W, False, False, T, K, N, extra=fc.OUT_F32, workspace=False)
        assert np.array_equal(host_f64(out), C)
    else:
        force_split("dgrad", T, K, N, fc.ACCUM_F32, split)
        base = torch.full((T, K), -1.5, dtype=torch.float32, device="cuda")
        out = run_gpu(fc, "dgrad", dY, W, False, False, T, K, N, extra=fc.ACCUM_F32, out=base,
                      workspace=False)
        assert np.array_equal(host_f64(out), C - 1.5)
    assert fc.axonn_last_choice()[1] == split


def test_split_block_of_the_grid_exact(cuda_lib, force_split):
    """One block product of a 2x2x2 grid addressed inside the full operands,
    split in 4: its window of the fp32 output and nothing else written."""
    fc = cuda_lib
    T, K, N = 520, 1000, 776
    grid, coords = (2, 2, 2), (1, 1, 0)
    X = make_operand("X", T, K, N, False, seed=713, kind="int")
    W = make_operand("W", T, K, N, False, seed=713, kind="int")
    flags = fc.FULL_OPERANDS | fc.OUT_F32
    force_split("fwd", T, K, N, flags, 4, grid=grid, coords=coords)
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, grid=grid, coords=coords, extra=flags,
                  workspace=False)
    assert fc.axonn_last_choice()[1] == 4
    Cb, _, rows, cols = oracle.fc_block("fwd", X, W, False, False, T, K, N, grid, coords)
    got = host_f64(out)
    assert np.array_equal(got[rows[0]:rows[1], cols[0]:cols[1]], Cb)
    mask = np.ones(got.shape, bool)
    mask[rows[0]:rows[1], cols[0]:cols[1]] = False
    assert not np.any(got[mask])


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_split_with_exchanged_roles_exact(cuda_lib, force_split, op):
    fc = cuda_lib
    T, K, N = 300, 1000, 520
    if op == "wgrad":
        T, K, N = 1000, 300, 520
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=715, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=715, kind="int")
    force_split(op, T, K, N, 0, 4, swap=1)
    out = run_gpu(fc, op, P, Q, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[1] == 4 and fc.axonn_last_swap() == 1
    C, _ = oracle.fc(op, P, Q)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


def test_split_rounded_to_a_power_of_two_within_the_reduction(cuda_lib, force_split):
    """Pieces are whole 64-deep stages and the tile's rows are dealt out in
    equal bands: a request of 8 over 3 stages runs as 2."""
    fc = cuda_lib
    T, K, N = 256, 192, 512   # 3 stages
    X = make_operand("X", T, K, N, False, seed=705, kind="int")
    W = make_operand("W", T, K, N, False, seed=705, kind="int")
    force_split("fwd", T, K, N, 0, 8)
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[1] == 2
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))


@pytest.mark.parametrize("split", [4, 8])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_split_single_layer_random(cuda_lib, force_split, op, split):
    """The single FC layer (X[256x512], W[512x2048] ~N(0,0.02), dY[256x2048])
    with every product split: within the bound."""
    fc = cuda_lib
    T, K, N = 256, 512, 2048
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1001)
    Q = make_operand(qn, T, K, N, False, seed=1001)
    force_split(op, T, K, N, 0, split)
    out = run_gpu(fc, op, P, Q, False, False, T, K, N, workspace=False)
    # the weight gradient reduces over T = 256: 4 stages, at most 4 pieces
    assert fc.axonn_last_choice()[1] == (min(split, 4) if op == "wgrad" else split)
    C, S = oracle.fc(op, P, Q)
    assert_within_bound(host_f64(out), C, S, f"split {op}")


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("p_t,q_t", [(False, False), (True, True)])
def test_split_128x64_integer_exact(cuda_lib, force_split, split, op, p_t, q_t):
    """The same split on 128 x 64 tiles: bit for bit, ragged in every
    dimension."""
    fc = cuda_lib
    T, K, N = 300, 1000, 520
    if op == "wgrad":
        T, K, N = 1000, 300, 520
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, p_t, seed=721, kind="int")
    Q = make_operand(qn, T, K, N, q_t, seed=721, kind="int")
    flags = (fc.A_T if p_t else 0) | (fc.B_T if q_t else 0)
    force_split(op, T, K, N, flags, split, config="1cta_128x64")
    out = run_gpu(fc, op, P, Q, p_t, q_t, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[:2] == (7, split)
    C, _ = oracle.fc(op, P, Q, p_t, q_t)
    bad = np.argwhere(host_bits(out) != oracle.bf16_rne(C))
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("split", [2, 8])
def test_split_128x64_many_tiles_and_single_layer(cuda_lib, force_split, split):
    """128 x 64 tiles: more tiles than resident clusters (the inbox reused),
    and the single layer's data gradient within the bound."""
    fc = cuda_lib
    T, K, N = 2048, 1024, 2040
    X = make_operand("X", T, K, N, False, seed=723, kind="int")
    W = make_operand("W", T, K, N, False, seed=723, kind="int")
    force_split("fwd", T, K, N, 0, split, config="1cta_128x64")
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[:2] == (7, split)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
    T, K, N = 256, 512, 2048
    dY = make_operand("dY", T, K, N, False, seed=1001)
    Wr = make_operand("W", T, K, N, False, seed=1001)
    force_split("dgrad", T, K, N, 0, split, config="1cta_128x64")
    out = run_gpu(fc, "dgrad", dY, Wr, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[:2] == (7, split)
    C, S = oracle.fc("dgrad", dY, Wr)
    assert_within_bound(host_f64(out), C, S, "split dgrad on 128 x 64 tiles")


def test_split_not_on_other_configurations(cuda_lib, force_split):
    fc = cuda_lib
    T, K, N = 256, 2048, 512
    dY = make_operand("dY", T, K, N, False, seed=707, kind="int")
    W = make_operand("W", T, K, N, False, seed=707, kind="int")
    want = oracle.bf16_rne(oracle.fc_dgrad(dY, W)[0])
    force_split("dgrad", T, K, N, 0, 4)
    fc.axonn_set_kernel_config(5)
    try:
        out = run_gpu(fc, "dgrad", dY, W, False, False, T, K, N)
        assert fc.axonn_last_choice()[:2] == (5, 1)
        assert np.array_equal(host_bits(out), want)
    finally:
        fc.axonn_set_kernel_config(-1)


@pytest.mark.parametrize("split", [2, 8])
def test_split_bounded_wait_timeout_reports_and_recovers(cuda_lib, force_split, split):
    """A producer that withholds its loads: every CTA of every cluster times
    out in its own bounded waits (no piece ever stages its rows), all reach
    the final cluster barrier, the library reports AXONN_ERR_TIMEOUT and the
    context stays usable for a correct split product."""
    fc = cuda_lib
    T, K, N = 256, 1024, 512
    X = make_operand("X", T, K, N, False, seed=709, kind="int")
    W = make_operand("W", T, K, N, False, seed=709, kind="int")
    force_split("fwd", T, K, N, 0, split)
    try:
        fc.axonn_set_wait_timeout_ns(20_000_000)
        fc.axonn_debug_set_inject(1)
        with pytest.raises(fc.AxonnError) as ei:
            run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
        assert ei.value.status == fc.ERR_TIMEOUT
    finally:
        fc.axonn_debug_set_inject(0)
        fc.axonn_set_wait_timeout_ns(4_000_000_000)
    out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
    assert fc.axonn_last_choice()[1] == split
    assert np.array_equal(host_bits(out), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
