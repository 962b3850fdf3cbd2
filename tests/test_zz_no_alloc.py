"""The virtual-grid entry point that allocates nothing.

Some callers cannot call cudaMalloc: code running inside a host framework
that hands out all device memory itself, or code that must not allocate
once it is running.  They use axonn_fc_vgrid_static, which keeps the fp32
partials of the grid's reduced axis in a fixed scratch array inside the
library instead of a caller workspace.

The scratch holds the partials of the two-launch form of the grid's sum
(AXONN_VGRID_PARTIALS); the default form, which chains a tile's block
products in one accumulator, needs none.  What is checked, through the C
ABI, on two calls in a row of the two-launch form (the second smaller than
the first, so partials the first call left in the shared scratch would show
if the second one read them):

* integer-valued inputs: the output is bit for bit the oracle's exact
  product rounded once to bf16, and bit for bit the workspace entry
  point's output;
* random inputs: bit for bit the workspace entry point's output (both run
  the same fixed-order kernels) and within the bound
  |C - C_ref| <= 1e-2 * (|A|.|B|) + 1e-5 of the oracle's C;
* the size limit: partials of exactly the scratch size run, one more row
  of 8 columns is refused with AXONN_ERR_WORKSPACE;
* the default chained form through the same entry point: bit for bit the
  workspace entry point's output and the oracle's exact product.

This file is collected last so that a failure here stops a -x run only after
every other test has run.
"""
import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_bits, host_f64, make_operand, operand_names,
                      run_gpu, to_device)

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _static_call(fc, op, P, Q, T, K, N, grid, flags=0):
    import torch
    Pd, Qd = to_device(P), to_device(Q)
    M, Nn = fc.out_shape(op, T, K, N)
    ld = ((Nn + 7) // 8) * 8
    out = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :Nn]
    fc.axonn_fc_vgrid_static(op, Pd, Qd, out, fc.Shape(T, K, N, grid), flags)
    fc.axonn_sync_status()
    return out


CASES = ((91, (520, 384, 640)), (92, (300, 200, 264)))


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_static_scratch_exact_on_integer_inputs(cuda_lib, op):
    fc = cuda_lib
    grid = (2, 2, 2)
    for seed, (T, K, N) in CASES:
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=seed, kind="int")
        Q = make_operand(qn, T, K, N, False, seed=seed, kind="int")
        got = host_bits(_static_call(fc, op, P, Q, T, K, N, grid, fc.VGRID_PARTIALS))
        C, _ = oracle.fc(op, P, Q)
        assert np.array_equal(got, oracle.bf16_rne(C)), f"static-scratch {op} {T}x{K}x{N}"
        ws = host_bits(run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid,
                               extra=fc.VGRID | fc.VGRID_PARTIALS))
        assert np.array_equal(got, ws)


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_static_scratch_matches_workspace_entry_point(cuda_lib, op):
    fc = cuda_lib
    grid = (2, 2, 2)
    for seed, (T, K, N) in CASES:
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=seed)
        Q = make_operand(qn, T, K, N, False, seed=seed)
        out = _static_call(fc, op, P, Q, T, K, N, grid, fc.VGRID_PARTIALS)
        ws = run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid,
                     extra=fc.VGRID | fc.VGRID_PARTIALS)
        assert np.array_equal(host_bits(out), host_bits(ws)), f"{op} {T}x{K}x{N}"
        C, S = oracle.fc(op, P, Q)
        assert_within_bound(host_f64(out), C, S, f"static-scratch {op} {T}x{K}x{N}")


def test_static_scratch_size_limit(cuda_lib):
    """A 2x1x1 forward grid keeps one fp32 partial of M x ceil8(N): 4096 x
    4096 fills the 64 MiB exactly and runs; 4096 x 4104 is refused."""
    fc = cuda_lib
    T, K, N = 4096, 24, 4096
    assert (T * N * 4) == SCRATCH_BYTES
    X = make_operand("X", T, K, N, False, seed=93, kind="int")
    W = make_operand("W", T, K, N, False, seed=93, kind="int")
    got = host_bits(_static_call(fc, "fwd", X, W, T, K, N, (2, 1, 1), fc.VGRID_PARTIALS))
    C, _ = oracle.fc("fwd", X, W)
    assert np.array_equal(got, oracle.bf16_rne(C))
    shape = fc.Shape(T, K, N + 8, (2, 1, 1))
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_fc_vgrid_static("fwd", 1 << 20, 1 << 20, 1 << 20, shape, fc.VGRID_PARTIALS,
                                 ldp=K, ldq=N + 8, ldc=N + 8)
    assert ei.value.status == fc.ERR_WORKSPACE
    assert "scratch" in str(ei.value)


def test_static_scratch_rejects_oversize(cuda_lib):
    fc = cuda_lib
    shape = fc.Shape(8192, 6144, 24576, (2, 2, 2))   # needs 0.8 GB of partials
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_fc_vgrid_static("fwd", 1 << 20, 1 << 20, 1 << 20, shape, fc.VGRID_PARTIALS,
                                 ldp=6144, ldq=24576, ldc=24576)
    assert ei.value.status == fc.ERR_WORKSPACE
    assert "scratch" in str(ei.value)


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_static_entry_point_chained_form(cuda_lib, op):
    """Without AXONN_VGRID_PARTIALS the entry point runs the chained sum,
    which keeps partials in TMEM and touches no scratch."""
    fc = cuda_lib
    grid = (2, 2, 2)
    for seed, (T, K, N) in CASES:
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=seed, kind="int")
        Q = make_operand(qn, T, K, N, False, seed=seed, kind="int")
        got = host_bits(_static_call(fc, op, P, Q, T, K, N, grid))
        C, _ = oracle.fc(op, P, Q)
        assert np.array_equal(got, oracle.bf16_rne(C))
        ws = host_bits(run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid, extra=fc.VGRID))
        assert np.array_equal(got, ws)
