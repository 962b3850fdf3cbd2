"""The virtual-grid entry point that allocates nothing.

Callers that cannot call cudaMalloc (code inside a host framework that owns
all device memory, or code that must not allocate once running) use
axonn_fc_vgrid_static, which keeps its fp32 partials in a fixed scratch array
inside the library.  Its results must agree with the workspace entry point's
within the tests' bound |C - C_ref| <= 1e-2 * (|A|.|B|) + 1e-5, on two calls
in a row: the second call is smaller than the first, so partials left in the
shared scratch by the first call would show if the second one read them.

This file is collected last so that a failure here stops a -x run only after
every other test has run.
"""
import numpy as np
import pytest

import oracle
from fc_cases import assert_within_bound, host_f64, make_operand, operand_names, run_gpu

pytestmark = pytest.mark.gpu


def _static_call(fc, op, P, Q, T, K, N, grid):
    import torch
    from fc_cases import to_device
    Pd, Qd = to_device(P), to_device(Q)
    M, Nn = fc.out_shape(op, T, K, N)
    ld = ((Nn + 7) // 8) * 8
    out = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :Nn]
    fc.axonn_fc_vgrid_static(op, Pd, Qd, out, fc.Shape(T, K, N, grid))
    fc.axonn_sync_status()
    return out


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_static_scratch_matches_workspace_entry_point(cuda_lib, op):
    fc = cuda_lib
    grid = (2, 2, 2)
    for seed, (T, K, N) in ((91, (520, 384, 640)), (92, (300, 200, 264))):
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=seed)
        Q = make_operand(qn, T, K, N, False, seed=seed)
        got = host_f64(_static_call(fc, op, P, Q, T, K, N, grid))
        ref = host_f64(run_gpu(fc, op, P, Q, False, False, T, K, N, grid=grid, extra=fc.VGRID))
        _, S = oracle.fc(op, P, Q)
        assert_within_bound(got, ref, S, f"static-scratch {op} {T}x{K}x{N}")


def test_static_scratch_rejects_oversize(cuda_lib):
    fc = cuda_lib
    shape = fc.Shape(8192, 6144, 24576, (2, 2, 2))   # needs 1.6 GB of partials
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_fc_vgrid_static("fwd", 1 << 20, 1 << 20, 1 << 20, shape,
                                 ldp=6144, ldq=24576, ldc=24576)
    assert ei.value.status == fc.ERR_WORKSPACE
    assert "scratch" in str(ei.value)
