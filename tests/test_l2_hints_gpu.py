"""The L2 priorities of the operand loads (axonn_set_l2_budget) change where
lines live in L2, never a result: bit-identical outputs with the hints off,
at the default budget and at a budget smaller than every panel, for every
configuration, both rasterisation directions and a chained virtual grid."""
import numpy as np
import pytest

import oracle
from fc_cases import host_bits, make_operand, operand_names, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture
def budget(cuda_lib):
    old = cuda_lib.axonn_l2_budget()
    yield cuda_lib.axonn_set_l2_budget
    cuda_lib.axonn_set_l2_budget(old)
    cuda_lib.axonn_set_kernel_config(-1)
    cuda_lib.axonn_tune_cache_clear()


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("op", ["fwd", "wgrad"])
def test_l2_budget_leaves_results_unchanged(cuda_lib, budget, cfg, op):
    fc = cuda_lib
    fc.axonn_set_kernel_config(cfg)
    T, K, N = 1040, 1000, 2056
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=801, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=801, kind="int")
    want = oracle.bf16_rne(oracle.fc(op, P, Q)[0])
    outs = []
    for b in (0, 64 << 20, 4096):   # off, default, a fraction of every panel
        budget(b)
        outs.append(host_bits(run_gpu(fc, op, P, Q, False, False, T, K, N, workspace=False)))
    for o in outs:
        assert np.array_equal(o, want)


def test_l2_budget_with_column_groups_and_chained_grid(cuda_lib, budget, tmp_path):
    import json
    fc = cuda_lib
    T, K, N = 520, 1000, 776
    X = make_operand("X", T, K, N, False, seed=803, kind="int")
    W = make_operand("W", T, K, N, False, seed=803, kind="int")
    sms, _ = fc.axonn_device_info()
    key = f"op0_T{T}_K{K}_N{N}_g1x1x1_at0.0.0_f0_sm{sms}"
    path = tmp_path / "t.jsonl"
    path.write_text(json.dumps({"key": key, "config": "1cta_128x256", "split": 1, "group_m": -8,
                                "us": 1.0}) + "\n")
    fc.axonn_tune_cache_load(str(path))
    want = oracle.bf16_rne(oracle.fc_fwd(X, W)[0])
    Cg, _ = oracle.fc_vgrid("fwd", X, W, False, False, T, K, N, (2, 2, 2))
    want_g = oracle.bf16_rne(Cg)
    for b in (0, 64 << 20, 4096):
        budget(b)
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, workspace=False)
        assert fc.axonn_last_choice()[2] == -8
        assert np.array_equal(host_bits(out), want)
        out = run_gpu(fc, "fwd", X, W, False, False, T, K, N, grid=(2, 2, 2), extra=fc.VGRID)
        assert np.array_equal(host_bits(out), want_g)
