"""Per-shape tuning and the split of the reduction range, on the GPU.

Integer-valued operands make every fp32 sum exact, so each way of running a
product (kernel configuration, reduction split, rasterisation group) must
give the oracle's result bit for bit."""
import json

import numpy as np
import pytest

import oracle
from fc_cases import host_bits, make_operand, operand_names, to_device

pytestmark = pytest.mark.gpu


def _call(fc, op, P, Q, T, K, N, use_ws=True):
    import torch
    Pd, Qd = to_device(P), to_device(Q)
    M, Nn = fc.out_shape(op, T, K, N)
    ld = ((Nn + 7) // 8) * 8
    out = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :Nn]
    shape = fc.Shape(T, K, N)
    nbytes = fc.axonn_fc_workspace_size(op, shape, 0)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if (nbytes and use_ws) else None
    fc.call(op, Pd, Qd, out, shape, 0, ws)
    fc.axonn_sync_status()
    return out, fc.axonn_last_choice(), (Pd, Qd, out, shape, ws)


@pytest.fixture
def clean_cache(cuda_lib):
    cuda_lib.axonn_tune_cache_clear()
    cuda_lib.axonn_set_kernel_config(-1)
    yield cuda_lib
    cuda_lib.axonn_tune_cache_clear()


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_small_layer_splits_reduction(clean_cache, op):
    """The 256x512x2048 layer leaves most SMs idle.  The default choice
    splits only long reductions: the data gradient's 32 stages over 8 tiles,
    with or without a workspace (the split needs none); not the forward
    product's 8 stages, nor the weight gradient's 4."""
    fc = clean_cache
    T, K, N = 256, 512, 2048
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=101, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=101, kind="int")
    want = oracle.bf16_rne(oracle.fc(op, P, Q)[0])
    for use_ws in (True, False):
        out, choice, _ = _call(fc, op, P, Q, T, K, N, use_ws=use_ws)
        assert np.array_equal(host_bits(out), want)
        if op == "dgrad":
            assert choice[0] == 0 and choice[1] == 8, choice
        else:
            assert choice[1] == 1, choice


def test_every_split_and_config_exact(clean_cache, tmp_path):
    """Drive each (config, split, group) through a loaded tuning entry.  The
    reduction split runs on configurations 0 and 7 (128 x 128 and 128 x 64
    tiles); the others run such an entry unsplit."""
    fc = clean_cache
    T, K, N = 300, 1000, 520
    P = make_operand("X", T, K, N, False, seed=103, kind="int")
    Q = make_operand("W", T, K, N, False, seed=103, kind="int")
    want = oracle.bf16_rne(oracle.fc_fwd(P, Q)[0])
    sms, _ = fc.axonn_device_info()
    key = f"op0_T{T}_K{K}_N{N}_g1x1x1_at0.0.0_f0_sm{sms}"
    for cfg in range(fc.axonn_num_kernel_configs()):
        for split in (1, 2, 4, 8):
            for gm in (1, 16, -8):
                path = tmp_path / f"t{cfg}_{split}_{gm}.jsonl"
                path.write_text(json.dumps({"key": key, "config": fc.axonn_kernel_config_name(cfg),
                                            "split": split, "group_m": gm, "us": 1.0}) + "\n")
                fc.axonn_tune_cache_load(str(path))
                out, choice, _ = _call(fc, "fwd", P, Q, T, K, N)
                assert choice == (cfg, split if cfg in (0, 7) else 1, gm)
                bad = np.argwhere(host_bits(out) != want)
                assert bad.size == 0, (cfg, split, gm, bad[:3].tolist())


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_tune_records_fastest_and_reuses_it(clean_cache, op):
    fc = clean_cache
    T, K, N = 1024, 768, 1536
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=105, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=105, kind="int")
    want = oracle.bf16_rne(oracle.fc(op, P, Q)[0])
    out, _, (Pd, Qd, outd, shape, ws) = _call(fc, op, P, Q, T, K, N)
    cfg, split, gm, us = fc.axonn_fc_tune(op, Pd, Qd, outd, shape, 0, ws)
    assert 0 <= cfg < fc.axonn_num_kernel_configs() and split >= 1 and gm != 0 and us > 0
    assert fc.axonn_tune_cache_size() == 1
    assert np.array_equal(host_bits(outd), want)     # tuning leaves a correct product
    out2, choice, _ = _call(fc, op, P, Q, T, K, N)
    assert choice == (cfg, split, gm)
    assert np.array_equal(host_bits(out2), want)
