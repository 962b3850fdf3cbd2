"""GPU parity at the full sizes of the FC workloads, in the library's own
kernel choice and, for the GPT block, also in the choices of the tuning
table shipped for it, which are the launches the benchmark times.

The fp64 oracle is too slow for whole products of this size, so each check
covers the entries the oracle can compute one by one: 2 full rows, 2 full
columns, up to 4096 entries of every ragged tail band, and seeded random
entries.  Every checked entry must satisfy |C - C_ref| <= 1e-2 * S + 1e-5.

Workloads (seeded synthetic bf16; activations and gradients ~N(0,1), weights
~N(0,0.02), the layout sweep N(0,1) * 0.05):
  * GPT block, H = 6144, T = 8192: qkv, out, up, down layers, all three ops;
  * the same block as a 2x2x2 virtual grid (and one block on its own);
  * hidden 16384, MLP 53248, T = 4096: up and down layers, full and as a
    1x4x4 virtual grid;
  * the layout sweep: T in {512, 16384}, (K, N) with 1000/5000 tails.
"""
import zlib

import numpy as np
import pytest

import fc_inputs
import oracle
from fc_cases import assert_within_bound, host_f64, sample_indices

pytestmark = pytest.mark.gpu

H6, T6 = 6144, 8192
LAYERS6 = {"qkv": (H6, 3 * H6), "out": (H6, H6), "up": (H6, 4 * H6), "down": (4 * H6, H6)}


def _inputs(T, K, N, seed, tid_base, scale=None):
    sw = scale if scale is not None else 0.02
    sa = scale if scale is not None else 1.0
    X = fc_inputs.normal_bf16((T, K), seed, tid_base + 1, sigma=sa)
    W = fc_inputs.normal_bf16((K, N), seed, tid_base + 2, sigma=sw)
    dY = fc_inputs.normal_bf16((T, N), seed, tid_base + 3, sigma=sa)
    return X, W, dY


def _run_and_check(fc, op, X, W, dY, T, K, N, grid=(1, 1, 1), flags=0, n_random=65536,
                   seed=0):
    import torch
    P, Q = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (X, dY)}[op]
    Pd = fc_inputs.as_torch_bf16(P, "cuda")
    Qd = fc_inputs.as_torch_bf16(Q, "cuda")
    M, Nn = fc.out_shape(op, T, K, N)
    ld = ((Nn + 7) // 8) * 8
    out = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")[:, :Nn]
    shape = fc.Shape(T, K, N, grid)
    nbytes = fc.axonn_fc_workspace_size(op, shape, flags)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    fc.call(op, Pd, Qd, out, shape, flags, ws)
    fc.axonn_sync_status()
    del Pd, Qd, ws
    I, J = sample_indices(M, Nn, seed, n_random=n_random)
    got = host_f64(out[torch.from_numpy(I).cuda(), torch.from_numpy(J).cuda()])
    C, S = oracle.fc_entries(op, P, Q, False, False, I, J)
    del out
    torch.cuda.empty_cache()
    return assert_within_bound(got, C, S, f"{op} T={T} K={K} N={N} grid={grid}")


@pytest.fixture(scope="module")
def gpt6144():
    return {name: _inputs(T6, K, N, 1002, 16 * (i + 1))
            for i, (name, (K, N)) in enumerate(LAYERS6.items())}


@pytest.mark.parametrize("layer", list(LAYERS6))
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_gpt_block_h6144_t8192(cuda_lib, gpt6144, layer, op):
    K, N = LAYERS6[layer]
    X, W, dY = gpt6144[layer]
    _run_and_check(cuda_lib, op, X, W, dY, T6, K, N, n_random=32768,
                   seed=zlib.crc32(f"{layer}:{op}".encode()) & 0xFFFF)


@pytest.fixture
def shipped_table(cuda_lib):
    """Loads the GPT block's shipped tuning table; clears it afterwards."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "pmm_fc_layer_gb300", "tuned", "gpt_h6144_t8192.jsonl")
    fc = cuda_lib
    fc.axonn_tune_cache_clear()
    fc.axonn_tune_cache_load(path)
    yield {json.loads(l)["key"]: json.loads(l) for l in open(path).read().splitlines() if l.strip()}
    fc.axonn_tune_cache_clear()


@pytest.mark.parametrize("layer", list(LAYERS6))
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_gpt_block_h6144_t8192_shipped_choices(cuda_lib, gpt6144, shipped_table, layer, op):
    """Each GEMM runs the shipped table's configuration, rasterisation group,
    split and operand roles (with its stream-K mode), and is checked like
    the default choice above."""
    fc = cuda_lib
    sms, _ = fc.axonn_device_info()
    K, N = LAYERS6[layer]
    key = f"op{fc.OPS[op]}_T{T6}_K{K}_N{N}_g1x1x1_at0.0.0_f0_sm{sms}"
    if key not in shipped_table:
        pytest.skip(f"the shipped table is for another SM count ({sms} SMs here)")
    X, W, dY = gpt6144[layer]
    _run_and_check(fc, op, X, W, dY, T6, K, N, n_random=32768,
                   seed=zlib.crc32(f"shipped {layer}:{op}".encode()) & 0xFFFF)
    want = shipped_table[key]
    assert fc.axonn_kernel_config_name(fc.axonn_last_choice()[0]) == want["config"]
    assert fc.axonn_last_choice()[1:] == (want["split"], want["group_m"])
    assert fc.axonn_last_swap() == want["swap"]


@pytest.mark.parametrize("form", ["chained", "partials"])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_gpt_block_vgrid_2x2x2_up(cuda_lib, gpt6144, op, form):
    K, N = LAYERS6["up"]
    X, W, dY = gpt6144["up"]
    flags = cuda_lib.VGRID | (cuda_lib.VGRID_PARTIALS if form == "partials" else 0)
    _run_and_check(cuda_lib, op, X, W, dY, T6, K, N, grid=(2, 2, 2), flags=flags,
                   n_random=32768, seed=7)


def test_gpt_block_single_block_2x2x2_qkv(cuda_lib, gpt6144):
    """Block (1,0,1) of the 2x2x2 grid, fwd, fp32 partial at its place in
    the full output: X_blk[4096x3072] . W_blk[3072x9216]."""
    import torch
    fc = cuda_lib
    K, N = LAYERS6["qkv"]
    X, W, _ = gpt6144["qkv"]
    grid, coords = (2, 2, 2), (1, 0, 1)
    Xd, Wd = fc_inputs.as_torch_bf16(X, "cuda"), fc_inputs.as_torch_bf16(W, "cuda")
    out = torch.zeros((T6, N), dtype=torch.float32, device="cuda")
    fc.axonn_fc_fwd(Xd, Wd, out, fc.Shape(T6, K, N, grid, coords),
                    fc.FULL_OPERANDS | fc.OUT_F32)
    fc.axonn_sync_status()
    rows, red, cols = oracle.block_extents("fwd", T6, K, N, grid, coords)
    assert (rows, red, cols) == ((4096, 8192), (3072, 6144), (0, 9216))
    Xb = X[rows[0]:rows[1], red[0]:red[1]]
    Wb = W[red[0]:red[1], cols[0]:cols[1]]
    I, J = sample_indices(rows[1] - rows[0], cols[1] - cols[0], 11, n_random=32768)
    C, S = oracle.gemm_entries(Xb, False, Wb, False, I, J)
    got = host_f64(out[torch.from_numpy(I + rows[0]).cuda(), torch.from_numpy(J + cols[0]).cuda()])
    assert_within_bound(got, C, S, "block (1,0,1)")
    # outside the block nothing was written
    assert torch.count_nonzero(out[: rows[0]]).item() == 0
    assert torch.count_nonzero(out[:, cols[1]:]).item() == 0


@pytest.fixture(scope="module")
def large16384():
    H, F, T = 16384, 53248, 4096
    return {"up": _inputs(T, H, F, 1004, 64), "down": _inputs(T, F, H, 1004, 80)}


@pytest.mark.parametrize("layer", ["up", "down"])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_large_h16384_full(cuda_lib, large16384, layer, op):
    T = 4096
    K, N = (16384, 53248) if layer == "up" else (53248, 16384)
    X, W, dY = large16384[layer]
    _run_and_check(cuda_lib, op, X, W, dY, T, K, N, n_random=8192, seed=13)


@pytest.mark.parametrize("form", ["chained", "partials"])
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_large_h16384_vgrid_1x4x4_up(cuda_lib, large16384, op, form):
    T, K, N = 4096, 16384, 53248
    X, W, dY = large16384["up"]
    flags = cuda_lib.VGRID | (cuda_lib.VGRID_PARTIALS if form == "partials" else 0)
    _run_and_check(cuda_lib, op, X, W, dY, T, K, N, grid=(1, 4, 4), flags=flags,
                   n_random=8192, seed=17)


SWEEP = [(512, 1000, 5000), (512, 5000, 1000), (16384, 1000, 5000), (16384, 4096, 12288),
         (2048, 5000, 4096), (8192, 12288, 1000)]


@pytest.mark.parametrize("T,K,N", SWEEP)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])   # layouts NN, NT, TN
def test_layout_sweep(cuda_lib, T, K, N, op):
    X, W, dY = _inputs(T, K, N, 1005, 96, scale=0.05)
    _run_and_check(cuda_lib, op, X, W, dY, T, K, N, n_random=16384, seed=T + K + N)
