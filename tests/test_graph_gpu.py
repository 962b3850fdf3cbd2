"""ABI calls captured into a CUDA graph replay to the oracle's results: no
call on the product path synchronises or allocates, and every kernel
parameter (tensor maps included) is captured by value."""
import numpy as np
import pytest

import oracle
from fc_cases import host_bits, make_operand, to_device

pytestmark = pytest.mark.gpu


def test_captured_full_vgrid_and_split_calls_replay_exactly(cuda_lib):
    import torch
    fc = cuda_lib
    fc.axonn_tune_cache_clear()
    s = torch.cuda.Stream()
    T, K, N = 300, 200, 2100   # the data gradient reduces over 33 stages: split by default
    X = make_operand("X", T, K, N, False, seed=401, kind="int")
    W = make_operand("W", T, K, N, False, seed=401, kind="int")
    dY = make_operand("dY", T, K, N, False, seed=401, kind="int")
    Xd, Wd, dYd = to_device(X), to_device(W), to_device(dY)
    Y = torch.zeros((T, 2104), dtype=torch.bfloat16, device="cuda")[:, :N]
    dX = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    dW = torch.zeros((K, 2104), dtype=torch.bfloat16, device="cuda")[:, :N]
    g3 = fc.Shape(T, K, N, (2, 2, 2))
    ws = torch.empty(max(fc.axonn_fc_workspace_size("fwd", g3, fc.VGRID),
                         fc.axonn_fc_workspace_size("dgrad", fc.Shape(T, K, N), 0), 16),
                     dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        fc.axonn_fc_fwd(Xd, Wd, Y, g3, fc.VGRID, ws, stream=s)           # warm-up, outside
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fc.axonn_fc_fwd(Xd, Wd, Y, g3, fc.VGRID, ws, stream=s)       # virtual grid
            fc.axonn_fc_dgrad(dYd, Wd, dX, fc.Shape(T, K, N), 0, ws, stream=s)   # split
            split = fc.axonn_last_choice()[1]
            fc.axonn_fc_wgrad(Xd, dYd, dW, fc.Shape(T, K, N), 0, None, stream=s)
        Y.zero_(); dX.zero_(); dW.zero_()
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    fc.axonn_sync_status(s)
    assert split > 1
    assert np.array_equal(host_bits(Y), oracle.bf16_rne(oracle.fc_fwd(X, W)[0]))
    assert np.array_equal(host_bits(dX), oracle.bf16_rne(oracle.fc_dgrad(dY, W)[0]))
    assert np.array_equal(host_bits(dW), oracle.bf16_rne(oracle.fc_wgrad(X, dY)[0]))
