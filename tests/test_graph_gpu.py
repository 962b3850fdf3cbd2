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


def test_captured_pipeline_with_host_copies_replays_exactly(cuda_lib):
    """The benchmark's host-buffer pass as one graph: pinned-host inputs
    copied up on one stream, the three products through the ABI on
    another, the outputs copied down on a third, two layers pipelined by
    events.  Each replay moves and computes everything again: the host
    outputs match the oracle bit for bit, and inputs rewritten in the host
    buffers between replays are the ones used."""
    import fc_inputs
    import torch
    fc = cuda_lib
    fc.axonn_tune_cache_clear()
    T, K, N = 256, 384, 640
    data = [tuple(make_operand(n, T, K, N, False, seed=411 + li, kind="int") for n in ("X", "W", "dY"))
            for li in range(2)]
    shape = fc.Shape(T, K, N)
    hin = [{k: fc_inputs.as_torch_bf16(v).pin_memory() for k, v in zip(("X", "W", "dY"), d)}
           for d in data]
    dev = [{k: torch.empty_like(v, device="cuda") for k, v in h.items()} for h in hin]
    dout = [{"Y": torch.empty((T, N), dtype=torch.bfloat16, device="cuda"),
             "dX": torch.empty((T, K), dtype=torch.bfloat16, device="cuda"),
             "dW": torch.empty((K, N), dtype=torch.bfloat16, device="cuda")} for _ in data]
    hout = [{k: torch.empty(v.shape, dtype=torch.bfloat16).pin_memory() for k, v in d.items()}
            for d in dout]
    comp, up, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in data]
    done = [torch.cuda.Event() for _ in data]

    def one_pass():
        for li in range(len(data)):
            with torch.cuda.stream(up):
                for k, hb in hin[li].items():
                    dev[li][k].copy_(hb, non_blocking=True)
            in_ready[li].record(up)
            comp.wait_event(in_ready[li])
            d, o = dev[li], dout[li]
            fc.axonn_fc_fwd(d["X"], d["W"], o["Y"], shape, 0, None, stream=comp)
            fc.axonn_fc_dgrad(d["dY"], d["W"], o["dX"], shape, 0, None, stream=comp)
            fc.axonn_fc_wgrad(d["X"], d["dY"], o["dW"], shape, 0, None, stream=comp)
            done[li].record(comp)
            down.wait_event(done[li])
            with torch.cuda.stream(down):
                for k, hb in hout[li].items():
                    hb.copy_(o[k], non_blocking=True)

    with torch.cuda.stream(comp):
        one_pass()                                  # warm-up, outside
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=comp):
        up.wait_stream(comp)
        down.wait_stream(comp)
        one_pass()
        comp.wait_stream(up)
        comp.wait_stream(down)

    def check(expect):
        for li, (X, W, dY) in enumerate(expect):
            want = {"Y": oracle.fc_fwd(X, W)[0], "dX": oracle.fc_dgrad(dY, W)[0],
                    "dW": oracle.fc_wgrad(X, dY)[0]}
            for k, C in want.items():
                assert np.array_equal(fc_inputs.from_torch_bf16(hout[li][k]), oracle.bf16_rne(C)), (li, k)

    for h in hout:
        for t in h.values():
            t.zero_()
    with torch.cuda.stream(comp):
        graph.replay()
    torch.cuda.synchronize()
    fc.axonn_sync_status(comp)
    check(data)
    # new inputs in the same pinned buffers: the layers' inputs exchanged
    saved = [{k: v.clone() for k, v in h.items()} for h in hin]
    for li in range(2):
        for k in hin[li]:
            hin[li][k].copy_(saved[1 - li][k])
    with torch.cuda.stream(comp):
        graph.replay()
    torch.cuda.synchronize()
    fc.axonn_sync_status(comp)
    check([data[1], data[0]])
