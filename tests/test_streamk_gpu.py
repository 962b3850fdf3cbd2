"""GPU parity of the stream-K tail against the fp64 oracle.

A launch runs stream-K pieces only when its output tiles outnumber the
persistent grid (152 CTAs, or 76 CTA pairs) and leave a partial round, so
the shapes here are sized per operation so that every kernel configuration
gets there.  Output 2600 x 4200 with a reduction of 520 (9 steps of 64, the
last one ragged) gives:

  config           tiles   units   stream-K tiles   whole-tile rounds
  1cta_128x128      693     152        237               3
  1cta_128x256      357     152        205               1
  pair_256x256      187      76        111               1
  1cta_256x256      187     152        187               0
  1cta_128x192      462     152        158               2
  1cta_256x192      242     152        242               0
  pair_512x256      102      76        102               0

Integer-valued operands make every order of summation exact, so those
results must match the oracle bit for bit whether the pieces are split or
not.  Random operands must satisfy |C_gpu - C| <= 1e-2 * S + 1e-5 with
stream-K on and off.
"""
import numpy as np
import pytest

import oracle
from fc_cases import (assert_within_bound, host_bits, host_f64, make_operand, operand_names,
                      run_gpu)

pytestmark = pytest.mark.gpu

CONFIGS = [0, 1, 2, 3, 4, 5, 6, 7]
# (T, K, N) per op so that the output is 2600 x 4200 and the reduction 520
SHAPES = {"fwd": (2600, 520, 4200), "dgrad": (2600, 4200, 520), "wgrad": (520, 2600, 4200)}
EXPECTED_SK = {0: 237, 1: 205, 2: 111, 3: 187, 4: 158, 5: 242, 6: 102, 7: 170}


@pytest.fixture
def forced(cuda_lib, request):
    cfg = request.param
    cuda_lib.axonn_set_kernel_config(cfg)
    yield cfg
    cuda_lib.axonn_set_kernel_config(-1)
    cuda_lib.axonn_set_streamk(-1)


def _expected_sk(fc, cfg):
    sms, pairs = fc.axonn_device_info()
    if (sms, pairs) != (152, 76):
        return None      # table above is for a 152-SM GB300
    return EXPECTED_SK[cfg]


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_streamk_integer_exact(cuda_lib, forced, op):
    T, K, N = SHAPES[op]
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=61, kind="int")
    Q = make_operand(qn, T, K, N, False, seed=61, kind="int")
    C, _ = oracle.fc(op, P, Q)
    want = oracle.bf16_rne(C)
    for mode in (1, 0):
        cuda_lib.axonn_set_streamk(mode)
        out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N)
        assert cuda_lib.axonn_last_kernel_config() == forced
        sk = cuda_lib.axonn_last_streamk_tiles()
        if mode == 0:
            assert sk == 0
        else:
            exp = _expected_sk(cuda_lib, forced)
            assert sk > 0 and (exp is None or sk == exp)
        got = host_bits(out)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"streamk={mode}: {len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("forced", CONFIGS, indirect=True)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_streamk_random(cuda_lib, forced, op):
    T, K, N = SHAPES[op]
    pn, qn = operand_names(op)
    P = make_operand(pn, T, K, N, False, seed=1061)
    Q = make_operand(qn, T, K, N, False, seed=1061)
    C, S = oracle.fc(op, P, Q)
    for mode in (1, 0):
        cuda_lib.axonn_set_streamk(mode)
        out = run_gpu(cuda_lib, op, P, Q, False, False, T, K, N)
        assert (cuda_lib.axonn_last_streamk_tiles() > 0) == (mode == 1)
        assert_within_bound(host_f64(out), C, S, f"config {forced} {op} streamk={mode}")


@pytest.mark.parametrize("forced", [5, 6], indirect=True)
@pytest.mark.parametrize("p_t,q_t", [(False, True), (True, False), (True, True)])
def test_streamk_layouts_integer_exact(cuda_lib, forced, p_t, q_t):
    """Transposed storage (MN-major tiles, 3-D boxes) through the stream-K path."""
    T, K, N = SHAPES["fwd"]
    P = make_operand("X", T, K, N, p_t, seed=62, kind="int")
    Q = make_operand("W", T, K, N, q_t, seed=62, kind="int")
    cuda_lib.axonn_set_streamk(1)
    out = run_gpu(cuda_lib, "fwd", P, Q, p_t, q_t, T, K, N)
    assert cuda_lib.axonn_last_streamk_tiles() > 0
    C, _ = oracle.fc("fwd", P, Q, p_t, q_t)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


@pytest.mark.parametrize("forced", [0, 5, 6], indirect=True)
@pytest.mark.parametrize("mode", ["out_f32", "accum_f32"])
def test_streamk_fp32_outputs(cuda_lib, forced, mode):
    """fp32 output, and accumulation into an fp32 output: the head piece adds
    the tail's partial and then the existing output."""
    import torch
    T, K, N = SHAPES["fwd"]
    P = make_operand("X", T, K, N, False, seed=1062)
    Q = make_operand("W", T, K, N, False, seed=1062)
    C, S = oracle.fc("fwd", P, Q)
    ld = ((N + 7) // 8) * 8
    out = torch.zeros((T, ld), dtype=torch.float32, device="cuda")[:, :N]
    base = None
    if mode == "accum_f32":
        g = torch.Generator().manual_seed(5)
        base = torch.randn((T, N), generator=g, dtype=torch.float32)
        out.copy_(base.cuda())
    flag = cuda_lib.ACCUM_F32 if mode == "accum_f32" else cuda_lib.OUT_F32
    cuda_lib.axonn_set_streamk(1)
    run_gpu(cuda_lib, "fwd", P, Q, False, False, T, K, N, extra=flag, out=out)
    assert cuda_lib.axonn_last_streamk_tiles() > 0
    want = C if base is None else C + base.double().numpy()
    S2 = S if base is None else S + np.abs(base.double().numpy())
    assert_within_bound(host_f64(out), want, S2, f"config {forced} {mode}")


@pytest.mark.parametrize("forced", [0, 5, 6], indirect=True)
@pytest.mark.parametrize("R", [64, 128, 200])
def test_streamk_short_reductions(cuda_lib, forced, R):
    """One reduction step (no stream-K: a tile cannot be cut), two steps, and
    a ragged four: every piece boundary a step boundary."""
    T, N = 2600, 4200
    P = make_operand("X", T, R, N, False, seed=63, kind="int")
    Q = make_operand("W", T, R, N, False, seed=63, kind="int")
    cuda_lib.axonn_set_streamk(1)
    out = run_gpu(cuda_lib, "fwd", P, Q, False, False, T, R, N)
    assert (cuda_lib.axonn_last_streamk_tiles() > 0) == (R > 64)
    C, _ = oracle.fc("fwd", P, Q)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


def test_streamk_without_workspace(cuda_lib):
    """No workspace: the same call runs whole tiles only, still exact."""
    import torch
    import fc_inputs
    T, K, N = SHAPES["fwd"]
    P = make_operand("X", T, K, N, False, seed=64, kind="int")
    Q = make_operand("W", T, K, N, False, seed=64, kind="int")
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    cuda_lib.axonn_set_kernel_config(5)
    cuda_lib.axonn_set_streamk(1)
    try:
        cuda_lib.call("fwd", fc_inputs.as_torch_bf16(P, "cuda"), fc_inputs.as_torch_bf16(Q, "cuda"),
                      out, cuda_lib.Shape(T, K, N), 0, None)
        cuda_lib.axonn_sync_status()
        assert cuda_lib.axonn_last_streamk_tiles() == 0
    finally:
        cuda_lib.axonn_set_kernel_config(-1)
        cuda_lib.axonn_set_streamk(-1)
    C, _ = oracle.fc("fwd", P, Q)
    assert np.array_equal(host_bits(out), oracle.bf16_rne(C))


def test_streamk_repeat_and_graph(cuda_lib):
    """The counters are cleared in stream order before every launch, so
    back-to-back calls and replays of a captured graph stay exact."""
    import torch
    import fc_inputs
    T, K, N = SHAPES["fwd"]
    P = make_operand("X", T, K, N, False, seed=65, kind="int")
    Q = make_operand("W", T, K, N, False, seed=65, kind="int")
    want = oracle.bf16_rne(oracle.fc("fwd", P, Q)[0])
    Pd, Qd = fc_inputs.as_torch_bf16(P, "cuda"), fc_inputs.as_torch_bf16(Q, "cuda")
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    shape = cuda_lib.Shape(T, K, N)
    ws = torch.empty(cuda_lib.axonn_fc_workspace_size("fwd", shape, 0), dtype=torch.uint8,
                     device="cuda")
    cuda_lib.axonn_set_kernel_config(5)
    cuda_lib.axonn_set_streamk(1)
    try:
        for _ in range(3):
            cuda_lib.call("fwd", Pd, Qd, out, shape, 0, ws)
        cuda_lib.axonn_sync_status()
        assert np.array_equal(host_bits(out), want)
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                cuda_lib.call("fwd", Pd, Qd, out, shape, 0, ws, stream=s)
            for _ in range(4):
                out.zero_()
                g.replay()
        torch.cuda.synchronize()
        cuda_lib.axonn_sync_status(s)
        assert np.array_equal(host_bits(out), want)
    finally:
        cuda_lib.axonn_set_kernel_config(-1)
        cuda_lib.axonn_set_streamk(-1)


def test_streamk_concurrent_streams(cuda_lib):
    """Two stream-K products on two streams at once.  The two pieces of a
    tile never wait for each other (the second to finish completes the
    tile), so a launch does not need all of its CTAs resident together and
    concurrent launches cannot stall each other."""
    import torch
    import fc_inputs
    fc = cuda_lib
    jobs = []
    for op, seed in (("fwd", 66), ("dgrad", 67)):
        T, K, N = SHAPES[op]
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=seed, kind="int")
        Q = make_operand(qn, T, K, N, False, seed=seed, kind="int")
        want = oracle.bf16_rne(oracle.fc(op, P, Q)[0])
        M, Nn = fc.out_shape(op, T, K, N)
        out = torch.zeros((M, Nn), dtype=torch.bfloat16, device="cuda")
        shape = fc.Shape(T, K, N)
        ws = torch.empty(fc.axonn_fc_workspace_size(op, shape, 0), dtype=torch.uint8, device="cuda")
        jobs.append((op, fc_inputs.as_torch_bf16(P, "cuda"), fc_inputs.as_torch_bf16(Q, "cuda"),
                     out, shape, ws, want, torch.cuda.Stream()))
    fc.axonn_set_kernel_config(5)
    fc.axonn_set_streamk(1)
    try:
        torch.cuda.synchronize()
        for _ in range(4):
            for op, Pd, Qd, out, shape, ws, _, s in jobs:
                fc.call(op, Pd, Qd, out, shape, 0, ws, stream=s)
                assert fc.axonn_last_streamk_tiles() > 0
        torch.cuda.synchronize()
        for *_, s in jobs:
            fc.axonn_sync_status(s)
    finally:
        fc.axonn_set_kernel_config(-1)
        fc.axonn_set_streamk(-1)
    for op, _, _, out, _, _, want, _ in jobs:
        assert np.array_equal(host_bits(out), want), op
