"""Programmatic dependent launch keeps stream order: GEMMs that read the
previous GEMM's output (read after write) or overwrite its input (write
after read) give the oracle's exact result with the launches overlapped and
with plain launches, eagerly and replayed from a CUDA graph."""
import numpy as np
import pytest

import oracle
from fc_cases import host_bits, make_operand, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture
def restore(cuda_lib):
    yield
    cuda_lib.axonn_set_pdl(1)
    cuda_lib.axonn_set_kernel_config(-1)


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("cfg", [-1, 0, 5, 6])
@pytest.mark.parametrize("graph", [False, True])
def test_dependent_gemm_chain_exact(cuda_lib, restore, pdl, cfg, graph):
    import torch
    fc = cuda_lib
    fc.axonn_set_pdl(pdl)
    fc.axonn_set_kernel_config(cfg)
    T, K, N, N2 = 1024, 64, 768, 512
    X = make_operand("X", T, K, N, False, seed=601, kind="int")
    W = make_operand("W", T, K, N, False, seed=601, kind="int")
    W2 = make_operand("W", T, N, N2, False, seed=602, kind="int")
    A = make_operand("X", T, 96, K, False, seed=603, kind="int")
    B = make_operand("W", T, 96, K, False, seed=603, kind="int")
    Xd, Wd, W2d, Ad, Bd = (to_device(a) for a in (X, W, W2, A, B))
    Y = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    Z = torch.zeros((T, N2), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def chain():
        # Y = X.W; Z = Y.W2 reads Y (read after write); X = A.B then
        # overwrites X, which the first product read (write after read)
        fc.axonn_fc_fwd(Xd, Wd, Y, fc.Shape(T, K, N), 0, None, stream=s)
        fc.axonn_fc_fwd(Y, W2d, Z, fc.Shape(T, N, N2), 0, None, stream=s)
        fc.axonn_fc_fwd(Ad, Bd, Xd, fc.Shape(T, 96, K), 0, None, stream=s)

    torch.cuda.synchronize()
    if graph:
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                chain()
            g.replay()
    else:
        with torch.cuda.stream(s):
            chain()
    torch.cuda.synchronize()
    fc.axonn_sync_status(s)
    Yc, _ = oracle.fc_fwd(X, W)
    Yb = oracle.bf16_rne(Yc)
    Zc, _ = oracle.fc_fwd(Yb, W2)
    Xn, _ = oracle.fc_fwd(A, B)
    assert np.array_equal(host_bits(Y), Yb)
    assert np.array_equal(host_bits(Z), oracle.bf16_rne(Zc))
    assert np.array_equal(host_bits(Xd), oracle.bf16_rne(Xn))
