"""Several host threads calling the C ABI at once, each on its own stream."""
import threading

import numpy as np
import pytest

import oracle
from fc_cases import host_bits, make_operand, operand_names, to_device

pytestmark = pytest.mark.gpu


def test_concurrent_calls_on_separate_streams(cuda_lib):
    import torch
    fc = cuda_lib
    cases = []
    for i, (op, (T, K, N)) in enumerate([("fwd", (300, 200, 520)), ("dgrad", (256, 384, 640)),
                                         ("wgrad", (512, 136, 264)), ("fwd", (1024, 512, 768))]):
        pn, qn = operand_names(op)
        P = make_operand(pn, T, K, N, False, seed=300 + i, kind="int")
        Q = make_operand(qn, T, K, N, False, seed=300 + i, kind="int")
        want = oracle.bf16_rne(oracle.fc(op, P, Q)[0])
        cases.append((op, T, K, N, to_device(P), to_device(Q), want))
    results, errors = {}, []

    def worker(idx):
        try:
            op, T, K, N, Pd, Qd, _ = cases[idx]
            s = torch.cuda.Stream()
            M, Nn = fc.out_shape(op, T, K, N)
            out = torch.empty((M, ((Nn + 7) // 8) * 8), dtype=torch.bfloat16, device="cuda")[:, :Nn]
            for _ in range(20):
                fc.call(op, Pd, Qd, out, fc.Shape(T, K, N), 0, None, stream=s)
            fc.axonn_sync_status(s)
            results[idx] = host_bits(out)
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, case in enumerate(cases):
        assert np.array_equal(results[i], case[-1]), i
