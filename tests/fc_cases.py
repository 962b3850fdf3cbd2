"""Shared helpers for the GPU parity tests: seeded operands, a call through
the C ABI, and the comparison against the fp64 oracle.

Seeds: one stream per (case seed, tensor id); tensor ids 1 = X, 2 = W,
3 = dY.  Value distributions follow the FC workloads: activations and
gradients N(0, 1), weights N(0, 0.02); the layout sweep scales N(0, 1) by
0.05; the exact-arithmetic cases draw integers in [-h, h].
"""
from __future__ import annotations

import numpy as np

import fc_inputs
import oracle

TID = {"X": 1, "W": 2, "dY": 3}


def operand_names(op):
    return {"fwd": ("X", "W"), "dgrad": ("dY", "W"), "wgrad": ("X", "dY")}[op]


def logical_shape(name, T, K, N):
    return {"X": (T, K), "W": (K, N), "dY": (T, N)}[name]


def make_operand(name, T, K, N, stored_t, seed, kind="normal", scale=None, h=1, pad=False):
    """bf16 bits of one operand in its stored layout.  The row stride is the
    row length rounded up to a multiple of 8 (TMA needs 16-byte strides),
    plus 8 more with ``pad``; a wider stride is returned as a view into the
    wider array."""
    r, c = logical_shape(name, T, K, N)
    if stored_t:
        r, c = c, r
    pad = ((c + 7) // 8) * 8 + (8 if pad else 0) - c
    if kind == "int":
        full = fc_inputs.small_int_bf16((r, c + pad), seed, TID[name], h=h)
    else:
        sigma = scale if scale is not None else (0.02 if name == "W" else 1.0)
        full = fc_inputs.normal_bf16((r, c + pad), seed, TID[name], sigma=sigma)
    return full[:, :c] if pad else full


def to_device(bits):
    """bf16 bits (possibly a row-padded view) -> CUDA tensor view with the
    same row stride."""
    base = bits.base
    padded_view = (base is not None and isinstance(base, np.ndarray) and base.ndim == 2
                   and base.shape[0] == bits.shape[0] and bits.strides == base.strides
                   and bits.ctypes.data == base.ctypes.data and base.flags.c_contiguous)
    if padded_view:       # a column slice of a wider array: keep its row stride
        return fc_inputs.as_torch_bf16(base, "cuda")[:, : bits.shape[1]]
    return fc_inputs.as_torch_bf16(np.ascontiguousarray(bits).copy(), "cuda")


def run_gpu(fc, op, P, Q, p_t, q_t, T, K, N, grid=(1, 1, 1), coords=(0, 0, 0), extra=0,
            out=None, out_f32=False, local_shape=None, workspace=True):
    """Call the op through the C ABI; returns the output tensor.  With
    workspace=False no workspace is passed (no stream-K tail, no two-launch
    grid sum)."""
    import torch
    Pd, Qd = to_device(P), to_device(Q)
    flags = (fc.A_T if p_t else 0) | (fc.B_T if q_t else 0) | extra
    shape = fc.Shape(T, K, N, grid, coords)
    if out is None:
        oshape = local_shape or fc.out_shape(op, T, K, N)
        dt = torch.float32 if (out_f32 or extra & (fc.ACCUM_F32 | fc.OUT_F32)) else torch.bfloat16
        ld = ((oshape[1] + 7) // 8) * 8
        out = torch.zeros((oshape[0], max(ld, 8)), dtype=dt, device="cuda")[:, : oshape[1]]
    nbytes = fc.axonn_fc_workspace_size(op, shape, flags) if workspace else 0
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    fc.call(op, Pd, Qd, out, shape, flags, ws)
    fc.axonn_sync_status()
    return out


def host_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def host_bits(t):
    return fc_inputs.from_torch_bf16(t)


def assert_within_bound(c_gpu, C, S, what=""):
    ratio = oracle.error_ratio(c_gpu, C, S)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, f"{what}: max |err|/(1e-2*S+1e-5) = {worst:.3g}"
    return worst


def sample_indices(M, N, seed, n_random=65536, band=4096):
    """Sampled (i, j): 2 full rows, 2 full columns, the ragged tail band
    (up to `band` entries) and n_random seeded random entries."""
    rng = np.random.default_rng(seed)
    I, J = [], []
    for i in (0, M - 1):
        I.append(np.full(N, i)); J.append(np.arange(N))
    for j in (0, N - 1):
        I.append(np.arange(M)); J.append(np.full(M, j))
    tm, tn = M % 128, N % 128
    if tm:
        k = min(band, tm * N)
        I.append(M - tm + rng.integers(0, tm, k)); J.append(rng.integers(0, N, k))
    if tn:
        k = min(band, tn * M)
        I.append(rng.integers(0, M, k)); J.append(N - tn + rng.integers(0, tn, k))
    I.append(rng.integers(0, M, n_random)); J.append(rng.integers(0, N, n_random))
    return np.concatenate(I).astype(np.int64), np.concatenate(J).astype(np.int64)
