"""Seeded synthetic inputs shared by the oracle checks and the GPU path.

Holds none of the method's arithmetic: it only draws bf16 bit patterns from a
counter-based SplitMix64 stream (definition in ``gen.c``), so that the fp64
oracle and the CUDA kernels see identical inputs.  The shapes and value
distributions follow the FC-layer workloads of the GEMM benchmarks:
activations and gradients ~N(0, 1), weights ~N(0, 0.02) (0.02 is the standard
deviation), the layout sweep at N(0, 1) * 0.05, and small-integer operands for
the exact-arithmetic cases.

Arrays are ``numpy.uint16`` holding bf16 bits, C-contiguous, in the stored
(physical) shape the caller asks for.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libfc_inputs.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into an in-tree shared library (gcc + OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
        _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.fc_inputs_splitmix64.argtypes = [u64, i64, vp]
            lib.fc_inputs_normal_bf16.argtypes = [u64, u64, i64, i64, f64, f64, vp]
            lib.fc_inputs_small_int_bf16.argtypes = [u64, u64, i64, i64, i64, vp]
            for f in (lib.fc_inputs_splitmix64, lib.fc_inputs_normal_bf16,
                      lib.fc_inputs_small_int_bf16):
                f.restype = None
            _lib = lib
    return _lib


def splitmix64(x0: int, count: int) -> np.ndarray:
    """The first ``count`` outputs of a SplitMix64 generator seeded with x0."""
    out = np.empty(count, dtype=np.uint64)
    _load().fc_inputs_splitmix64(x0 & (2**64 - 1), count, out.ctypes.data)
    return out


def normal_bf16(shape, seed: int, tid: int, sigma: float = 1.0,
                mean: float = 0.0, start: int = 0) -> np.ndarray:
    """bf16 bits of N(mean, sigma^2) draws; element n of the flat array uses
    counter n + start of stream (seed, tid)."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size:
        _load().fc_inputs_normal_bf16(seed, tid, start, out.size, float(mean),
                                      float(sigma), out.ctypes.data)
    return out


def small_int_bf16(shape, seed: int, tid: int, h: int = 1,
                   start: int = 0) -> np.ndarray:
    """bf16 bits of integers drawn uniformly from [-h, h] (h=1: ternary)."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size:
        _load().fc_inputs_small_int_bf16(seed, tid, start, out.size, int(h),
                                         out.ctypes.data)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (for building test operands
    such as identity and rank-1 matrices; finite inputs only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def as_torch_bf16(bits: np.ndarray, device=None):
    """Wrap bf16 bits as a torch.bfloat16 tensor (copied to ``device``)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def from_torch_bf16(t) -> np.ndarray:
    """bf16 bits of a torch.bfloat16 tensor (moved to the host)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
