"""Python binding of libaxonn_fc.so -- argument marshalling only.

Every function named ``axonn_*`` here calls the C entry point of the same
name (declared in include/axonn_fc.h); all arithmetic runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no fallback: if the library is missing or cannot load, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

OP_FWD, OP_DGRAD, OP_WGRAD = 0, 1, 2
OPS = {"fwd": OP_FWD, "dgrad": OP_DGRAD, "wgrad": OP_WGRAD}

A_T = 0x1
B_T = 0x2
ACCUM_F32 = 0x4
VGRID = 0x8
FULL_OPERANDS = 0x10
OUT_F32 = 0x20
ZSHARDED = 0x40
REDUCE_ADD = 0x80
VGRID_PARTIALS = 0x100

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)
STATUS_NAMES = ["OK", "INVALID_ARG", "ALIGNMENT", "UNSUPPORTED", "WORKSPACE", "CUDA", "TIMEOUT"]

EXPORTS = ("axonn_fc_fwd", "axonn_fc_dgrad", "axonn_fc_wgrad", "axonn_fc_vgrid_static",
           "axonn_shards_gather", "axonn_fc_wgrad_zsharded", "axonn_goldfish_ce",
           "axonn_fc_workspace_size", "axonn_fc_tune", "axonn_tune_cache_save",
           "axonn_tune_cache_load", "axonn_tune_cache_clear", "axonn_tune_cache_size",
           "axonn_tune_lookup",
           "axonn_last_choice",
           "axonn_block_range", "axonn_fc_block_extents", "axonn_sync_status", "axonn_set_wait_timeout_ns",
           "axonn_debug_set_inject", "axonn_set_kernel_config", "axonn_num_kernel_configs",
           "axonn_set_streamk", "axonn_last_streamk_tiles", "axonn_set_swap", "axonn_last_swap",
           "axonn_set_pdl", "axonn_set_l2_budget", "axonn_l2_budget",
           "axonn_device_info",
           "axonn_kernel_config_name", "axonn_last_kernel_config", "axonn_last_error",
           "axonn_version")


class AxonnError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"AXONN_ERR_{name}: {message}")


class Shape(ctypes.Structure):
    """axonn_fc_shape_t: layer sizes, 3D grid and block coordinate."""
    _fields_ = [("T", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int64),
                ("gx", ctypes.c_int32), ("gy", ctypes.c_int32), ("gz", ctypes.c_int32),
                ("x", ctypes.c_int32), ("y", ctypes.c_int32), ("z", ctypes.c_int32)]

    def __init__(self, T, K, N, grid=(1, 1, 1), coords=(0, 0, 0)):
        super().__init__(T, K, N, *grid, *coords)


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the built library (raises if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libaxonn_fc.so not built at {p}; run pmm_fc_layer_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i64, u32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_int32
        sz = ctypes.c_size_t
        sig = [vp, vp, vp, i64, i64, i64, ctypes.POINTER(Shape), u32, vp, sz, vp]
        for name in ("axonn_fc_fwd", "axonn_fc_dgrad", "axonn_fc_wgrad"):
            f = getattr(lib, name)
            f.argtypes = sig
            f.restype = ctypes.c_int
        lib.axonn_shards_gather.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, vp, i64, vp]
        lib.axonn_shards_gather.restype = ctypes.c_int
        lib.axonn_fc_wgrad_zsharded.argtypes = [vp, vp, ctypes.POINTER(vp), i64, i64, i64,
                                                ctypes.POINTER(Shape), u32, vp, sz, vp]
        lib.axonn_fc_wgrad_zsharded.restype = ctypes.c_int
        lib.axonn_goldfish_ce.argtypes = [vp, i64, vp, vp, i64, i64, i64, i32, i32, vp, vp, vp, vp,
                                          vp, i64, vp]
        lib.axonn_goldfish_ce.restype = ctypes.c_int
        lib.axonn_fc_vgrid_static.argtypes = [ctypes.c_int, vp, vp, vp, i64, i64, i64,
                                              ctypes.POINTER(Shape), u32, vp]
        lib.axonn_fc_vgrid_static.restype = ctypes.c_int
        lib.axonn_fc_tune.argtypes = [ctypes.c_int, vp, vp, vp, i64, i64, i64, ctypes.POINTER(Shape),
                                      u32, vp, sz, vp, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_float)]
        lib.axonn_fc_tune.restype = ctypes.c_int
        lib.axonn_tune_cache_save.argtypes = [ctypes.c_char_p]
        lib.axonn_tune_cache_save.restype = ctypes.c_int
        lib.axonn_tune_cache_load.argtypes = [ctypes.c_char_p]
        lib.axonn_tune_cache_load.restype = ctypes.c_int
        lib.axonn_tune_cache_clear.restype = None
        lib.axonn_tune_cache_size.restype = ctypes.c_int
        lib.axonn_tune_lookup.argtypes = [ctypes.c_int, ctypes.POINTER(Shape), u32,
                                          ctypes.POINTER(ctypes.c_int)]
        lib.axonn_tune_lookup.restype = ctypes.c_int
        lib.axonn_last_choice.argtypes = [ctypes.POINTER(ctypes.c_int)] * 3
        lib.axonn_last_choice.restype = None
        lib.axonn_fc_workspace_size.argtypes = [ctypes.c_int, ctypes.POINTER(Shape), u32,
                                                ctypes.POINTER(sz)]
        lib.axonn_fc_workspace_size.restype = ctypes.c_int
        lib.axonn_block_range.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.axonn_block_range.restype = ctypes.c_int
        lib.axonn_fc_block_extents.argtypes = [ctypes.c_int, ctypes.POINTER(Shape),
                                               ctypes.POINTER(i64), ctypes.POINTER(i64),
                                               ctypes.POINTER(i64)]
        lib.axonn_fc_block_extents.restype = ctypes.c_int
        lib.axonn_sync_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
        lib.axonn_sync_status.restype = ctypes.c_int
        lib.axonn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.axonn_set_wait_timeout_ns.restype = None
        lib.axonn_debug_set_inject.argtypes = [ctypes.c_int]
        lib.axonn_debug_set_inject.restype = None
        lib.axonn_set_kernel_config.argtypes = [ctypes.c_int]
        lib.axonn_set_kernel_config.restype = ctypes.c_int
        lib.axonn_set_streamk.argtypes = [ctypes.c_int]
        lib.axonn_set_streamk.restype = ctypes.c_int
        lib.axonn_last_streamk_tiles.argtypes = []
        lib.axonn_last_streamk_tiles.restype = ctypes.c_int
        lib.axonn_set_pdl.argtypes = [ctypes.c_int]
        lib.axonn_set_pdl.restype = ctypes.c_int
        lib.axonn_set_l2_budget.argtypes = [ctypes.c_int64]
        lib.axonn_set_l2_budget.restype = ctypes.c_int
        lib.axonn_l2_budget.argtypes = []
        lib.axonn_l2_budget.restype = ctypes.c_int64
        lib.axonn_set_swap.argtypes = [ctypes.c_int]
        lib.axonn_set_swap.restype = ctypes.c_int
        lib.axonn_last_swap.argtypes = []
        lib.axonn_last_swap.restype = ctypes.c_int
        lib.axonn_num_kernel_configs.restype = ctypes.c_int
        lib.axonn_device_info.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.axonn_device_info.restype = ctypes.c_int
        lib.axonn_kernel_config_name.argtypes = [ctypes.c_int]
        lib.axonn_kernel_config_name.restype = ctypes.c_char_p
        lib.axonn_last_kernel_config.restype = ctypes.c_int
        lib.axonn_last_error.restype = ctypes.c_char_p
        lib.axonn_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int):
    if status != OK:
        raise AxonnError(status, load().axonn_last_error().decode())


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ld(t, ld):
    if ld is not None:
        return int(ld)
    if t is None or isinstance(t, int):
        return 0
    if t.dim() != 2 or (t.stride(1) != 1 and t.size(1) > 1):
        raise ValueError("operands must be 2-D with unit column stride")
    return t.stride(0)


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, P, Q, C, shape, flags, ws, ldp, ldq, ldc, stream):
    lib = load()
    ws_bytes = 0
    if ws is not None and not isinstance(ws, int):
        ws_bytes = ws.numel() * ws.element_size()
    elif isinstance(ws, int):
        raise ValueError("pass the workspace as a tensor")
    st = getattr(lib, name)(_ptr(P), _ptr(Q), _ptr(C), _ld(P, ldp), _ld(Q, ldq), _ld(C, ldc),
                            ctypes.byref(shape), flags, _ptr(ws), ws_bytes, _stream(stream))
    _check(st)


def axonn_fc_fwd(X, W, Y, shape: Shape, flags: int = 0, ws=None, ldx=None, ldw=None, ldy=None,
                 stream=None):
    """Y = X . W (layer, block or virtual grid); see include/axonn_fc.h."""
    _call("axonn_fc_fwd", X, W, Y, shape, flags, ws, ldx, ldw, ldy, stream)


def axonn_fc_dgrad(dY, W, dX, shape: Shape, flags: int = 0, ws=None, lddy=None, ldw=None,
                   lddx=None, stream=None):
    """dX = dY . W^T (layer, block or virtual grid)."""
    _call("axonn_fc_dgrad", dY, W, dX, shape, flags, ws, lddy, ldw, lddx, stream)


def axonn_fc_wgrad(X, dY, dW, shape: Shape, flags: int = 0, ws=None, ldx=None, lddy=None,
                   lddw=None, stream=None):
    """dW = X^T . dY (layer, block or virtual grid)."""
    _call("axonn_fc_wgrad", X, dY, dW, shape, flags, ws, ldx, lddy, lddw, stream)


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


def axonn_shards_gather(shards, out, rows: int, cols: int, ld_shard=None, ld_out=None,
                        stream=None):
    """All-gather of row shards on one GPU: out[rows x cols] <- shards
    (shard z holds rows split_range(rows, len(shards), z))."""
    ld_s = ld_shard if ld_shard is not None else next(
        (_ld(t, None) for t in shards if t is not None and t.numel()), cols)
    _check(load().axonn_shards_gather(_ptr_array(shards), len(shards), rows, cols, ld_s, _ptr(out),
                                      _ld(out, ld_out), _stream(stream)))


def axonn_fc_wgrad_zsharded(X, dY, dW_shards, shape: Shape, flags: int = 0, ws=None, ldx=None,
                            lddy=None, ld_shard=None, stream=None):
    """Weight gradient of block (x, y) summed over the Z group and written as
    row shards (the grid's reduce-scatter) into dW_shards."""
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    ld_s = ld_shard if ld_shard is not None else next(
        (_ld(t, None) for t in dW_shards if t is not None and t.numel()), 8)
    _check(load().axonn_fc_wgrad_zsharded(_ptr(X), _ptr(dY), _ptr_array(dW_shards), _ld(X, ldx),
                                          _ld(dY, lddy), ld_s, ctypes.byref(shape), flags,
                                          _ptr(ws), ws_bytes, _stream(stream)))


def axonn_fc_vgrid_static(op, P, Q, C, shape: Shape, flags: int = 0, ldp=None, ldq=None,
                          ldc=None, stream=None):
    """Virtual-grid product with the library's fixed scratch: nothing is
    allocated and no workspace is passed (for callers that cannot allocate
    device memory).  ``op`` is 'fwd', 'dgrad' or 'wgrad'."""
    op = OPS.get(op, op)
    st = load().axonn_fc_vgrid_static(int(op), _ptr(P), _ptr(Q), _ptr(C), _ld(P, ldp), _ld(Q, ldq),
                                      _ld(C, ldc), ctypes.byref(shape), flags, _stream(stream))
    _check(st)


def axonn_goldfish_ce(logits, input_ids, labels, keep, token_loss, loss, kept, k=2, h=13,
                      dlogits=None, ld_logits=None, ld_dlogits=None, stream=None):
    """Goldfish-masked cross-entropy of bf16 logits [B*S x V] for int32
    input_ids / labels [B x S]: fills keep [B*S] (uint8), token_loss [B*S],
    loss [1], kept [1] (int32) and, if given, dlogits (bf16, the gradient of
    the mean loss)."""
    B, S = input_ids.shape
    V = logits.shape[1]
    _check(load().axonn_goldfish_ce(_ptr(logits), _ld(logits, ld_logits), _ptr(input_ids),
                                    _ptr(labels), B, S, V, int(k), int(h), _ptr(keep),
                                    _ptr(token_loss), _ptr(loss), _ptr(kept), _ptr(dlogits),
                                    _ld(dlogits, ld_dlogits) if dlogits is not None else 0,
                                    _stream(stream)))


def axonn_fc_tune(op, P, Q, C, shape: Shape, flags: int = 0, ws=None, ldp=None, ldq=None,
                  ldc=None, stream=None):
    """Time every candidate way to run this call and remember the fastest;
    returns (config, split, group_m, microseconds).  Overwrites C."""
    op = OPS.get(op, op)
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    c, sp, gm, us = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_float()
    _check(load().axonn_fc_tune(int(op), _ptr(P), _ptr(Q), _ptr(C), _ld(P, ldp), _ld(Q, ldq),
                                _ld(C, ldc), ctypes.byref(shape), flags, _ptr(ws), ws_bytes,
                                _stream(stream), ctypes.byref(c), ctypes.byref(sp),
                                ctypes.byref(gm), ctypes.byref(us)))
    return c.value, sp.value, gm.value, us.value


def axonn_tune_cache_save(path: str):
    _check(load().axonn_tune_cache_save(os.fsencode(path)))


def axonn_tune_cache_load(path: str):
    _check(load().axonn_tune_cache_load(os.fsencode(path)))


def axonn_tune_cache_clear():
    load().axonn_tune_cache_clear()


def axonn_tune_cache_size() -> int:
    return int(load().axonn_tune_cache_size())


def axonn_last_choice():
    """(config, split, group_m) of the last call on this thread."""
    c, s, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    load().axonn_last_choice(ctypes.byref(c), ctypes.byref(s), ctypes.byref(g))
    return c.value, s.value, g.value


def axonn_tune_lookup(op, shape: Shape, flags: int = 0) -> bool:
    """True when the tuning table holds an entry for this call on the
    current device."""
    op = OPS.get(op, op)
    found = ctypes.c_int(0)
    _check(load().axonn_tune_lookup(int(op), ctypes.byref(shape), flags, ctypes.byref(found)))
    return bool(found.value)


def axonn_fc_workspace_size(op, shape: Shape, flags: int = 0) -> int:
    op = OPS.get(op, op)
    n = ctypes.c_size_t(0)
    _check(load().axonn_fc_workspace_size(int(op), ctypes.byref(shape), flags, ctypes.byref(n)))
    return n.value


def axonn_block_range(D: int, G: int, b: int):
    s, e = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load().axonn_block_range(D, G, b, ctypes.byref(s), ctypes.byref(e)))
    return s.value, e.value


def axonn_fc_block_extents(op, shape: Shape):
    """((rows), (red), (cols)) of block (shape.x, shape.y, shape.z) of `op`,
    each a [start, stop) pair in the full matrices."""
    op = OPS.get(op, op)
    r, k, c = (ctypes.c_int64 * 2)(), (ctypes.c_int64 * 2)(), (ctypes.c_int64 * 2)()
    _check(load().axonn_fc_block_extents(int(op), ctypes.byref(shape), r, k, c))
    return (r[0], r[1]), (k[0], k[1]), (c[0], c[1])


def axonn_sync_status(stream=None, raise_on_error: bool = True):
    """Waits for the stream and returns (status, detail word)."""
    detail = ctypes.c_uint64(0)
    st = load().axonn_sync_status(_stream(stream), ctypes.byref(detail))
    if raise_on_error:
        _check(st)
    return st, detail.value


def axonn_set_wait_timeout_ns(ns: int):
    load().axonn_set_wait_timeout_ns(int(ns))


def axonn_debug_set_inject(mode: int):
    load().axonn_debug_set_inject(int(mode))


def axonn_set_kernel_config(config: int):
    """Force kernel configuration `config` (-1: automatic choice)."""
    _check(load().axonn_set_kernel_config(int(config)))


def axonn_set_streamk(mode: int):
    """Stream-K tail: -1 as tuned (default on), 0 off, 1 on."""
    _check(load().axonn_set_streamk(int(mode)))


def axonn_last_streamk_tiles() -> int:
    """Stream-K tiles of the last GEMM launch on this thread (0: none)."""
    return int(load().axonn_last_streamk_tiles())


def axonn_set_pdl(on: int):
    """1 (default): GEMMs are programmatic dependent launches; 0: plain launches."""
    _check(load().axonn_set_pdl(int(on)))


def axonn_set_l2_budget(nbytes: int):
    """L2 bytes a rasterisation group's kept operand panel may hold as
    evict-last lines (0: operand loads without L2 priorities)."""
    _check(load().axonn_set_l2_budget(int(nbytes)))


def axonn_l2_budget() -> int:
    return int(load().axonn_l2_budget())


def axonn_set_swap(mode: int):
    """Operand roles: -1 as tuned, 0 never exchanged, 1 exchanged (C^T = B^T.A^T)."""
    _check(load().axonn_set_swap(int(mode)))


def axonn_last_swap() -> int:
    """1 if the last call on this thread ran with exchanged operand roles."""
    return int(load().axonn_last_swap())


def axonn_device_info():
    """(SM count, resident CTA pairs) of the current device."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().axonn_device_info(ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def axonn_num_kernel_configs() -> int:
    return int(load().axonn_num_kernel_configs())


def axonn_kernel_config_name(config: int) -> str:
    return load().axonn_kernel_config_name(int(config)).decode()


def axonn_last_kernel_config() -> int:
    return int(load().axonn_last_kernel_config())


def axonn_last_error() -> str:
    return load().axonn_last_error().decode()


def axonn_version() -> str:
    return load().axonn_version().decode()


# ---------------------------------------------------------------- helpers
def out_shape(op, T, K, N):
    """Logical output shape of an op on the full layer."""
    op = OPS.get(op, op)
    return {OP_FWD: (T, N), OP_DGRAD: (T, K), OP_WGRAD: (K, N)}[op]


def call(op, P, Q, C, shape: Shape, flags: int = 0, ws=None, stream=None):
    """Dispatch by op name ('fwd' | 'dgrad' | 'wgrad') to the entry point."""
    op = OPS.get(op, op)
    fn = {OP_FWD: axonn_fc_fwd, OP_DGRAD: axonn_fc_dgrad, OP_WGRAD: axonn_fc_wgrad}[op]
    fn(P, Q, C, shape, flags, ws, stream=stream)
