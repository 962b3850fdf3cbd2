"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point the header declares, resolves 3D-grid
blocks like the oracle's split rule, sizes workspaces, and rejects bad
arguments before touching a device."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "axonn_fc.h")


@pytest.fixture(scope="module")
def fc():
    from pmm_fc_layer_gb300 import build
    build.build()
    import pmm_fc_layer_gb300 as m
    m.load()
    return m


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(axonn_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(fc):
    syms = declared_symbols()
    assert len(syms) >= 10
    lib = ctypes.CDLL(fc.library_path())
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in the header but not exported"
    assert set(syms) == set(fc.EXPORTS)


def test_version(fc):
    assert "sm_103a" in fc.axonn_version()


def test_kernel_config_table(fc):
    n = fc.axonn_num_kernel_configs()
    assert n == 8
    assert [fc.axonn_kernel_config_name(i) for i in range(n)] == \
        ["1cta_128x128", "1cta_128x256", "pair_256x256", "1cta_256x256", "1cta_128x192",
         "1cta_256x192", "pair_512x256", "1cta_128x64"]
    with pytest.raises(fc.AxonnError):
        fc.axonn_set_kernel_config(n)
    fc.axonn_set_kernel_config(2)
    fc.axonn_set_kernel_config(-1)


@pytest.mark.parametrize("D", [0, 1, 7, 8, 300, 1000, 5000, 6144, 24576, 53248])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
def test_block_range_matches_oracle_rule(fc, D, G):
    for b in range(G):
        assert fc.axonn_block_range(D, G, b) == oracle.split_range(D, G, b)


def test_block_extents_hand_table(fc):
    """The library's own block resolution (which grid axis cuts which
    dimension, and each op's rows / reduced range / columns) against the
    hand-worked table in tests/golden/, on the CPU."""
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "fc_hand_examples.json")))
    for case in g["block_extents"]["cases"]:
        shape = fc.Shape(*case["TKN"], tuple(case["grid"]), tuple(case["coords"]))
        for op in ("fwd", "dgrad", "wgrad"):
            got = fc.axonn_fc_block_extents(op, shape)
            assert [list(r) for r in got] == case[op], (case["TKN"], op)
    with pytest.raises(fc.AxonnError):
        fc.axonn_fc_block_extents("fwd", fc.Shape(64, 64, 64, (2, 1, 1), (2, 0, 0)))


def test_block_range_errors(fc):
    with pytest.raises(fc.AxonnError):
        fc.axonn_block_range(10, 0, 0)
    with pytest.raises(fc.AxonnError):
        fc.axonn_block_range(10, 2, 2)


def test_workspace_size(fc):
    s = fc.Shape(8192, 6144, 24576, (2, 2, 2))
    assert fc.axonn_fc_workspace_size("fwd", s, 0) == 0
    P = fc.VGRID | fc.VGRID_PARTIALS   # the two-launch form keeps G-1 partials
    assert fc.axonn_fc_workspace_size("fwd", s, fc.VGRID) == 0   # chained: none
    assert fc.axonn_fc_workspace_size("fwd", s, P) == 1 * 8192 * 24576 * 4
    assert fc.axonn_fc_workspace_size("dgrad", s, P) == 1 * 8192 * 6144 * 4
    assert fc.axonn_fc_workspace_size("wgrad", s, P) == 1 * 6144 * 24576 * 4
    s4 = fc.Shape(4096, 16384, 18432, (1, 4, 4))
    assert fc.axonn_fc_workspace_size("fwd", s4, P) == 0      # G_x = 1
    assert fc.axonn_fc_workspace_size("dgrad", s4, P) == 3 * 4096 * 16384 * 4
    odd = fc.Shape(100, 60, 1001, (1, 1, 3))
    assert fc.axonn_fc_workspace_size("wgrad", odd, P) == 2 * 60 * 1008 * 4


def _status(fc, fn, *args):
    return fn(*args)


def _raw(fc, name, P, Q, C, ldp, ldq, ldc, shape, flags, ws=0, ws_bytes=0):
    lib = fc.load()
    return getattr(lib, name)(P, Q, C, ldp, ldq, ldc, ctypes.byref(shape), flags, ws, ws_bytes, 0)


FAKE = 0x10000000  # never dereferenced: every case below fails validation


@pytest.mark.parametrize("case,expect", [
    (dict(shape=(64, 64, 64), grid=(0, 1, 1)), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), coords=(2, 0, 0)), 1),
    (dict(shape=(-1, 64, 64)), 1),
    (dict(shape=(64, 64, 64), flags=0x400), 1),
    (dict(shape=(64, 64, 64), flags=0x4 | 0x20), 1),
    (dict(shape=(64, 64, 64), grid=(8, 4, 4), flags=0x8), 3),
    (dict(shape=(64, 64, 64), P=FAKE + 8), 2),
    (dict(shape=(64, 64, 64), ldp=68), 2),
    (dict(shape=(64, 64, 64), ldp=32), 1),
    (dict(shape=(64, 64, 64), C=FAKE + 4), 2),
    (dict(shape=(64, 64, 64), P=0), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x8 | 0x100), 4),
    # the two-launch grid sum needs the virtual grid and excludes the order-free one
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x100), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x8 | 0x100 | 0x80 | 0x4), 1),
    # the order-free sum needs the virtual grid and an accumulating fp32 output
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x80), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x80 | 0x8), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x80 | 0x4), 1),
    (dict(shape=(64, 64, 64), grid=(2, 1, 1), flags=0x80 | 0x8 | 0x20), 1),
])
def test_validation_errors(fc, case, expect):
    T, K, N = case["shape"]
    shape = fc.Shape(T, K, N, case.get("grid", (1, 1, 1)), case.get("coords", (0, 0, 0)))
    st = _raw(fc, "axonn_fc_fwd", case.get("P", FAKE), case.get("Q", FAKE), case.get("C", FAKE),
              case.get("ldp", 64), case.get("ldq", 64), case.get("ldc", 64), shape,
              case.get("flags", 0))
    assert st == expect, fc.axonn_last_error()
    assert fc.axonn_last_error()


def test_no_device_is_an_error_not_a_fallback(fc):
    """Valid arguments on a machine without a GPU must fail loudly."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _raw(fc, "axonn_fc_fwd", FAKE, FAKE, FAKE, 64, 64, 64, fc.Shape(64, 64, 64), 0)
    assert st in (fc.ERR_CUDA, fc.ERR_UNSUPPORTED)


def test_reduce_add_needs_no_workspace(fc):
    """The order-free virtual grid adds every block into the output: no
    partials, so no workspace, and a call without one passes validation
    (here it then fails for want of a GPU, not of workspace)."""
    s = fc.Shape(64, 64, 64, (2, 2, 2))
    f = fc.VGRID | fc.ACCUM_F32
    for op in ("fwd", "dgrad", "wgrad"):
        assert fc.axonn_fc_workspace_size(op, s, f | fc.VGRID_PARTIALS) == 1 * 64 * 64 * 4
        assert fc.axonn_fc_workspace_size(op, s, f) == 0
        assert fc.axonn_fc_workspace_size(op, s, f | fc.REDUCE_ADD) == 0
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _raw(fc, "axonn_fc_fwd", FAKE, FAKE, FAKE, 64, 64, 64, s, f | fc.REDUCE_ADD)
    assert st in (fc.ERR_CUDA, fc.ERR_UNSUPPORTED), fc.axonn_last_error()
    st = _raw(fc, "axonn_fc_fwd", FAKE, FAKE, FAKE, 64, 64, 64, s, f | fc.VGRID_PARTIALS)
    assert st == fc.ERR_WORKSPACE


def test_binding_refuses_missing_library(tmp_path):
    import pmm_fc_layer_gb300 as m
    saved = m._lib
    m._lib = None
    try:
        with pytest.raises(RuntimeError):
            m.load(str(tmp_path / "absent.so"))
    finally:
        m._lib = saved


def test_tune_lookup_checks_arguments_before_the_device(fc):
    """A bad shape is rejected as an argument error; a good one needs the
    device's SM count, so on a host without a GPU the lookup reports a CUDA
    error rather than an answer."""
    import torch
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_tune_lookup("fwd", fc.Shape(-1, 8, 8))
    assert ei.value.status == fc.ERR_INVALID_ARG
    if torch.cuda.is_available():
        pytest.skip("a device is present: the lookup answers")
    with pytest.raises(fc.AxonnError) as ei:
        fc.axonn_tune_lookup("fwd", fc.Shape(8, 8, 8))
    assert ei.value.status == fc.ERR_CUDA


def test_shipped_tuning_tables_cover_their_workloads(fc):
    """Every table shipped in the package loads, and holds exactly one entry
    per GEMM of its workload as the benchmark calls them (single GPU, whole
    operands, default flags) on a 152-SM GB300."""
    import glob
    import json
    import bench
    tables = sorted(glob.glob(os.path.join(ROOT, "pmm_fc_layer_gb300", "tuned", "*.jsonl")))
    assert tables
    for path in tables:
        wl = bench.WORKLOADS[os.path.basename(path)[:-len(".jsonl")]]
        keys = [json.loads(l)["key"] for l in open(path).read().splitlines() if l.strip()]
        grid = "x".join(str(g) for g in wl.get("grid", (1, 1, 1)))
        want = {f"op{fc.OPS[op]}_T{T}_K{K}_N{N}_g{grid}_at0.0.0_f0_sm152"
                for _, T, K, N in wl["layers"] for op in ("fwd", "dgrad", "wgrad")}
        assert sorted(keys) == sorted(want), path
        fc.axonn_tune_cache_clear()
        fc.axonn_tune_cache_load(path)
        assert fc.axonn_tune_cache_size() == len(want)
    fc.axonn_tune_cache_clear()


def test_tune_cache_roundtrip(fc, tmp_path):
    import json
    fc.axonn_tune_cache_clear()
    entries = [
        {"key": "op0_T8_K8_N8_g1x1x1_at0.0.0_f0_sm152", "config": "pair_256x256", "split": 1,
         "group_m": 8, "streamk": 0, "swap": 1, "us": 12.5},
        {"key": "op1_T64_K512_N16_g1x1x1_at0.0.0_f0_sm152", "config": "1cta_128x128",
         "split": 4, "group_m": 16, "streamk": 2, "swap": 0, "us": 3.25},
    ]
    # a line written before the stream-K and swap fields existed loads with
    # the tail on and the roles as given
    legacy = {"key": "op2_T8_K8_N8_g1x1x1_at0.0.0_f0_sm152", "config": "pair_512x256", "split": 1,
              "group_m": -16, "us": 7.0}
    src = tmp_path / "tune.jsonl"
    src.write_text("".join(json.dumps(e) + "\n" for e in entries + [legacy]))
    fc.axonn_tune_cache_load(str(src))
    assert fc.axonn_tune_cache_size() == 3
    out = tmp_path / "saved.jsonl"
    fc.axonn_tune_cache_save(str(out))
    saved = sorted((json.loads(l) for l in out.read_text().splitlines()), key=lambda e: e["key"])
    assert saved == sorted(entries + [dict(legacy, streamk=1, swap=0)], key=lambda e: e["key"])
    # malformed or unknown entries are rejected and leave the table as it was
    bad = tmp_path / "bad.jsonl"
    bad.write_text('{"key": "x", "config": "no_such_config", "split": 1, "group_m": 8, "us": 1}\n')
    with pytest.raises(fc.AxonnError):
        fc.axonn_tune_cache_load(str(bad))
    bad.write_text('{"key": "x", "split": 1}\n')
    with pytest.raises(fc.AxonnError):
        fc.axonn_tune_cache_load(str(bad))
    bad.write_text('{"key": "x", "config": "pair_512x256", "split": 1, "group_m": 8, '
                   '"streamk": 3, "us": 1}\n')
    with pytest.raises(fc.AxonnError):
        fc.axonn_tune_cache_load(str(bad))
    # integers are whole and in range: rasterisation groups of at most 64
    # (a larger one would overflow the kernel's tile walk), splits 1..8
    for field in ('"group_m": 100000', '"group_m": -65', '"group_m": 0', '"group_m": "8x"',
                  '"group_m": 8.5', '"split": 0', '"split": 9', '"split": 99999999999999999999',
                  '"streamk": -1', '"streamk": "1 "', '"swap": 2', '"swap": -1'):
        entry = {"key": "x", "config": "pair_512x256", "split": 1, "group_m": 8, "streamk": 1,
                 "swap": 0, "us": 1}
        name = field.split(":")[0].strip('"')
        line = json.dumps(entry).replace(f'"{name}": {json.dumps(entry[name])}', field)
        assert field in line
        bad.write_text(line + "\n")
        with pytest.raises(fc.AxonnError):
            fc.axonn_tune_cache_load(str(bad))
    ok_line = {"key": "y", "config": "pair_512x256", "split": 8, "group_m": -64, "streamk": 2,
               "us": 1}
    good = tmp_path / "edge.jsonl"
    good.write_text(json.dumps(ok_line) + "\n")
    fc.axonn_tune_cache_load(str(good))
    assert fc.axonn_tune_cache_size() == 4
    fc.axonn_tune_cache_clear()
    fc.axonn_tune_cache_load(str(src))
    with pytest.raises(fc.AxonnError):
        fc.axonn_tune_cache_load(str(tmp_path / "absent.jsonl"))
    assert fc.axonn_tune_cache_size() == 3
    fc.axonn_tune_cache_clear()
    assert fc.axonn_tune_cache_size() == 0


def test_set_swap(fc):
    for mode in (-1, 0, 1, -1):
        fc.axonn_set_swap(mode)
    for bad in (-2, 2):
        with pytest.raises(fc.AxonnError):
            fc.axonn_set_swap(bad)


def test_set_streamk(fc):
    for mode in (-1, 0, 1, -1):
        fc.axonn_set_streamk(mode)
    for bad in (-2, 2):
        with pytest.raises(fc.AxonnError):
            fc.axonn_set_streamk(bad)


def test_zsharded_validation(fc):
    lib = fc.load()
    shards = (ctypes.c_void_p * 2)(FAKE, FAKE)
    # row length not a multiple of 8
    assert lib.axonn_shards_gather(shards, 2, 64, 12, 16, FAKE, 16, 0) == fc.ERR_ALIGNMENT
    # too many shards
    big = (ctypes.c_void_p * 65)(*([FAKE] * 65))
    assert lib.axonn_shards_gather(big, 65, 640, 8, 8, FAKE, 8, 0) == fc.ERR_INVALID_ARG
    # the flag is only for the workspace query of the weight gradient
    s = fc.Shape(64, 64, 64, (2, 2, 2))
    with pytest.raises(fc.AxonnError):
        fc.axonn_fc_workspace_size("fwd", s, fc.ZSHARDED)
    assert fc.axonn_fc_workspace_size("wgrad", s, fc.ZSHARDED) == 1 * 32 * 32 * 4
    assert _raw(fc, "axonn_fc_fwd", FAKE, FAKE, FAKE, 64, 64, 64, fc.Shape(64, 64, 64),
                fc.ZSHARDED) == fc.ERR_INVALID_ARG
    # missing workspace
    st = lib.axonn_fc_wgrad_zsharded(FAKE, FAKE, shards, 64, 64, 32, ctypes.byref(s), 0, 0, 0, 0)
    assert st == fc.ERR_WORKSPACE


def test_l2_budget_setting(fc):
    old = fc.axonn_l2_budget()
    assert old == 64 << 20
    try:
        fc.axonn_set_l2_budget(0)
        assert fc.axonn_l2_budget() == 0
        fc.axonn_set_l2_budget(96 << 20)
        assert fc.axonn_l2_budget() == 96 << 20
        with pytest.raises(fc.AxonnError):
            fc.axonn_set_l2_budget(-1)
        assert fc.axonn_l2_budget() == 96 << 20
    finally:
        fc.axonn_set_l2_budget(old)
