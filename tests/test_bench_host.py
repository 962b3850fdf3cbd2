"""Host logic of the benchmark, on CPU: the reference arm's JSON line, the
argument checks, the peak and clock bookkeeping, and the FLOP accounting
that every reported rate divides."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None, timeout=300):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    p = _run(["--impl", "reference", "--workload", "single_layer_t256", "--steps", "2",
              "--warmup", "3"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert (d["steps"], d["warmup"], d["n_gpus"]) == (2, 3, 1)
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "whole" in cb["sample"]      # a 1.6 GFLOP step is computed in full
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("single_layer_t256")


def test_reference_arm_other_ranks_do_no_work():
    p = _run(["--impl", "reference", "--workload", "single_layer_t256", "--steps", "2",
              "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2"})
    assert p.returncode == 0 and p.stdout.strip() == ""


@pytest.mark.parametrize("args,msg", [
    (["--warmup", "2"], "--warmup must be at least 3"),
    (["--order-free"], "--order-free needs --accum-f32"),
    (["--order-free", "--accum-f32"], "--order-free needs a virtual-grid workload"),
])
def test_argument_checks(args, msg):
    p = _run(args)
    assert p.returncode == 2 and msg in p.stderr


def test_peaks_fallback_and_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_peaks() == {"burst": 1900.0, "sustained": 1700.0, "hbm_gbs": 6800.0,
                                  "source": "fallback"}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1950.5}))
    p = bench.read_peaks()
    assert p["source"] == "measured" and p["burst"] == p["sustained"] == 1950.5
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"bf16_tflops": 1950.5, "bf16_tflops_sustained": 1720.0, "hbm_gbs": 7100}))
    p = bench.read_peaks()
    assert (p["burst"], p["sustained"], p["hbm_gbs"]) == (1950.5, 1720.0, 7100.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.read_peaks()["source"] == "fallback"


def test_clock_summary_keeps_the_timed_window():
    import datetime
    cs = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def row(dt_s, mhz, cap):
        ts = (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (f"{ts}, 0, {mhz}, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, "
                f"{'Active' if cap else 'Not Active'}")

    cs.lines = [row(0.0, 2070, False), row(1.0, 1500, True), row(1.1, 1520, True),
                row(1.2, 1510, False), row(3.0, 2070, False), "garbage"]
    cs.t0 = (base + datetime.timedelta(seconds=0.5)).timestamp()
    cs.t1 = (base + datetime.timedelta(seconds=2.0)).timestamp()
    s = cs.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1510 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    cs.t0 = cs.t1 = (base + datetime.timedelta(seconds=10)).timestamp()
    assert bench.ClockSampler.summary(cs)["window"].startswith("whole sampler run")


def test_gemm_flops_of_the_gpt_block():
    """12 products; 2*M*N*R summed equals 3 ops x 2*T*K*N per layer, 22.27
    TFLOP for H = 6144, T = 8192 (qkv, out, up, down)."""
    wl = bench.WORKLOADS["gpt_h6144_t8192"]
    g = bench.gemms(wl["layers"])
    assert len(g) == 12
    for name, op, T, K, N, M, Nc, R, _ in g:
        assert (M, Nc, R) == {"fwd": (T, N, K), "dgrad": (T, K, N), "wgrad": (K, N, T)}[op]
    flops = sum(2.0 * m * n * r for *_, m, n, r, _ in g)
    closed = sum(3 * 2.0 * T * K * N for _, T, K, N in wl["layers"])
    assert flops == closed
    assert round(flops / 1e12, 2) == 22.27


def test_cpu_rows_whole_small_steps_stripe_large_ones():
    small = bench.gemms(bench.WORKLOADS["single_layer_t256"]["layers"])
    assert bench.cpu_rows(small) == 512          # every row of every GEMM
    for w in ("gpt_h6144_t8192", "large_h16384_t4096", "layout_sweep"):
        assert bench.cpu_rows(bench.gemms(bench.WORKLOADS[w]["layers"])) == bench.CPU_STRIPE_ROWS


def test_config_block_labels():
    c = bench.config_block(bench.WORKLOADS["gpt_h6144_t8192"], "gpt_h6144_t8192", 1)
    assert c["l2"].startswith("operands exceed") and c["grid"] == "1x1x1"
    assert (c["global_batch"], c["seq_len"], c["parallelism"]) == (4, 2048, "single GPU")
    c = bench.config_block(bench.WORKLOADS["single_layer_t256"], "single_layer_t256", 2,
                           output="fp32")
    assert c["l2"].startswith("L2 flushed") and c["parallelism"] == "replicas x2"
    assert c["output"] == "fp32" and c["global_batch"] == 2
    c = bench.config_block(bench.WORKLOADS["gpt_h6144_t8192_vgrid_2x2x2"], "v", 1)
    assert c["grid"] == "2x2x2"
    assert bench.config_block(bench.WORKLOADS["layout_sweep"], "s", 1)["l2"].startswith("mixed")


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_torch_context_products_are_the_ops(op):
    """The cuBLAS context leg computes the same three products (checked here
    with torch's CPU matmul against the oracle, within the parity bound)."""
    import numpy as np
    import torch
    import fc_inputs
    import oracle
    T, K, N = 24, 40, 16
    X = fc_inputs.normal_bf16((T, K), 3, 1)
    W = fc_inputs.normal_bf16((K, N), 3, 2, sigma=0.02)
    dY = fc_inputs.normal_bf16((T, N), 3, 3)
    P, Q = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (X, dY)}[op]
    M, Nn = oracle.out_shape(op, T, K, N)
    C = torch.empty((M, Nn), dtype=torch.bfloat16)
    bench.torch_product(op, fc_inputs.as_torch_bf16(P), fc_inputs.as_torch_bf16(Q), C)
    ref, S = oracle.fc(op, P, Q)
    assert float(oracle.error_ratio(C.to(torch.float64).numpy(), ref, S).max()) <= 1.0


@pytest.mark.parametrize("M,N", [(256, 2048), (8192, 6144), (300, 1000), (1, 1), (33, 65)])
def test_check_bands_cover_every_cell(M, N):
    """The whole-output check's rows and columns put an entry in every 32 x
    64 cell of the output (so in every epilogue warp's rows of every tile)
    and include the first and last row and column."""
    import numpy as np
    I, J = bench.check_bands(M, N, np.random.default_rng(1))
    assert I.min() == 0 and I.max() == M - 1 and J.min() == 0 and J.max() == N - 1
    assert set(range(0, M, 32)) == {32 * (i // 32) for i in I}
    assert set(range(0, N, 64)) == {64 * (j // 64) for j in J}


@pytest.mark.parametrize("planted", [None, "cell", "last_row", "last_col"])
def test_whole_output_check_finds_a_wrong_entry(planted):
    """Fed the oracle's own full product (transposed storages included), the
    check reports ratios of bf16 rounding alone (at most 2^-9 |C| against
    1e-2 S, so below 0.2); with one entry moved well outside the
    bound (in a random 32 x 64 cell, in the last row, or in the last
    column), it reports a ratio above 1."""
    import numpy as np
    import fc_inputs
    import oracle
    layers = [("a", 96, 130, 200)]
    wl = {"layers": layers, "seed": 5}
    data = bench.host_inputs(wl, layers)
    glist = bench.gemms(layers)
    rng = np.random.default_rng(3)
    full = {}
    for gi, (name, op, T, K, N, m, n, r, (pn, qn, _)) in enumerate(glist):
        C, S = oracle.fc(op, data[name][pn], data[name][qn])
        got = oracle.bf16_to_f64(oracle.bf16_rne(C))
        if planted and gi == 1:
            i, j = {"cell": (int(rng.integers(1, m - 1)), int(rng.integers(1, n - 1))),
                    "last_row": (m - 1, int(rng.integers(0, n))),
                    "last_col": (int(rng.integers(0, m)), n - 1)}[planted]
            # a wrong entry in every 32 x 64 cell of the row band and column
            # band of (i, j): the check samples one row per band
            got[32 * (i // 32): 32 * (i // 32) + 32, 64 * (j // 64): 64 * (j // 64) + 64] += \
                1.0 + 0.1 * S[32 * (i // 32): 32 * (i // 32) + 32, 64 * (j // 64): 64 * (j // 64) + 64]
        full[gi] = got
    outputs = {gi: (lambda g: (lambda ri, cj: g[np.ix_(ri, cj)]))(full[gi]) for gi in full}
    worst, entries = bench.whole_output_check(data, glist, outputs)
    assert entries > 0
    if planted:
        assert worst > 1.0
    else:
        assert worst < 0.2


def test_traffic_reported_only_for_captured_choices(monkeypatch):
    """roofline.traffic is the captured DRAM bytes of the step's GEMMs when
    every GEMM ran a choice in the committed table (and the kernel sources
    are the capture's); any other choice, source or workload gives null."""
    # one captured choice per GEMM of the step (the table may hold several)
    first = {}
    for (gemm, choice), b in bench.TRAFFIC["bytes"].items():
        first.setdefault(gemm, (choice, b))
    assert len(first) == 12
    per = []
    for gemm, (choice, _) in first.items():
        layer, op = gemm.split(":")
        config, group, sk, swap = choice.split("/")
        per.append({"layer": layer, "op": op, "config": config, "group_m": int(group),
                    "streamk_tiles": int(sk), "swap": int(swap)})
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: bench.TRAFFIC["kernel_sources"])
    want = sum(b for _, b in first.values()) / 12
    assert bench.traffic_per_launch("gpt_h6144_t8192", per, None) == pytest.approx(want)
    assert bench.traffic_per_launch("gpt_h6144_t8192", per, ("up", "fwd")) is None
    assert bench.traffic_per_launch("large_h16384_t4096", per, None) is None
    other = [dict(p) for p in per]
    other[0]["group_m"] = 99
    assert bench.traffic_per_launch("gpt_h6144_t8192", other, None) is None
    # the same configuration with the operand roles exchanged is another choice
    flipped = [dict(p) for p in per]
    flipped[0]["swap"] = 1 - flipped[0]["swap"]
    if (f"{flipped[0]['layer']}:{flipped[0]['op']}",
            "/".join(str(flipped[0][k]) for k in ("config", "group_m", "streamk_tiles", "swap"))) \
            not in bench.TRAFFIC["bytes"]:
        assert bench.traffic_per_launch("gpt_h6144_t8192", flipped, None) is None
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "0" * 16)
    assert bench.traffic_per_launch("gpt_h6144_t8192", per, None) is None


def test_kernel_hash_follows_code_not_comments():
    """The traffic table is tied to the kernels' code: comments and layout
    leave the hash alone, a changed token does not."""
    a = "int f(int x) {  // doubles x\n  return 2 * x; /* fast\n path */ }\n"
    b = "int f(int x) {\n    return 2 * x;\n}  // another note\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench.code_text(a) == bench.code_text(b) == "int f(int x) { return 2 * x; }"
    assert bench.code_text(c) != bench.code_text(a)
    assert len(bench.kernel_sources_hash()) == 16


def test_shipped_table_choices_have_captured_traffic():
    """The default line runs the tuning table shipped for its workload; each
    of its choices has captured DRAM bytes in the traffic table, so the
    line reports roofline.traffic (a retuned table needs a new capture)."""
    import json
    path = os.path.join(bench.TUNED_DIR, f"{bench.DEFAULT_WORKLOAD}.jsonl")
    entries = [json.loads(l) for l in open(path).read().splitlines() if l.strip()]
    assert len(entries) == 12
    names = {0: "fwd", 1: "dgrad", 2: "wgrad"}
    layers = {(T, K, N): name for name, T, K, N in bench.WORKLOADS[bench.DEFAULT_WORKLOAD]["layers"]}
    for e in entries:
        key = e["key"]
        op = int(key.split("_")[0][2:])
        T, K, N = (int(key.split("_")[i][1:]) for i in (1, 2, 3))
        gemm = f"{layers[(T, K, N)]}:{names[op]}"
        # the stream-K tiles of a choice are fixed by its mode and the shape;
        # every capture of this GEMM in this configuration, group and roles
        # is listed with the tiles it ran
        prefix = f"{e['config']}/{e['group_m']}/"
        suffix = f"/{e['swap']}"
        assert any(g == gemm and c.startswith(prefix) and c.endswith(suffix)
                   for (g, c) in bench.TRAFFIC["bytes"]), (gemm, e)
