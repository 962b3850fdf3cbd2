#!/usr/bin/env python
"""Benchmark of the FC-layer GEMMs of a GPT block on GB300.

A step is one pass of the whole path over one batch.  For each FC layer of
the workload it computes the forward product Y = X.W, the data gradient
dX = dY.W^T and the weight gradient dW = X^T.dY, all through the C ABI of
libaxonn_fc.so.  The default workload, on which the metric is quoted, is a GPT
block with hidden size H = 6144 and T = 8192 tokens (batch 4 x sequence 2048).
Its four layers are QKV [H -> 3H], attention-out [H -> H], MLP-up [H -> 4H]
and MLP-down [4H -> H], for 12 GEMM launches per step.  `--workload` selects
the other FC workloads: the single small layer, the 3D-grid shards on a
virtual grid, the hidden-16384 model and the layout sweep.

Inputs are seeded synthetic bf16: activations and gradients ~N(0,1), weights
~N(0,0.02), and the sweep N(0,1)*0.05.  Every large GEMM's operands exceed the
129 MB L2.  The small single-layer workload flushes L2 between timed steps by
writing a 512 MB buffer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--config C]

Rank 0 prints one JSON line.  Under torchrun with N > 1, every rank runs an
independent replica on its own GPU; the path needs no collective when each
rank has its own GPU.  The value is then the total over ranks divided by the
slowest rank's time.  `--impl reference` times the fp64 CPU oracle on the
host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOP/s per FC GEMM (fwd/dgrad/wgrad) and % of GB300 dense bf16 peak, 1 GPU"
UNIT = "TFLOP/s"
CPU_STRIPE_ROWS = 64      # output rows of every GEMM the CPU oracle computes per sample
CPU_FULL_STEP_FLOPS = 50e9  # steps up to this size are computed whole by the CPU oracle
L2_FLUSH_BYTES = 512 << 20


def _gpt(H, T, mlp):
    return [("qkv", T, H, 3 * H), ("out", T, H, H), ("up", T, H, mlp), ("down", T, mlp, H)]


SWEEP_DIMS = (1000, 4096, 5000, 12288)
WORKLOADS = {
    "gpt_h6144_t8192": dict(
        desc="GPT block FC layers, H=6144, T=8192 (batch 4 x seq 2048): qkv [H->3H], "
             "out [H->H], up [H->4H], down [4H->H]; fwd+dgrad+wgrad each, full layers",
        layers=_gpt(6144, 8192, 4 * 6144), batch=4, seq=2048, seed=1002),
    "single_layer_t256": dict(
        desc="single FC layer X[256x512] W[512x2048], grid 1x1x1; L2 flushed between steps",
        layers=[("fc", 256, 512, 2048)], batch=1, seq=256, seed=1001, flush=True),
    "single_layer_t256_warm": dict(
        desc="single FC layer X[256x512] W[512x2048], grid 1x1x1; operands L2-resident (warm)",
        layers=[("fc", 256, 512, 2048)], batch=1, seq=256, seed=1001),
    "gpt_h6144_t8192_vgrid_2x2x2": dict(
        desc="GPT block H=6144, T=8192 as a virtual 2x2x2 grid of 3D-PMM block products "
             "(T by Gz, K by Gx, N by Gy), partials summed on device",
        layers=_gpt(6144, 8192, 4 * 6144), batch=4, seq=2048, seed=1003, grid=(2, 2, 2)),
    "large_h16384_t4096": dict(
        desc="large-model FC layers, hidden 16384, MLP 53248, T=4096: qkv [16384->18432], "
             "out [16384->16384], up [16384->53248], down [53248->16384]; full layers",
        layers=[("qkv", 4096, 16384, 18432), ("out", 4096, 16384, 16384),
                ("up", 4096, 16384, 53248), ("down", 4096, 53248, 16384)],
        batch=2, seq=2048, seed=1004),
    "large_h16384_t4096_vgrid_1x4x4": dict(
        desc="large-model FC layers (hidden 16384, MLP 53248, T=4096) as a virtual 1x4x4 "
             "grid (T_blk=1024), partials summed on device",
        layers=[("qkv", 4096, 16384, 18432), ("out", 4096, 16384, 16384),
                ("up", 4096, 16384, 53248), ("down", 4096, 53248, 16384)],
        batch=2, seq=2048, seed=1004, grid=(1, 4, 4)),
    "layout_sweep": dict(
        desc="layout/shape sweep: T in {512,2048,8192,16384} x K,N in {1000,4096,5000,12288}, "
             "NN (fwd) / NT (dgrad) / TN (wgrad), values N(0,1)*0.05",
        layers=[(f"T{T}_K{K}_N{N}", T, K, N) for T in (512, 2048, 8192, 16384)
                for K in SWEEP_DIMS for N in SWEEP_DIMS],
        batch=None, seq=None, seed=1005, scale=0.05, device_inputs=True),
}
DEFAULT_WORKLOAD = "gpt_h6144_t8192"
# Tuning tables shipped for workloads (<workload>.jsonl, the library's tune
# cache format): choices from a tuning run on a GB300, keyed by SM count.
TUNED_DIR = os.path.join(ROOT, "pmm_fc_layer_gb300", "tuned")

# DRAM traffic of the GEMM kernel from ncu captures of the default workload:
# dram__bytes_read.sum + dram__bytes_write.sum of each GEMM ("layer:op") in
# each tuned choice ("config/group/stream-K tiles/swap") captured (summary and command
# in profiles/).  Reported only while the kernel sources hash to the value
# the capture was taken with and every GEMM's choice of this run is in it.
TRAFFIC = {
    "workload": "gpt_h6144_t8192", "kernel_sources": "17f9e09df4a99f33",
    "bytes": {
        ("qkv:fwd", "pair_512x256/-8/88/0"): 2033709568,
        ("qkv:fwd", "pair_512x256/16/88/0"): 2480573696,
        ("qkv:dgrad", "1cta_256x192/-8/0/0"): 1863450112,
        ("qkv:dgrad", "1cta_256x192/16/0/0"): 1770873344,
        ("qkv:wgrad", "pair_512x256/-16/104/0"): 2358818816,
        ("qkv:wgrad", "pair_512x256/16/0/0"): 1756339200,
        ("out:fwd", "1cta_256x192/-8/0/0"): 612682411,
        ("out:dgrad", "1cta_256x192/-8/0/0"): 598803883,
        ("out:wgrad", "pair_512x256/-8/0/0"): 573971072,
        ("out:wgrad", "pair_512x256/16/0/1"): 569758464,
        ("up:fwd", "1cta_256x192/16/0/0"): 2034324480,
        ("up:fwd", "pair_512x256/16/0/1"): 3029764864,
        ("up:fwd", "pair_512x256/16/92/0"): 3113689600,
        ("up:dgrad", "1cta_256x192/-8/0/0"): 2458654720,
        ("up:dgrad", "1cta_256x192/16/0/0"): 2353478144,
        ("up:dgrad", "1cta_256x192/8/0/0"): 2313691136,
        ("up:wgrad", "pair_512x256/16/88/0"): 2767284096,
        ("up:wgrad", "pair_512x256/8/88/0"): 2247602176,
        ("down:fwd", "1cta_256x192/16/0/0"): 2343909120,
        ("down:fwd", "1cta_256x192/8/0/0"): 2312553728,
        ("down:fwd", "pair_512x256/8/80/1"): 3004876288,
        ("down:dgrad", "1cta_256x192/16/0/0"): 2037140864,
        ("down:dgrad", "pair_512x256/16/92/0"): 3128448768,
        ("down:wgrad", "pair_512x256/-16/88/0"): 2537176064,
    }}


def traffic_per_launch(workload, per, only):
    """Mean DRAM bytes per GEMM launch of the step from the captured table,
    or None when a GEMM's choice (or the kernel sources) was not captured."""
    if workload != TRAFFIC["workload"] or only is not None or not per:
        return None
    if kernel_sources_hash() != TRAFFIC["kernel_sources"]:
        return None
    tot = 0.0
    for p in per:
        key = (f"{p['layer']}:{p['op']}",
               f"{p['config']}/{p['group_m']}/{p['streamk_tiles']}/{int(p.get('swap', 0))}")
        if key not in TRAFFIC["bytes"]:
            return None
        tot += TRAFFIC["bytes"][key]
    return tot / len(per)


def code_text(src):
    """C++ source with comments removed and whitespace collapsed: the part
    of a file that decides what the compiler builds."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_sources_hash():
    """Hash of the GEMM kernels' code (comments and layout ignored)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm_kernel.cuh", "gemm_pair_kernel.cuh", "ptx.cuh", "kernel_instances.cuh"):
        with open(os.path.join(ROOT, "pmm_fc_layer_gb300", "csrc", name)) as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]
DATA = ("synthetic, seeded: SplitMix64 + Box-Muller bf16; activations/grads N(0,1), "
        "weights N(0,0.02)")


def gemms(layers):
    """The products of one step: (layer, op, T, K, N, M, Ncols, R, tensor names)."""
    out = []
    for name, T, K, N in layers:
        out.append((name, "fwd", T, K, N, T, N, K, ("X", "W", "Y")))
        out.append((name, "dgrad", T, K, N, T, K, N, ("dY", "W", "dX")))
        out.append((name, "wgrad", T, K, N, K, N, T, ("X", "dY", "dW")))
    return out


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"burst": float(d["bf16_tflops"]),
                "sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d.get("hbm_gbs", 6800.0)),
                "source": "measured"}
    except (OSError, KeyError, ValueError, TypeError):
        return {"burst": 1900.0, "sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ inputs
def host_inputs(wl, layers):
    """Seeded bf16 bits of the layers' X, W and dY (numpy uint16)."""
    import fc_inputs
    scale = wl.get("scale")
    data = {}
    names = [l[0] for l in wl["layers"]]
    for name, T, K, N in layers:
        tid = 16 * (names.index(name) + 1)
        data[name] = {
            "X": fc_inputs.normal_bf16((T, K), wl["seed"], tid + 1, sigma=scale or 1.0),
            "W": fc_inputs.normal_bf16((K, N), wl["seed"], tid + 2, sigma=scale or 0.02),
            "dY": fc_inputs.normal_bf16((T, N), wl["seed"], tid + 3, sigma=scale or 1.0),
        }
    return data


def device_inputs(wl, layers, dev):
    """Seeded bf16 operands drawn on the device (for workloads too large to
    draw on the host in a benchmark run), with the workload's distributions:
    activations and gradients N(0,1), weights N(0,0.02), or every operand
    N(0,1) times the workload's scale."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(wl["seed"])
    scale = wl.get("scale")
    out = {}
    for name, T, K, N in layers:
        out[name] = {k: (torch.randn(shape, generator=g, device=dev)
                         * (scale or (0.02 if k == "W" else 1.0))).to(torch.bfloat16)
                     for k, shape in (("X", (T, K)), ("W", (K, N)), ("dY", (T, N)))}
    return out


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region.
    Samples are timestamped; only those taken between entering and leaving
    the `with` block count (the sampler starts before and stops after it, so
    samples at either edge would see an idle GPU)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        import datetime
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = {name for r in use for name, val in zip(self.NAMES, r[3])
                   if val.lower().startswith("active")}
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "samples": len(use),
                "window": "timed region" if inside else "whole sampler run (no sample fell inside)"}


# ------------------------------------------------------------------ CPU oracle
def oracle_stripes(data, glist, which, rows, gpu_rows=None):
    """fp64 oracle on the first `rows` output rows of the listed GEMMs;
    returns (flops, seconds, threads used, worst error ratio).  With
    `gpu_rows` (GEMM index -> float64 array of the GPU's first `rows`
    output rows) the oracle's stripe is also compared with the GPU's:
    worst |C - C_ref| / (1e-2 * |A|.|B| + 1e-5), which must be <= 1."""
    import oracle
    flops, secs, worst = 0.0, 0.0, 0.0
    for gi in which:
        name, op, T, K, N, m, n, r, (pn, qn, _) = glist[gi]
        d = data[name]
        if op == "wgrad":
            P = d[pn][:, :rows]        # X[:, k-stripe] -> rows of dW
        else:
            P = d[pn][:rows]
        Q = d[qn]
        t0 = time.perf_counter()
        C, S = oracle.fc(op, P, Q)
        secs += time.perf_counter() - t0
        flops += 2.0 * min(rows, m) * n * r
        if gpu_rows is not None and gi in gpu_rows:
            worst = max(worst, float(oracle.error_ratio(gpu_rows[gi], C, S).max()))
    return flops, secs, min(oracle.max_threads(), rows), worst


def check_bands(M, N, rng, row_band=32, col_band=64):
    """Rows and columns of the whole-output check: rows 0 and M-1 plus one
    seeded random row in every `row_band`-row band, columns 0 and N-1 plus
    one random column in every `col_band`-column band.  Their cross product
    puts an entry in every 32 x 64 cell of the output, so every output tile
    of every kernel configuration (at least 128 x 128) is checked on the rows
    of each of its epilogue warps (32 rows each), stream-K tiles included."""
    import numpy as np
    rows = [0, M - 1] + [b + int(rng.integers(0, min(row_band, M - b)))
                         for b in range(0, M, row_band)]
    cols = [0, N - 1] + [b + int(rng.integers(0, min(col_band, N - b)))
                         for b in range(0, N, col_band)]
    return np.unique(np.array(rows, np.int64)), np.unique(np.array(cols, np.int64))


def _rows_of(view, t, idx):
    """Stored copy of logical rows `idx` of an operand stored transposed if t."""
    import numpy as np
    return np.ascontiguousarray(view[:, idx] if t else view[idx, :])


def _cols_of(view, t, idx):
    """Stored copy of logical columns `idx` of an operand stored transposed if t."""
    import numpy as np
    return np.ascontiguousarray(view[idx, :] if t else view[:, idx])


def whole_output_check(data, glist, outputs, seed=7):
    """The GPU's outputs of the timed steps against the fp64 oracle over the
    whole output of every GEMM: full rows 0 and M-1, full columns 0 and
    N-1, and the cross product of one random row per 32-row band with one
    random column per 64-column band (see check_bands).  `outputs` maps a
    GEMM index to a function (rows, cols) -> float64 array of the GPU's
    output there.  Returns the worst |C - C_ref| / (1e-2 |A|.|B| + 1e-5)
    and the number of entries checked."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    worst, entries = 0.0, 0
    for gi, (name, op, T, K, N, m, n, r, (pn, qn, _)) in enumerate(glist):
        A, a_t, B, b_t = oracle.operands(op, data[name][pn], data[name][qn], False, False)
        I, J = check_bands(m, n, rng)
        full_i = np.array(sorted({0, m - 1}), np.int64)
        full_j = np.array(sorted({0, n - 1}), np.int64)
        all_j, all_i = np.arange(n, dtype=np.int64), np.arange(m, dtype=np.int64)
        for ri, cj, Ablk, Bblk in ((I, J, _rows_of(A, a_t, I), _cols_of(B, b_t, J)),
                                   (full_i, all_j, _rows_of(A, a_t, full_i), B),
                                   (all_i, full_j, A, _cols_of(B, b_t, full_j))):
            C, S = oracle.gemm(Ablk, a_t, Bblk, b_t)
            got = outputs[gi](ri, cj)
            worst = max(worst, float(oracle.error_ratio(got, C, S).max()))
            entries += C.size
    return worst, entries


def cpu_rows(glist):
    """Output rows per GEMM that the CPU oracle computes: every row when the
    whole step is small (a few seconds on the host), else a stripe."""
    full = sum(2.0 * m * n * r for _, _, _, _, _, m, n, r, _ in glist)
    if full <= CPU_FULL_STEP_FLOPS:
        return max(m for _, _, _, _, _, m, _, _, _ in glist)
    return CPU_STRIPE_ROWS


def cpu_baseline(data, glist, gpu_rows=None, rows=CPU_STRIPE_ROWS):
    flops, secs, cores, worst = oracle_stripes(data, glist, range(len(glist)), rows, gpu_rows)
    full = sum(2.0 * m * n * r for _, _, _, _, _, m, n, r, _ in glist)
    whole = flops >= full
    what = (f"the whole step, every output row of the {len(glist)} GEMMs" if whole else
            f"first {rows} output rows of each of the {len(glist)} GEMMs")
    out = {"value": flops / secs / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{what} ({flops / 1e9:.1f} GFLOP, {secs:.1f} s)"}
    if not whole:
        out["full_step_s_extrapolated"] = round(full / (flops / secs), 1)
    if gpu_rows is not None:
        out["max_error_ratio"] = worst
        out["error_bound"] = ("|C - C_ref| <= 1e-2 * (|A|.|B|) + 1e-5 on "
                              + ("every output element" if whole else "the sampled rows"))
    return out


STEP_TIMING = {
    1: "one step per graph replay, CUDA events around each step",
    0: "the K timed steps back to back in one CUDA graph, CUDA events around the "
       "span (steps of a few microseconds with L2-resident operands)"}


def config_block(wl, name, world, output=None, reps=1):
    cfg = {"workload": f"{name}: {wl['desc']}"}
    if output:
        cfg["output"] = output
    if wl.get("batch"):
        cfg.update(global_batch=wl["batch"] * world, seq_len=wl["seq"])
    cfg["grid"] = "x".join(str(g) for g in wl.get("grid", (1, 1, 1)))
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    big = [2 * (T * K + K * N + T * N) > (129 << 20) for _, T, K, N in wl["layers"]]
    cfg["l2"] = ("L2 flushed between timed steps (512 MB write)" if wl.get("flush")
                 else "operands exceed the 129 MB L2; no flush" if all(big)
                 else "operands L2-resident (warm), by design of this workload" if not any(big)
                 else "mixed: the larger shapes exceed L2, the smallest can stay resident")
    cfg["step_timing"] = STEP_TIMING[1 if reps == 1 else 0]
    return cfg


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    # Rank 0 runs alone on the host: every core, also where the launcher set
    # OMP_NUM_THREADS=1 for each of its processes.
    oracle.set_threads(os.cpu_count() or 1)
    wl = WORKLOADS[args.workload]
    if wl.get("device_inputs"):
        layers = wl["layers"][:: max(1, len(wl["layers"]) // 8)]
    else:
        layers = wl["layers"]
    data = host_inputs(wl, layers)
    glist = gemms(layers)
    n = len(glist)
    rows = cpu_rows(glist)
    for s in range(args.warmup):
        oracle_stripes(data, glist, [s % n], rows)
    tot_f, tot_s, cores = 0.0, 0.0, 1
    for s in range(args.steps):
        f, sec, cores, _ = oracle_stripes(data, glist, [s % n], rows)
        tot_f += f
        tot_s += sec
    value = tot_f / tot_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
            "config": {**config_block(wl, args.workload, 1),
                       "parallelism": "host cores (OpenMP)",
                       "step_timing": "host wall clock around each step's oracle products"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": ("each step: one of the " + str(n) + " GEMMs, whole"
                                        if rows != CPU_STRIPE_ROWS else
                                        f"each step: first {rows} output rows of one of the "
                                        f"{n} GEMMs")
                                       + ", cycling through them"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def torch_product(op, P, Q, C):
    """The op through torch.matmul (cuBLAS on a GPU), written into C: the
    context leg's products.  P, Q are the op's stored operands (X, W for
    fwd; dY, W for dgrad; X, dY for wgrad), untransposed."""
    import torch
    if op == "fwd":
        torch.matmul(P, Q, out=C)
    elif op == "dgrad":
        torch.matmul(P, Q.t(), out=C)
    else:
        torch.matmul(P.t(), Q, out=C)
    return C


def max_over_ranks(value, device):
    """The largest `value` over all ranks of the default process group (the
    slowest rank's time); `value` itself when there is no group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ GPU arm
def measure(wl_name, args, fc, dev, world, local, steps, tune_cache=None, on_device=False):
    """Times one GEMM workload: inputs, per-shape tuning, warm-up, then
    `steps` CUDA-graph replays of a step (or eager steps with --no-graph)
    and of each GEMM alone, with clocks sampled over the timed region.
    Returns the state the caller reports from (a namespace)."""
    import types

    import torch
    import torch.distributed as dist

    import fc_inputs
    only = tuple(args.only.split(":")) if args.only and wl_name == args.workload else None
    wl = WORKLOADS[wl_name]
    grid = wl.get("grid", (1, 1, 1))
    flags = fc.VGRID if grid != (1, 1, 1) else 0
    if args.accum_f32:
        flags |= fc.ACCUM_F32
    if args.order_free:
        flags |= fc.REDUCE_ADD
    if args.vgrid_partials:
        flags |= fc.VGRID_PARTIALS
    out_dtype = torch.float32 if args.accum_f32 else torch.bfloat16
    layers = [l for l in wl["layers"] if only is None or l[0] == only[0]]
    if args.shrink > 1 and wl_name == args.workload:
        # a smaller case of the same kernels for profiling (not a bench line)
        layers = [(n, max(8, T // args.shrink // 8 * 8), max(8, K // args.shrink // 8 * 8),
                   max(8, N // args.shrink // 8 * 8)) for n, T, K, N in layers]
    glist = [g for g in gemms(layers) if only is None or (g[0], g[1]) == only]

    data = None
    if wl.get("device_inputs") or on_device:
        dbuf = device_inputs(wl, layers, dev)
    else:
        data = host_inputs(wl, layers)
        dbuf = {name: {k: fc_inputs.as_torch_bf16(v, dev) for k, v in data[name].items()}
                for name in data}
    for name, T, K, N in layers:
        dbuf[name]["Y"] = torch.zeros((T, N), dtype=out_dtype, device=dev)
        dbuf[name]["dX"] = torch.zeros((T, K), dtype=out_dtype, device=dev)
        dbuf[name]["dW"] = torch.zeros((K, N), dtype=out_dtype, device=dev)

    plan = []
    ws_need = 0
    for name, op, T, K, N, m, n, r, (pn, qn, cn) in glist:
        shape = fc.Shape(T, K, N, grid)
        ws_need = max(ws_need, fc.axonn_fc_workspace_size(op, shape, flags))
        plan.append(dict(name=name, op=op, flops=2.0 * m * n * r, mnr=(m, n, r),
                         P=dbuf[name][pn], Q=dbuf[name][qn], C=dbuf[name][cn], shape=shape,
                         bytes=2.0 * (m * r + r * n) + (8.0 if args.accum_f32 else 2.0) * m * n))
    ws = torch.empty(ws_need, dtype=torch.uint8, device=dev) if ws_need else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if wl.get("flush") else None
    stream = torch.cuda.Stream(device=dev)
    used = [None] * len(plan)
    # the two-launch virtual-grid sum is a second launch per GEMM whose
    # reduced grid axis has more than one block; the chained and the
    # order-free ones are not
    reduce_launches = sum(1 for g in glist
                          if (flags & fc.VGRID) and (flags & fc.VGRID_PARTIALS)
                          and {"fwd": grid[0], "dgrad": grid[1], "wgrad": grid[2]}[g[1]] > 1)

    sk_tiles = [0] * len(plan)

    swapped = [0] * len(plan)

    def call_gemm(gi):
        g = plan[gi]
        fc.call(g["op"], g["P"], g["Q"], g["C"], g["shape"], flags, ws, stream=stream)
        used[gi] = fc.axonn_last_choice()
        sk_tiles[gi] = fc.axonn_last_streamk_tiles()
        swapped[gi] = fc.axonn_last_swap()

    def step(events=None):
        for gi in range(len(plan)):
            if events is not None:
                events[gi][0].record(stream)
            call_gemm(gi)
            if events is not None:
                events[gi][1].record(stream)

    # Per-shape tuning (outside every timed region): each GEMM's candidate
    # configurations are timed once and the fastest is kept by the library.
    # A workload with a tuning table shipped in the package loads it first
    # (unless --retune) and tunes only the GEMMs it holds no entry for.
    tuning = "none: default choices"
    if tune_cache and os.path.exists(tune_cache):
        fc.axonn_tune_cache_load(tune_cache)
        tuning = f"loaded from {tune_cache}"
    elif not args.no_tune:
        shipped = os.path.join(TUNED_DIR, f"{wl_name}.jsonl")
        if not args.retune and os.path.exists(shipped):
            fc.axonn_tune_cache_load(shipped)
        todo = [g for g in plan if not fc.axonn_tune_lookup(g["op"], g["shape"], flags)]
        with torch.cuda.stream(stream):
            for g in todo:
                fc.axonn_fc_tune(g["op"], g["P"], g["Q"], g["C"], g["shape"], flags, ws,
                                 stream=stream)
        tuning = ("tuned at run time" if len(todo) == len(plan) else
                  f"shipped table {os.path.relpath(shipped, ROOT)}" if not todo else
                  f"shipped table, {len(todo)} of {len(plan)} GEMMs tuned at run time")
        if tune_cache:
            fc.axonn_tune_cache_save(tune_cache)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
            if flush is not None:
                flush.fill_(1)
    fc.axonn_sync_status(stream)

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in plan]
          for _ in range(steps)]
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    gpu_index = int(vis) if vis.isdigit() else local
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # Steps of a few microseconds (the single layer) with L2-resident
    # operands: the K timed steps run back to back from one graph and are
    # timed as one span, as consecutive layers would run in a model step;
    # one graph launch per step would put its launch latency (several us,
    # larger than such a GEMM) into every step.  Flushed and large steps are
    # timed one step per replay.
    batched = (not args.no_graph) and flush is None and \
        sum(g["flops"] for g in plan) < 2e10
    reps = steps if batched else 1
    if not args.no_graph:
        # One step (or K), and each GEMM on its own (or K times), captured as
        # CUDA graphs: the timed loops replay them, so host-side launch
        # overhead (which dominates the small products) is not part of the
        # device timeline.
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=stream):
            for _ in range(reps):
                step()
        gemm_graphs = []
        for gi in range(len(plan)):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=stream):
                for _ in range(reps):
                    call_gemm(gi)
            gemm_graphs.append(gg)
        with torch.cuda.stream(stream):
            step_graph.replay()
            for gg in gemm_graphs:
                gg.replay()
        torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clocks:
        with torch.cuda.stream(stream):
            for s in range(steps // reps):
                step_ev[s][0].record(stream)
                if args.no_graph:
                    step(ev[s])
                else:
                    step_graph.replay()
                step_ev[s][1].record(stream)
                if flush is not None:
                    flush.fill_(1)        # outside the step's events
            if not args.no_graph:
                for gi, gg in enumerate(gemm_graphs):
                    for s in range(steps // reps):
                        ev[s][gi][0].record(stream)
                        gg.replay()
                        ev[s][gi][1].record(stream)
                        if flush is not None:
                            flush.fill_(1)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    fc.axonn_sync_status(stream)
    elapsed_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in step_ev[:steps // reps]), dev)
    # the counter-zeroing kernel before a stream-K call (a split reduction
    # is one launch)
    sk_zeroing = sum(1 for t in sk_tiles if t > 0)
    # timed steps, plus (with graphs) the per-GEMM replays
    launches = (steps * (len(plan) + reduce_launches + sk_zeroing)
                * (1 if args.no_graph else 2))

    peaks = read_peaks()
    per = []
    gemm_ms_total = 0.0
    flops_per_step = sum(g["flops"] for g in plan)
    for gi, g in enumerate(plan):
        if reps > 1:   # one span of K back-to-back calls: K equal shares
            ms = [ev[0][gi][0].elapsed_time(ev[0][gi][1]) / reps] * steps
        else:
            ms = [ev[s][gi][0].elapsed_time(ev[s][gi][1]) for s in range(steps)]
        gemm_ms_total += sum(ms)
        med = statistics.median(ms)
        # the pages' own style: the mean of the last 8 of 10 runs
        last8 = statistics.mean(ms[2:10]) if len(ms) >= 10 else None
        tf = g["flops"] / med / 1e9
        gbs = g["bytes"] / med / 1e6
        m, n, r = g["mnr"]
        per.append({"layer": g["name"], "op": g["op"], "M": m, "N": n, "R": r,
                    "layout": {"fwd": "NN", "dgrad": "NT", "wgrad": "TN"}[g["op"]],
                    "ms": round(med, 4), "tflops": round(tf, 1),
                    "frac_of_sustained": round(tf / peaks["sustained"], 4),
                    "frac_of_burst": round(tf / peaks["burst"], 4),
                    "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "mean_last8_of_10_ms": round(last8, 4) if last8 is not None else None,
                    "config": fc.axonn_kernel_config_name(used[gi][0]),
                    "split": used[gi][1], "group_m": used[gi][2],
                    "streamk_tiles": sk_tiles[gi], "swap": swapped[gi]})
    # Exchanged operand roles, forced off and on, each GEMM in its tuned
    # configuration otherwise (a comparison, after the timed region).
    if getattr(args, "swap_compare", False) and not args.no_graph:
        for mode in (0, 1):
            fc.axonn_set_swap(mode)
            for gi in range(len(plan)):
                gg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gg, stream=stream):
                    call_gemm(gi)
                applied = swapped[gi]
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    gg.replay()
                    e0.record(stream)
                    for _ in range(5):
                        gg.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                per[gi][f"ms_swap{mode}"] = round(e0.elapsed_time(e1) / 5, 4)
                if mode == 1:
                    per[gi]["swap_applies"] = applied
        fc.axonn_set_swap(-1)
        fc.axonn_sync_status(stream)

    # The dominant kernel's rate: with graphs the timed step is nothing but
    # this library's GEMM launches back to back, so the step's device time is
    # their summed duration; eagerly, the sum of the per-call events.
    if args.no_graph:
        achieved = flops_per_step * steps / (gemm_ms_total * 1e9)
    else:
        achieved = flops_per_step * steps / (elapsed_ms * 1e9)

    return types.SimpleNamespace(**{k: v for k, v in locals().items() if k != "types"})


def sampled_check(m, fc, row_band=256, col_band=512, seed=11):
    """A lighter whole-output check for the workloads object: every GEMM of
    the step at one random row per `row_band` rows x one random column per
    `col_band` columns (plus the first and last row and column), against the
    fp64 oracle.  Operand rows and columns are copied from the device
    tensors the GEMMs read (the seeded inputs), so workloads drawn on the
    device are covered too.  Returns (worst error ratio, entries)."""
    import numpy as np
    import torch

    import fc_inputs
    import oracle
    rng = np.random.default_rng(seed)
    worst, entries = 0.0, 0
    for g in m.plan:
        A, a_t, B, b_t = oracle.operands(g["op"], g["P"], g["Q"], False, False)
        M, N, _ = g["mnr"]
        # finer bands on small outputs: at least 16 x 16 sampled rows x columns
        I, J = check_bands(M, N, rng, min(row_band, max(32, M // 16)),
                           min(col_band, max(64, N // 16)))
        ii = torch.from_numpy(I).to(A.device)
        jj = torch.from_numpy(J).to(A.device)
        Ab = fc_inputs.from_torch_bf16(A.index_select(1 if a_t else 0, ii))
        Bb = fc_inputs.from_torch_bf16(B.index_select(0 if b_t else 1, jj))
        C, S = oracle.gemm(Ab, a_t, Bb, b_t)
        got = g["C"].index_select(0, ii).index_select(1, jj).to(torch.float64).cpu().numpy()
        if m.flags & fc.ACCUM_F32:
            continue      # accumulated outputs hold every step's sum
        worst = max(worst, float(oracle.error_ratio(got, C, S).max()))
        entries += C.size
    return worst, entries


def workload_summary(m, fc, check=True):
    """One entry of the `workloads` object: the step's rate and fractions,
    the clocks, and for shapes below the ridge point the HBM rate."""
    peaks = m.peaks
    tf = m.flops_per_step * m.steps / (m.elapsed_ms * 1e9)
    ridge = peaks["burst"] * 1e12 / (peaks["hbm_gbs"] * 1e9)   # FLOP per byte
    mem = [p for p in m.per if 2.0 * p["M"] * p["N"] * p["R"] / (
        2.0 * (p["M"] * p["R"] + p["R"] * p["N"] + p["M"] * p["N"])) < ridge]
    out = {"tflops": round(tf, 2), "frac_of_burst": round(tf / peaks["burst"], 4),
           "frac_of_sustained": round(tf / peaks["sustained"], 4),
           "ms_per_step": round(m.elapsed_ms / m.steps, 4), "gemms": len(m.plan),
           "steps": m.steps, "sm_mhz": m.clocks.summary().get("sm_mhz"),
           "clock_reasons": m.clocks.summary().get("reasons"),
           "kernel_configs": sorted({p["config"] for p in m.per}),
           "grid_sum": ("none" if m.grid == (1, 1, 1) else
                        "two launches, fp32 partials" if m.flags & fc.VGRID_PARTIALS else
                        "order-free reduction adds" if m.flags & fc.REDUCE_ADD else
                        "chained in one accumulator"),
           "l2": config_block(m.wl, "", 1)["l2"],
           "step_timing": STEP_TIMING[1 if m.reps == 1 else 0]}
    if len(m.per) <= 12:
        out["per_gemm_tflops"] = {f"{p['layer']}:{p['op']}": p["tflops"] for p in m.per}
    else:
        by_t = {}
        for p in m.per:
            by_t.setdefault(p["M"] if p["op"] != "wgrad" else p["R"], []).append(p["tflops"])
        out["median_gemm_tflops_by_T"] = {str(t): round(statistics.median(v), 1)
                                          for t, v in sorted(by_t.items())}
        out["min_gemm_tflops"] = min(p["tflops"] for p in m.per)
    if mem:
        gbs = [p["gbs"] for p in mem]
        out["below_ridge"] = {"gemms": len(mem), "max_gbs": max(gbs),
                              "median_gbs": round(statistics.median(gbs), 1),
                              "frac_of_hbm_max": round(max(gbs) / peaks["hbm_gbs"], 4),
                              "rule": "algorithmic bytes 2(MR+RN+MN) over the median time; "
                                      "shapes whose FLOP per byte is below the ridge point"}
    if check:
        worst, entries = sampled_check(m, fc)
        out["check"] = {"max_error_ratio": worst, "entries": entries,
                        "what": "every GEMM, one random row per 256-row band x one random "
                                "column per 512-column band (finer on small outputs: at least "
                                "16 x 16), plus first/last rows and columns; "
                                "bound |C - C_ref| <= 1e-2 (|A|.|B|) + 1e-5"}
    return out


GOLDFISH = dict(name="goldfish_ce_t8192_v128256", B=4, S=2048, V=128256, k=2, h=13, seed=1007,
                desc="Goldfish-masked cross-entropy and its gradient over bf16 logits: 4 "
                     "sequences x 2048 tokens, a 128256-token vocabulary (the Llama-3 "
                     "vocabulary of the models the pages train), k = 2, h = 13")


def measure_goldfish(args, fc, dev, local, steps, check=True):
    """Times the Goldfish loss (mask, rows, mean) on seeded synthetic logits
    drawn on the device (N(0, 4)), token ids uniform over the vocabulary.
    Algorithmic bytes per step: the kept rows' logits read once, every
    gradient row written once (bf16), plus ids, labels and the per-token
    outputs.  Returns the entry of the `workloads` object."""
    import numpy as np
    import torch

    import fc_inputs
    from oracle import goldfish as gf
    c = GOLDFISH
    B, S, V = getattr(args, "gf_batch", c["B"]), c["S"], c["V"]
    T = B * S
    rng = np.random.default_rng(c["seed"])
    seqs = rng.integers(0, V, size=(B, S + 1))
    ids = torch.from_numpy(seqs[:, :-1].astype(np.int32)).to(dev)
    labels = torch.from_numpy(seqs[:, 1:].astype(np.int32)).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(c["seed"])
    logits = (2.0 * torch.randn((T, V), generator=gen, device=dev)).to(torch.bfloat16)
    dl = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    keep = torch.empty(T, dtype=torch.uint8, device=dev)
    tl = torch.empty(T, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    kept = torch.empty(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        fc.axonn_goldfish_ce(logits, ids, labels, keep, tl, loss, kept, k=c["k"], h=c["h"],
                             dlogits=dl, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    fc.axonn_sync_status(stream)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    with ClockSampler(int(vis) if vis.isdigit() else local) as clocks:
        with torch.cuda.stream(stream):
            for s in range(steps):
                ev[s][0].record(stream)
                gr.replay()
                ev[s][1].record(stream)
        torch.cuda.synchronize()
    fc.axonn_sync_status(stream)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    n = int(kept.item())
    nbytes = 2.0 * n * V + 2.0 * T * V + T * (4 + 4 + 1 + 4)
    peaks = read_peaks()
    gbs = nbytes / ms / 1e6
    out = {"desc": c["desc"], "ms_per_step": round(ms, 4), "gbs": round(gbs, 1),
           "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "bound": "hbm",
           "kept": n, "positions": T, "algorithmic_bytes_per_step": nbytes,
           "launches_per_step": 3, "steps": steps,
           "sm_mhz": clocks.summary().get("sm_mhz"),
           "clock_reasons": clocks.summary().get("reasons"),
           "timing": "CUDA-graph replays of one step (mask, rows, mean), median"}
    if check:
        # mask and count over every position; token losses and gradient rows
        # on a sample of 24 positions, against the fp64 oracle
        ids_h, lab_h = ids.cpu().numpy(), labels.cpu().numpy()
        ref_keep = gf.goldfish_keep(ids_h, lab_h, c["k"], c["h"], vocab=V).reshape(-1)
        sample = np.concatenate([np.arange(8), np.arange(T - 8, T), rng.choice(T, 8, replace=False)])
        st = torch.from_numpy(sample).to(dev)
        sample_bits = fc_inputs.from_torch_bf16(logits.index_select(0, st))
        ref = gf.goldfish_ce(sample_bits, ids_h, lab_h, c["k"], c["h"], rows=sample)
        g = dl.index_select(0, st).double().cpu().numpy()
        tok = tl.index_select(0, st).double().cpu().numpy()
        # bound of the gradient: bf16 rounding plus the fp32 softmax's error
        # (logsumexp, the exponent's products, exp2), as the GPU tests derive
        za = np.abs(fc_inputs.bf16_bits_to_f32(sample_bits).astype(np.float64))
        lse = np.abs(ref["lse"])[:, None]
        eps_p = 1e-5 + lse * 2.0 ** -22 + (za + lse) * 2.0 ** -23 + 2.0 ** -21
        tol_g = (2.0 ** -8 * np.abs(ref["dlogits"])
                 + (1 + 2.0 ** -8) * (ref["softmax"] * eps_p + 2.0 ** -23) / max(n, 1))
        out["check"] = {
            "mask_exact": bool(np.array_equal(keep.cpu().numpy(), ref_keep) and n == ref["n"]),
            "token_loss_max_error_ratio": float(np.max(np.abs(tok - ref["token_loss"])
                                                       / (1e-5 * (1 + np.abs(ref["lse"]))))),
            "dlogits_max_error_ratio": float(np.max(np.abs(g - ref["dlogits"]) / tol_g)),
            "what": "keep mask and count bit for bit over all positions; CE and gradient rows "
                    "of 24 positions against the fp64 oracle (bounds 1e-5 (1 + |lse|) and "
                    "2^-8 |g| + (p eps_p + 2^-23) / n; ratios <= 1 pass)"}
    del logits, dl
    torch.cuda.empty_cache()
    return out


def run_workloads(args, fc, dev, world, local, skip):
    """Every other configuration of the benchmark, each tuned and timed on
    its own (fewer steps), for the `workloads` object of the default line."""
    import torch
    steps = min(args.steps, 10)
    res = {}
    for name in ("single_layer_t256", "single_layer_t256_warm", "gpt_h6144_t8192_vgrid_2x2x2",
                 "large_h16384_t4096", "large_h16384_t4096_vgrid_1x4x4", "layout_sweep"):
        if name == skip:
            continue
        m = measure(name, args, fc, dev, world, local, steps, on_device=True)
        res[name] = {"desc": WORKLOADS[name]["desc"], **workload_summary(m, fc)}
        del m
        torch.cuda.empty_cache()
    res[GOLDFISH["name"]] = measure_goldfish(args, fc, dev, local, steps)
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    import fc_inputs
    import pmm_fc_layer_gb300 as fc

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from pmm_fc_layer_gb300 import build as _b
    _b.build()
    fc.load()
    fc.axonn_set_kernel_config(args.config)
    if args.no_streamk:
        fc.axonn_set_streamk(0)
    if args.l2_budget is not None:
        fc.axonn_set_l2_budget(int(args.l2_budget) << 20)
    sms, max_pairs = fc.axonn_device_info()

    m = measure(args.workload, args, fc, dev, world, local, args.steps, tune_cache=args.tune_cache)
    (wl, grid, flags, out_dtype, only, layers, glist, data, dbuf, plan, ws, flush, stream, used,
     sk_tiles, elapsed_ms, launches, peaks, per, flops_per_step, achieved, clocks) = (
        m.wl, m.grid, m.flags, m.out_dtype, m.only, m.layers, m.glist, m.data, m.dbuf, m.plan,
        m.ws, m.flush, m.stream, m.used, m.sk_tiles, m.elapsed_ms, m.launches, m.peaks, m.per,
        m.flops_per_step, m.achieved, m.clocks)

    # Context only, off the product path: the same products through
    # torch.matmul (cuBLAS), full layers, bf16 outputs, timed the same way.
    torch_mm = None
    if args.torch_matmul and not args.accum_f32:
        def torch_gemm(g):
            torch_product(g["op"], g["P"], g["Q"], g["C"])
        full = [g for g in plan if tuple(g["C"].shape) == tuple(g["mnr"][:2])]
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                for g in full:
                    torch_gemm(g)
            tev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in full]
            per_ms = [0.0] * len(full)
            for _ in range(args.steps):
                for gi, g in enumerate(full):
                    tev[gi][0].record(stream)
                    torch_gemm(g)
                    tev[gi][1].record(stream)
                torch.cuda.synchronize()
                for gi in range(len(full)):
                    per_ms[gi] += tev[gi][0].elapsed_time(tev[gi][1])
        torch.cuda.synchronize()
        tflops = [g["flops"] / (ms / args.steps) / 1e9 for g, ms in zip(full, per_ms)]
        torch_mm = {"value": round(sum(g["flops"] for g in full) * args.steps
                                   / (sum(per_ms) * 1e9), 2) if full else None,
                    "unit": UNIT, "library": "cuBLAS through torch.matmul",
                    "per_gemm_tflops": [round(t, 1) for t in tflops],
                    "timing": "CUDA events around each eager call, summed over the steps",
                    "note": "context only; not the product path"}

    # end to end: host (pinned) -> device copies, the GEMMs, device -> host
    h2d_bytes = d2h_bytes = 0
    io_bytes = sum(t.numel() * t.element_size() for d in dbuf.values() for t in d.values())
    e2e_steps = 0
    if not (args.no_e2e or only is not None or io_bytes > (24 << 30)):
        e2e_steps = max(1, min(args.steps, 10))
    hin, hout = {}, {}
    for name, T, K, N in (layers if e2e_steps else []):
        hin[name] = {k: torch.empty(dbuf[name][k].shape, dtype=torch.bfloat16, pin_memory=True)
                     for k in ("X", "W", "dY")}
        for k, hb in hin[name].items():
            hb.copy_(dbuf[name][k])
            h2d_bytes += hb.numel() * 2
        hout[name] = {k: torch.empty(dbuf[name][k].shape, dtype=out_dtype, pin_memory=True)
                      for k in ("Y", "dX", "dW")}
        d2h_bytes += sum(hb.numel() * hb.element_size() for hb in hout[name].values())

    # The host-buffer step is pipelined by layer on three streams: inputs of
    # layer l+1 go up while layer l's GEMMs run and layer l-1's outputs come
    # down.  Each layer's device buffers are reused every step, so a copy
    # into them waits for the previous step's use.
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    lnames = list(hin)
    in_ready = {n: torch.cuda.Event() for n in lnames}
    gemm_done = {n: torch.cuda.Event() for n in lnames}
    out_done = {n: torch.cuda.Event() for n in lnames}
    by_layer = {n: [g for g in plan if g["name"] == n] for n in lnames}
    first = {"step": True}

    def e2e_step():
        for n in lnames:
            if not first["step"]:
                h2d_stream.wait_event(gemm_done[n])      # previous step read the inputs
            with torch.cuda.stream(h2d_stream):
                for k, hb in hin[n].items():
                    dbuf[n][k].copy_(hb, non_blocking=True)
            in_ready[n].record(h2d_stream)
            stream.wait_event(in_ready[n])
            if not first["step"]:
                stream.wait_event(out_done[n])          # previous step's outputs are down
            for g in by_layer[n]:
                fc.call(g["op"], g["P"], g["Q"], g["C"], g["shape"], flags, ws, stream=stream)
            gemm_done[n].record(stream)
            d2h_stream.wait_event(gemm_done[n])
            with torch.cuda.stream(d2h_stream):
                for k, hb in hout[n].items():
                    hb.copy_(dbuf[n][k], non_blocking=True)
            out_done[n].record(d2h_stream)
        first["step"] = False

    e2e_ms = copies_ms = 0.0
    e2e_pass_ms = []
    e2e_issue = None
    if e2e_steps:
        e2e_step()
        torch.cuda.synchronize()
        # A pass of e2e_steps steps is captured once as a CUDA graph: the
        # pinned-host copies, the library's C ABI calls and the events that
        # pipeline them, on the three streams (forked from and joined to the
        # GEMM stream).  Replaying it runs every copy and every GEMM of every
        # step again; the host issues one replay per pass, so a stall of the
        # host thread cannot idle the GPU inside the pass.  Where capture is
        # refused the steps are issued eagerly, as they go.
        pass_graph = None
        if not args.no_graph:
            try:
                pass_graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(pass_graph, stream=stream):
                    h2d_stream.wait_stream(stream)
                    d2h_stream.wait_stream(stream)
                    first["step"] = True  # no waits on events outside the capture
                    for _ in range(e2e_steps):
                        e2e_step()
                    stream.wait_stream(h2d_stream)
                    stream.wait_stream(d2h_stream)
                e2e_issue = "one CUDA-graph replay per pass (captured C ABI calls and copies)"
            except Exception as exc:  # capture refused: issue eagerly
                pass_graph = None
                torch.cuda.synchronize()
                e2e_issue = f"eager, steps issued as they go (graph capture failed: {exc})"[:200]
            first["step"] = False
        if pass_graph is None and e2e_issue is None:
            e2e_issue = "eager, steps issued as they go"
        if pass_graph is not None:
            with torch.cuda.stream(stream):
                pass_graph.replay()  # warm
            torch.cuda.synchronize()
        # Two timed passes; the faster one is reported and both are listed.
        for _ in range(2):
            if world > 1:
                dist.barrier()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if pass_graph is not None:
                with torch.cuda.stream(stream):
                    t0.record(stream)
                    pass_graph.replay()
                    t1.record(stream)
            else:
                t0.record(h2d_stream)
                stream.wait_event(t0)
                d2h_stream.wait_event(t0)
                for _ in range(e2e_steps):
                    e2e_step()
                h2d_stream.wait_stream(d2h_stream)
                h2d_stream.wait_stream(stream)
                t1.record(h2d_stream)
            torch.cuda.synchronize()
            e2e_pass_ms.append(t0.elapsed_time(t1))
        fc.axonn_sync_status(stream)
        e2e_ms = max_over_ranks(min(e2e_pass_ms), dev)
        # The same host<->device copies with no GEMMs, both directions at
        # once as in the pipeline; their time bounds the end-to-end rate.
        # Best of three passes of up to 3 steps (the link rate varies from
        # pass to pass).
        c_steps = min(3, e2e_steps)
        best = None
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(h2d_stream)
            d2h_stream.wait_event(c0)
            for _ in range(c_steps):
                for n in lnames:
                    with torch.cuda.stream(h2d_stream):
                        for k, hb in hin[n].items():
                            dbuf[n][k].copy_(hb, non_blocking=True)
                    with torch.cuda.stream(d2h_stream):
                        for k, hb in hout[n].items():
                            hb.copy_(dbuf[n][k], non_blocking=True)
            h2d_stream.wait_stream(d2h_stream)
            c1.record(h2d_stream)
            torch.cuda.synchronize()
            ms = c0.elapsed_time(c1) / c_steps
            best = ms if best is None else min(best, ms)
        copies_ms = max_over_ranks(best, dev) * e2e_steps

    # Dense bf16 peak at the SM clock sampled during the timed region:
    # SMs x 8192 FLOP per clock per SM (tcgen05 kind::f16) x clock.
    clk = clocks.summary()
    peak_at_clock = (sms * 8192 * clk["sm_mhz"] * 1e6 / 1e12) if clk.get("sm_mhz") else None
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(world * flops_per_step * args.steps / (elapsed_ms * 1e9), 2),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": DATA if not wl.get("scale") else
            DATA.replace("activations/grads N(0,1), weights N(0,0.02)", "all operands N(0,1)*0.05"),
            "config": config_block(
                wl, args.workload, world, reps=m.reps,
                output=None if not args.accum_f32 else
                "fp32, every step adds its product into it (C += A.B)" + (
                    "; grid partials added by atomics in one launch (order-free)"
                    if args.order_free else "; grid partials summed in fixed order"
                    if grid != (1, 1, 1) else "")),
            "per_gemm": per,
            "per_gemm_note": ("each GEMM's rate from replays of that GEMM alone, after the timed "
                              "steps; the SM clock under the power cap differs from the step's "
                              "and is not sampled per GEMM"),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                         "peak": peaks["burst"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["burst"], 4),
                         "frac_of_sustained": round(achieved / peaks["sustained"], 4),
                         "peak_source": (f"{peaks['source']} burst (the timed region is "
                                         f"{elapsed_ms / 1e3:.2f} s, a burst; sustained "
                                         f"{peaks['sustained']})"),
                         "kernel": ("fc_gemm_tcgen05_kernel / fc_gemm_tcgen05_pair_kernel, "
                                    "every GEMM launch of the step in the configurations "
                                    "listed under device.kernel_configs") + (
                             " (virtual grid: blocks added into the output by reduction adds, one "
                             "launch per GEMM)" if flags & fc.REDUCE_ADD else
                             " (virtual grid: two launches per GEMM, the partials summed in "
                             "the second one's epilogue)" if flags & fc.VGRID_PARTIALS else
                             " (virtual grid: one launch per GEMM, each tile's block products "
                             "chained into one accumulator)" if flags & fc.VGRID else ""),
                         "traffic": traffic_per_launch(args.workload, per, only),
                         "traffic_unit": "bytes per launch (mean over the step)",
                         "traffic_rule": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of "
                                          "each GEMM in the configuration the tuner chose here, "
                                          "from the capture in profiles/; null when a choice or "
                                          "the kernel sources differ from the capture's"),
                         "peak_at_clock": round(peak_at_clock, 1) if peak_at_clock else None,
                         "frac_at_clock": (round(achieved / peak_at_clock, 4)
                                           if peak_at_clock else None),
                         "peak_at_clock_rule": "SMs x 8192 bf16 FLOP/clk x median SM clock "
                                               "of the timed region",
                         "algorithmic_bytes": round(sum(g["bytes"] for g in plan) / len(plan))},
            "e2e": ({"value": round(world * flops_per_step * e2e_steps / (e2e_ms * 1e9), 2),
                     "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                     "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps,
                     "pipelining": "per-layer H2D / GEMM / D2H on three streams",
                     "issue": e2e_issue,
                     "passes_ms_per_step": [round(x / e2e_steps, 3) for x in e2e_pass_ms],
                     "pass_rule": "the faster of two timed passes",
                     "copies_only_ms_per_step": round(copies_ms / e2e_steps, 3),
                     "host_link_gbs": round((h2d_bytes + d2h_bytes) * e2e_steps
                                            / (copies_ms * 1e6), 1),
                     # null when the copies alone measured slower than the
                     # whole overlapped pipeline (a noisy copy measurement)
                     "link_bound_value": (round(world * flops_per_step * e2e_steps
                                                / (max(copies_ms, elapsed_ms * e2e_steps
                                                       / args.steps) * 1e9), 2)
                                          if copies_ms <= e2e_ms else None)}
                    if e2e_steps else None),
            "gpu_launches": launches,
            "tuned": not args.no_tune,
            "tuning": m.tuning,
            "timing": ("eager ABI calls, CUDA events around each" if args.no_graph else
                       ("CUDA-graph replay of one step per timed step; per-GEMM table from "
                        "replays of each GEMM's own graph" if m.reps == 1 else
                        "the K timed steps back to back in one CUDA-graph replay; per-GEMM "
                        "table from one replay of K back-to-back calls of each GEMM")),
            "device": {"sms": sms, "resident_cta_pairs": max_pairs,
                       "kernel_configs": sorted({p["config"] for p in per})},
            "clocks": clk,
            **({"torch_matmul": torch_mm} if torch_mm is not None else {}),
        }
        if args.shrink > 1:
            line["profile_case"] = (f"dimensions divided by {args.shrink}"
                                    + (f", {only[0]}:{only[1]} only" if only else ""))
        elif only is not None:
            line["profile_case"] = f"{only[0]}:{only[1]} only"
        elif data is not None and not args.no_cpu_baseline and world == 1 and args.accum_f32:
            # accumulated outputs hold the sum of every step: no row check
            line["cpu_baseline"] = cpu_baseline(data, glist, rows=cpu_rows(glist))
        elif data is not None and not args.no_cpu_baseline and world == 1:
            # the GPU's first output rows of every GEMM (all of them for a
            # small step), as computed in the timed steps
            rows = cpu_rows(glist)
            gpu_rows = {gi: g["C"][:rows].to(torch.float64).cpu().numpy()
                        for gi, g in enumerate(plan)}
            line["cpu_baseline"] = cpu_baseline(data, glist, gpu_rows, rows)
            # and the whole output of every GEMM, sampled, as the tuned step
            # left it (every tile of every configuration, stream-K tiles
            # included)
            def gpu_at(gi):
                C = plan[gi]["C"]

                def f(ri, cj):
                    ii = torch.from_numpy(ri).to(C.device)
                    jj = torch.from_numpy(cj).to(C.device)
                    return C.index_select(0, ii).index_select(1, jj).to(torch.float64).cpu().numpy()
                return f
            t0 = time.perf_counter()
            worst, entries = whole_output_check(data, glist, {gi: gpu_at(gi) for gi in range(len(plan))})
            line["cpu_baseline"]["whole_output_check"] = {
                "max_error_ratio": worst, "entries": entries,
                "seconds": round(time.perf_counter() - t0, 1),
                "streamk_tiles_in_step": sum(sk_tiles),
                "what": ("sampled over the whole output of every GEMM, stream-K tiles included: "
                         "full rows 0 and M-1, full columns 0 and N-1, and one random row per "
                         "32-row band x one random column per 64-column band (an entry in every "
                         "32 x 64 cell); bound |C - C_ref| <= 1e-2 * (|A|.|B|) + 1e-5")}
        if (world == 1 and not args.no_workloads and only is None and args.shrink == 1
                and args.workload == DEFAULT_WORKLOAD
                and not (args.accum_f32 or args.order_free or args.vgrid_partials)):
            # every other configuration, each on its own after the metric's
            # workload, with fewer timed steps
            del plan, dbuf, ws, m
            torch.cuda.empty_cache()
            t0 = time.perf_counter()
            line["workloads"] = run_workloads(args, fc, dev, world, local, skip=args.workload)
            line["workloads_seconds"] = round(time.perf_counter() - t0, 1)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_goldfish(args):
    """The Goldfish-loss workload alone, as its own JSON line (HBM-bound)."""
    import torch
    import pmm_fc_layer_gb300 as fc
    from pmm_fc_layer_gb300 import build as _b
    torch.cuda.set_device(0)
    _b.build()
    fc.load()
    dev = torch.device("cuda", 0)
    r = measure_goldfish(args, fc, dev, 0, args.steps, check=not args.no_cpu_baseline)
    peaks = read_peaks()
    print(json.dumps({
        "metric": "Goldfish-masked cross-entropy with gradient: HBM GB/s", "value": r["gbs"],
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in/out, fp32 arithmetic",
        "data": "synthetic, seeded: logits N(0,4) drawn on the device, token ids uniform",
        "config": {"workload": f"{GOLDFISH['name']}: {GOLDFISH['desc']}"},
        "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": r["frac_of_hbm"], "traffic": None,
                     "algorithmic_bytes": r["algorithmic_bytes_per_step"]},
        "gpu_launches": 3 * args.steps, "detail": r,
        **({"profile_case": f"{args.gf_batch} sequences instead of {GOLDFISH['B']}"}
           if args.gf_batch != GOLDFISH["B"] else {})}), flush=True)
    return 0


def run_zsharded(args):
    """Z-sharded weights of the 2x2x2 grid on the GPT block (H=6144,
    T=8192): for every layer and weight block (x, y), the all-gather of its
    two row shards and the Z-group weight gradient written as
    reduce-scattered shards.  Reports the gather's HBM rate against the HBM
    peak (algorithmic bytes: each block read once and written once) and the
    sharded weight gradient's TFLOP/s."""
    import torch
    import pmm_fc_layer_gb300 as fc
    from pmm_fc_layer_gb300 import build as _b
    torch.cuda.set_device(0)
    _b.build()
    fc.load()
    dev = torch.device("cuda", 0)
    grid = (2, 2, 2)
    layers = _gpt(6144, 8192, 4 * 6144)
    g = torch.Generator(device=dev)
    g.manual_seed(1006)
    stream = torch.cuda.Stream(device=dev)
    jobs, gather_bytes, wgrad_flops, ws_need = [], 0.0, 0.0, 0
    for name, T, K, N in layers:
        X = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
        dY = torch.randn((T, N), generator=g, device=dev).to(torch.bfloat16)
        for x in range(grid[0]):
            for y in range(grid[1]):
                shape = fc.Shape(T, K, N, grid, (x, y, 0))
                k0, k1 = fc.axonn_block_range(K, grid[0], x)
                n0, n1 = fc.axonn_block_range(N, grid[1], y)
                rows, cols = k1 - k0, n1 - n0
                cuts = [fc.axonn_block_range(rows, grid[2], z) for z in range(grid[2])]
                W_sh = [(0.02 * torch.randn((b - a, cols), generator=g, device=dev)).to(torch.bfloat16)
                        for a, b in cuts]
                W_blk = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
                dW_sh = [torch.empty((b - a, cols), dtype=torch.bfloat16, device=dev) for a, b in cuts]
                ws_need = max(ws_need, fc.axonn_fc_workspace_size("wgrad", shape, fc.ZSHARDED))
                jobs.append((X, dY, W_sh, W_blk, dW_sh, shape, rows, cols))
                gather_bytes += 2.0 * 2 * rows * cols
                wgrad_flops += 2.0 * rows * cols * T
    ws = torch.empty(ws_need, dtype=torch.uint8, device=dev)

    def gathers():
        for X, dY, W_sh, W_blk, dW_sh, shape, rows, cols in jobs:
            fc.axonn_shards_gather(W_sh, W_blk, rows, cols, stream=stream)

    def wgrads():
        for X, dY, W_sh, W_blk, dW_sh, shape, rows, cols in jobs:
            fc.axonn_fc_wgrad_zsharded(X, dY, dW_sh, shape, 0, ws, stream=stream)

    times = {}
    with torch.cuda.stream(stream):
        for label, fn in (("gather", gathers), ("wgrad", wgrads)):
            for _ in range(args.warmup):
                fn()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            gr.replay()
            e0.record(stream)
            for _ in range(args.steps):
                gr.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times[label] = e0.elapsed_time(e1) / args.steps
    fc.axonn_sync_status(stream)
    peaks = read_peaks()
    gbs = gather_bytes / times["gather"] / 1e6
    tf = wgrad_flops / times["wgrad"] / 1e9
    print(json.dumps({
        "metric": "Z-sharded weights on a 2x2x2 grid: shard all-gather GB/s and sharded "
                  "weight-gradient TFLOP/s", "value": round(tf, 2), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic, seeded (torch generator on the device)",
        "config": {"workload": "zsharded_h6144_2x2x2: GPT block H=6144, T=8192, grid 2x2x2; "
                               "all four layers x four weight blocks (x, y)"},
        "gather": {"ms_per_step": round(times["gather"], 4), "gbs": round(gbs, 1),
                   "algorithmic_bytes_per_step": gather_bytes, "bound": "hbm",
                   "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                   "peak_source": peaks["source"]},
        "wgrad_zsharded": {"ms_per_step": round(times["wgrad"], 4), "tflops": round(tf, 1),
                           "frac_of_sustained": round(tf / peaks["sustained"], 4)},
        "timing": "CUDA-graph replays"}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["zsharded_h6144_2x2x2",
                                                               GOLDFISH["name"]],
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--config", type=int, default=-1,
                    help="force one kernel configuration (-1: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed CPU oracle sample")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-streamk", action="store_true",
                    help="run (and tune) every GEMM without a stream-K tail")
    ap.add_argument("--l2-budget", type=int, default=None, metavar="MB",
                    help="L2 budget of the operand loads' evict-last lines (0: no L2 hints)")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip the per-shape tuning before the warm-up (use default choices)")
    ap.add_argument("--retune", action="store_true",
                    help="tune every GEMM at run time, ignoring a tuning table shipped for "
                         "the workload")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager ABI calls instead of CUDA-graph replays")
    ap.add_argument("--tune-cache", default=None, metavar="PATH",
                    help="load tuned choices from PATH if it exists (no tuning), else tune "
                         "and save them there")
    ap.add_argument("--accum-f32", action="store_true",
                    help="fp32 outputs that every step adds into (the main-gradient form)")
    ap.add_argument("--order-free", action="store_true",
                    help="virtual grid with --accum-f32: blocks added into the output by "
                         "atomics in one launch, instead of the fixed-order sum")
    ap.add_argument("--shrink", type=int, default=1, metavar="S",
                    help="divide the workload's dimensions by S (a profiling case; not a bench "
                         "line)")
    ap.add_argument("--gf-batch", type=int, default=GOLDFISH["B"], metavar="B",
                    help="sequences of the Goldfish workload (smaller for profiling)")
    ap.add_argument("--swap-compare", action="store_true",
                    help="after the timed region, time every GEMM with the operand roles "
                         "forced unexchanged and exchanged (per_gemm ms_swap0 / ms_swap1)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations after the default workload")
    ap.add_argument("--vgrid-partials", action="store_true",
                    help="virtual grid in its two-launch form: fp32 partials in a workspace, "
                         "summed in the last block's epilogue (default: chained)")
    ap.add_argument("--torch-matmul", action="store_true",
                    help="also time the same products through torch.matmul (cuBLAS), as "
                         "context off the product path")
    ap.add_argument("--only", default=None, metavar="LAYER:OP",
                    help="time one GEMM (e.g. out:fwd) for profiling; not a bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.order_free and not args.accum_f32:
        ap.error("--order-free needs --accum-f32")
    if args.order_free and "grid" not in WORKLOADS.get(args.workload, {}):
        ap.error("--order-free needs a virtual-grid workload")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "zsharded_h6144_2x2x2":
        return run_zsharded(args)
    if args.workload == GOLDFISH["name"]:
        return run_goldfish(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
