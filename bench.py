#!/usr/bin/env python
"""Benchmark of the FC-layer GEMMs of one GPT block on GB300.

A step is one pass of the whole path over one batch: for each of the four
FC layers of a GPT block with hidden size H = 6144 and T = 8192 tokens
(batch 4 x sequence 2048) -- QKV [H -> 3H], attention-out [H -> H],
MLP-up [H -> 4H], MLP-down [4H -> H] -- the forward product Y = X.W, the
data gradient dX = dY.W^T and the weight gradient dW = X^T.dY, all through
the C ABI of libaxonn_fc.so (12 tcgen05 GEMM launches).

Inputs are seeded synthetic bf16 (SplitMix64 + Box-Muller): activations and
gradients ~N(0,1), weights ~N(0,0.02).  Every GEMM's operands are larger than
the 129 MB L2, so no flush is needed between timed iterations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun with N > 1 every rank runs
an independent replica on its own GPU (the path needs no collective on one
GPU per rank); the value is the total over ranks divided by the slowest
rank's time.  `--impl reference` times the fp64 CPU oracle on the host
cores over a bounded sample of the same workload.
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
H, T_TOK, BATCH, SEQ = 6144, 8192, 4, 2048
LAYERS = [("qkv", H, 3 * H), ("out", H, H), ("up", H, 4 * H), ("down", 4 * H, H)]
SEED = 1002
WORKLOAD = (f"GPT block FC layers, H={H}, T={T_TOK} (batch {BATCH} x seq {SEQ}): "
            "qkv [H->3H], out [H->H], up [H->4H], down [4H->H]; fwd+dgrad+wgrad each, full layers")
DATA = ("synthetic, seeded: SplitMix64 + Box-Muller bf16; activations/grads N(0,1), "
        "weights N(0,0.02)")
CPU_STRIPE_ROWS = 16      # rows of every GEMM the CPU oracle computes per sample


def gemms():
    """The 12 products of one step: (layer, op, M, N, R, tensor names)."""
    out = []
    for name, K, N in LAYERS:
        out.append((name, "fwd", T_TOK, N, K, ("X", "W", "Y")))
        out.append((name, "dgrad", T_TOK, K, N, ("dY", "W", "dX")))
        out.append((name, "wgrad", K, N, T_TOK, ("X", "dY", "dW")))
    return out


FLOPS_PER_STEP = sum(2.0 * m * n * r for _, _, m, n, r, _ in gemms())


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"burst": float(d["bf16_tflops"]),
                "sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d.get("hbm_gbs", 0.0)) or None,
                "source": "measured"}
    except (OSError, KeyError, ValueError, TypeError):
        return {"burst": 1900.0, "sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ inputs
def host_inputs(layers=LAYERS):
    """Seeded bf16 bits of the layers' X, W and dY (numpy uint16)."""
    import fc_inputs
    data = {}
    for name, K, N in layers:
        tid = 16 * ([l[0] for l in LAYERS].index(name) + 1)
        data[name] = {
            "X": fc_inputs.normal_bf16((T_TOK, K), SEED, tid + 1),
            "W": fc_inputs.normal_bf16((K, N), SEED, tid + 2, sigma=0.02),
            "dY": fc_inputs.normal_bf16((T_TOK, N), SEED, tid + 3),
        }
    return data


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
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
        sm, smax, reasons = [], [], set()
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
def oracle_stripes(data, which, rows):
    """fp64 oracle on the first `rows` output rows of the listed GEMMs;
    returns (flops, seconds, threads used)."""
    import oracle
    flops, secs = 0.0, 0.0
    for gi in which:
        name, op, m, n, r, (pn, qn, _) = gemms()[gi]
        d = data[name]
        if op == "wgrad":
            P = d[pn][:, :rows]        # X[:, k-stripe] -> rows of dW
        else:
            P = d[pn][:rows]
        Q = d[qn]
        t0 = time.perf_counter()
        oracle.fc(op, P, Q)
        secs += time.perf_counter() - t0
        flops += 2.0 * rows * n * r
    return flops, secs, min(oracle.max_threads(), rows)


def cpu_baseline(data):
    flops, secs, cores = oracle_stripes(data, range(len(gemms())), CPU_STRIPE_ROWS)
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {CPU_STRIPE_ROWS} output rows of each of the 12 GEMMs "
                      f"({flops / 1e9:.1f} GFLOP, {secs:.1f} s)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    data = host_inputs()
    n = len(gemms())
    for s in range(args.warmup):
        oracle_stripes(data, [s % n], CPU_STRIPE_ROWS)
    tot_f, tot_s, cores = 0.0, 0.0, 1
    for s in range(args.steps):
        f, sec, cores = oracle_stripes(data, [s % n], CPU_STRIPE_ROWS)
        tot_f += f
        tot_s += sec
    value = tot_f / tot_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
            "config": {"workload": WORKLOAD, "global_batch": BATCH, "seq_len": SEQ,
                       "parallelism": "host cores (OpenMP)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: first {CPU_STRIPE_ROWS} output rows of one "
                                       "of the 12 GEMMs, cycling"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import numpy as np
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
    sms, max_pairs = fc.axonn_device_info()

    only = tuple(args.only.split(":")) if args.only else None
    layers = [l for l in LAYERS if only is None or l[0] == only[0]]
    data = host_inputs(layers)
    dbuf, hbuf_in, hbuf_out = {}, {}, {}
    for name, K, N in layers:
        d = {k: fc_inputs.as_torch_bf16(v, dev) for k, v in data[name].items()}
        d["Y"] = torch.empty((T_TOK, N), dtype=torch.bfloat16, device=dev)
        d["dX"] = torch.empty((T_TOK, K), dtype=torch.bfloat16, device=dev)
        d["dW"] = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
        dbuf[name] = d
    stream = torch.cuda.Stream(device=dev)
    plan = []
    for name, op, m, n, r, (pn, qn, cn) in gemms():
        if only is not None and (name, op) != only:
            continue
        K = dict((l, k) for l, k, _ in LAYERS)[name]
        N = dict((l, nn) for l, _, nn in LAYERS)[name]
        plan.append((name, op, 2.0 * m * n * r, dbuf[name][pn], dbuf[name][qn], dbuf[name][cn],
                     fc.Shape(T_TOK, K, N), (m, n, r)))

    def step(events=None):
        for gi, (name, op, _, P, Q, C, shape, _mnr) in enumerate(plan):
            if events is not None:
                events[gi][0].record(stream)
            fc.call(op, P, Q, C, shape, 0, None, stream=stream)
            if events is not None:
                events[gi][1].record(stream)
                used[gi] = fc.axonn_last_kernel_config()

    used = [None] * len(plan)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    fc.axonn_sync_status(stream)

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in plan]
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clocks:
        t0.record(stream)
        for s in range(args.steps):
            step(ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    fc.axonn_sync_status(stream)
    elapsed_ms = t0.elapsed_time(t1)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    launches = args.steps * len(plan)

    # per-GEMM device times (median over steps) and the dominant kernel's rate
    per = []
    gemm_ms_total = 0.0
    flops_per_step = sum(p[2] for p in plan)
    for gi, (name, op, fl, P, Q, C, shape, (m, n, r)) in enumerate(plan):
        ms = [ev[s][gi][0].elapsed_time(ev[s][gi][1]) for s in range(args.steps)]
        gemm_ms_total += sum(ms)
        med = statistics.median(ms)
        per.append({"layer": name, "op": op, "M": m, "N": n, "R": r, "layout": {"fwd": "NN", "dgrad": "NT", "wgrad": "TN"}[op],
                    "ms": round(med, 4), "tflops": round(fl / med / 1e9, 1),
                    "config": fc.axonn_kernel_config_name(used[gi])})
    peaks = read_peaks()
    for p in per:
        p["frac_of_sustained"] = round(p["tflops"] / peaks["sustained"], 4)
        p["frac_of_burst"] = round(p["tflops"] / peaks["burst"], 4)
    achieved = flops_per_step * args.steps / (gemm_ms_total * 1e9)

    # end to end: host (pinned) -> device copies, the 12 GEMMs, device -> host
    h2d_bytes = d2h_bytes = 0
    e2e_steps = 0 if (args.no_e2e or only is not None) else max(1, min(args.steps, 10))
    for name, K, N in (layers if e2e_steps else []):
        hbuf_in[name] = {k: torch.empty(v.shape, dtype=torch.bfloat16, pin_memory=True)
                         for k, v in dbuf[name].items() if k in ("X", "W", "dY")}
        for k in hbuf_in[name]:
            hbuf_in[name][k].copy_(dbuf[name][k])
            h2d_bytes += hbuf_in[name][k].numel() * 2
        hbuf_out[name] = {k: torch.empty(dbuf[name][k].shape, dtype=torch.bfloat16,
                                         pin_memory=True) for k in ("Y", "dX", "dW")}
        for k in hbuf_out[name]:
            d2h_bytes += hbuf_out[name][k].numel() * 2

    def e2e_step():
        for name, _, _ in layers:
            for k, hb in hbuf_in[name].items():
                dbuf[name][k].copy_(hb, non_blocking=True)
        step()
        for name, _, _ in layers:
            for k, hb in hbuf_out[name].items():
                hb.copy_(dbuf[name][k], non_blocking=True)

    e2e_ms = 0.0
    if e2e_steps:
        with torch.cuda.stream(stream):
            e2e_step()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            t0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            t1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = t0.elapsed_time(t1)
    fc.axonn_sync_status(stream)
    if world > 1 and e2e_steps:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(world * flops_per_step * args.steps / (elapsed_ms * 1e9), 2),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": DATA,
            "config": {"workload": WORKLOAD, "global_batch": BATCH * world, "seq_len": SEQ,
                       "hidden": H, "tokens_per_gpu": T_TOK,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "every GEMM's operands exceed the 129 MB L2; no flush"},
            "per_gemm": per,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                         "peak": peaks["sustained"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["sustained"], 4),
                         "frac_of_burst": round(achieved / peaks["burst"], 4),
                         "peak_source": f"{peaks['source']} (sustained; burst {peaks['burst']})",
                         "kernel": "fc_gemm_tcgen05_kernel",
                         "traffic": None},
            "e2e": ({"value": round(world * flops_per_step * e2e_steps / (e2e_ms * 1e9), 2),
                     "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                     "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps}
                    if e2e_steps else None),
            "gpu_launches": launches,
            "device": {"sms": sms, "resident_cta_pairs": max_pairs,
                       "kernel_configs": sorted({p["config"] for p in per})},
            "clocks": clocks.summary(),
        }
        if only is not None:
            line["profile_case"] = f"{only[0]}:{only[1]} only"
            line["config"]["workload"] = f"{WORKLOAD}; this run: {only[0]} {only[1]} only"
        elif not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(data)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed CPU oracle sample")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--config", type=int, default=-1,
                    help="force one kernel configuration (-1: the library's choice)")
    ap.add_argument("--only", default=None, metavar="LAYER:OP",
                    help="time one GEMM (e.g. out:fwd) for profiling; not a bench line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
