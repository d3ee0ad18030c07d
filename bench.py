#!/usr/bin/env python3
"""Benchmark of the batch-1 dequant GEMV on one node.

One step = the Q4_K decode projections of a Llama-8B-like layer (QKV 6144x4096, gate+up
28672x4096, down 4096x14336): three GEMVs through the C-ABI.  Weights are synthetic and
seeded, resident in HBM, rotated over enough copies that each step reads from HBM (the
whole set of copies is > 3x the L2 size).  Timed on the device with CUDA events around
replays of a CUDA graph holding the steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead, on the
host cores, on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from quantized_weight_dequant_gb300 import synth  # noqa: E402

METRIC = "fused dequant-GEMV achieved HBM GB/s and µs/call at M=1 (fraction of GB300 peak)"

# name -> list of (label, fmt, N, K, activation key).  GEMVs sharing an activation key
# read the same x (the layer's hidden vector or its MLP activation).
WORKLOADS = {
    "q4k_llama8b_decode": [("qkv", synth.Q4_K, 6144, 4096, "h"), ("gate_up", synth.Q4_K, 28672, 4096, "h"),
                           ("down", synth.Q4_K, 4096, 14336, "m")],
    "q4k_1024x1024": [("w", synth.Q4_K, 1024, 1024, "h")],
    "nvfp4_4096x14336": [("w", synth.NVFP4, 4096, 14336, "h")],
    "nvfp4_14336x4096": [("w", synth.NVFP4, 14336, 4096, "h")],
    "tq1_0_4096x4096": [("w", synth.TQ1_0, 4096, 4096, "h")],
    "tq1_0_11008x4096": [("w", synth.TQ1_0, 11008, 4096, "h")],
    "layer_mixed": [(p, synth.LAYER_MIXED[p], n, k, "m" if p == "down" else "h") for p, n, k in synth.LAYER_SHAPES],
}
for _p, _n, _k in synth.LAYER_SHAPES:
    for _f in (synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.Q8_0):
        WORKLOADS[f"layer_{_p}_{synth.FORMAT_NAMES[_f]}"] = [(_p, _f, _n, _k, "h")]
DEFAULT_WORKLOAD = "q4k_llama8b_decode"
WEIGHT_SEED = 1000  # seed of a workload's first weight matrix; matrix i takes WEIGHT_SEED + i

# Layer launches: GEMVs of a workload that carry the same group tag run as ONE
# qgemv_run_group launch (they share x); a group listed in SWIGLU holds a gate and an up
# matrix (in that order) combined into one output silu(gate) * up.  Untagged GEMVs run alone.
WORKLOADS["layer_mixed_grouped"] = WORKLOADS["layer_mixed"]
WORKLOADS["q4k_llama8b_decode_swiglu"] = [("qkv", synth.Q4_K, 6144, 4096, "h"),
                                          ("gate", synth.Q4_K, 14336, 4096, "h"),
                                          ("up", synth.Q4_K, 14336, 4096, "h"),
                                          ("down", synth.Q4_K, 4096, 14336, "m")]
GROUPS = {"layer_mixed_grouped": {"q": "qkv", "k": "qkv", "v": "qkv", "gate": "mlp", "up": "mlp"},
          "q4k_llama8b_decode_swiglu": {"gate": "mlp", "up": "mlp"}}
SWIGLU = {"mlp"}


def launch_units(workload: str, gemvs):
    """[(label, [gemv indices], swiglu)] in workload order: one entry per kernel launch."""
    tags = GROUPS.get(workload, {})
    units, seen = [], {}
    for gi, g in enumerate(gemvs):
        tag = tags.get(g[0])
        if tag is None:
            units.append((g[0], [gi], False))
        elif tag in seen:
            units[seen[tag]][1].append(gi)
        else:
            seen[tag] = len(units)
            units.append((tag, [gi], tag in SWIGLU))
    for label, idx, sw in units:
        if sw and len(idx) != 2:
            raise ValueError(f"{workload}: SwiGLU group {label} needs a gate and an up matrix")
        if len({(gemvs[i][3], gemvs[i][4]) for i in idx}) != 1:
            raise ValueError(f"{workload}: group {label} must share K and x")
    return units


def unit_bytes(gemvs, idx, swiglu: bool, batch: int = 1) -> int:
    """Algorithmic bytes of one launch: packed weights once, x once per vector, the outputs
    (fp32) of every vector."""
    K = gemvs[idx[0]][3]
    outs = gemvs[idx[0]][2] if swiglu else sum(gemvs[i][2] for i in idx)
    return sum(synth.packed_bytes(gemvs[i][1], gemvs[i][2], gemvs[i][3]) for i in idx) + batch * (2 * K + 4 * outs)


def gemv_bytes(fmt, N, K) -> int:
    """Algorithmic bytes of one GEMV: packed weights + x (2 B/elem) + y (4 B/elem)."""
    return synth.packed_bytes(fmt, N, K) + 2 * K + 4 * N


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic(build_marker: str, kernel: str):
    """ncu DRAM bytes per launch of `kernel` recorded in profiles/roofline_traffic.json for
    this build (the library's source digest); None when the record is for another build."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("build") != build_marker.split(":", 1)[-1]:
        return None, f"recorded for build {rec.get('build')}, not this one"
    k = rec.get("kernels", {}).get(kernel)
    if not k:
        return None, None
    return float(k["dram_bytes_per_launch"]), rec.get("command")


# The benchmark configurations at M = 1, each GEMV timed on its own: (config, [(label, fmt,
# N, K)]).  Config 4 is the Qwen-like layer, in the mixed assignment and in every
# projection x format pair.
CONFIGS = [
    ("config0_q4k_1024x1024", [("w", synth.Q4_K, 1024, 1024)]),
    ("config1_q4k_llama8b_decode", [("qkv", synth.Q4_K, 6144, 4096), ("gate_up", synth.Q4_K, 28672, 4096),
                                    ("down", synth.Q4_K, 4096, 14336)]),
    ("config2_nvfp4_llama8b", [("4096x14336", synth.NVFP4, 4096, 14336), ("14336x4096", synth.NVFP4, 14336, 4096)]),
    ("config3_tq1_0", [("4096x4096", synth.TQ1_0, 4096, 4096), ("11008x4096", synth.TQ1_0, 11008, 4096)]),
    ("config4_layer_mixed", [(p, synth.LAYER_MIXED[p], n, k) for p, n, k in synth.LAYER_SHAPES]),
    ("config4_layer_every_projection_x_format",
     [(f"{p}:{synth.FORMAT_NAMES[f]}", f, n, k) for p, n, k in synth.LAYER_SHAPES
      for f in (synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.Q8_0)]),
]


# ------------------------------------------------------------------ clocks sampler
class Clocks:
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int, uuid: str | None):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"qgemv_clocks_{os.getpid()}.csv")
        target = f"GPU-{uuid}" if uuid else str(device_index)
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}",
                                          "--format=csv,noheader,nounits", "-lms", "100", "-i", target],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle timing
class OracleSampler:
    """Times the CPU oracle on row samples of every GEMV of a workload (host cores)."""

    def __init__(self, gemvs, threads: int, seed: int = 0, batch: int = 1):
        import oracle
        self.oracle = oracle
        self.threads = threads
        self.batch = batch  # activation vectors per GEMV (the oracle runs each one)
        self.pool = cf.ThreadPoolExecutor(max_workers=threads)  # the C oracle releases the GIL
        self.data = []
        for label, fmt, N, K, _ in gemvs:
            self.data.append((label, fmt, N, K, synth.make_weights(fmt, N, K, seed), synth.make_x(fmt, K, seed)))
        per_row = []
        for label, fmt, N, K, W, x in self.data:  # calibration: a few rows on one thread
            t0 = time.perf_counter()
            oracle.gemv(fmt, x, W, N, K, 0, 4)
            per_row.append((time.perf_counter() - t0) / 4)
        self.row_cost = batch * sum(per_row)  # seconds for one row of every GEMV and vector

    def run(self, budget_s: float):
        """One timed sample costing about `budget_s` of wall time.  Returns (GB/s, s, text)."""
        rows = max(1, int(budget_s * self.threads / max(self.row_cost, 1e-9)))
        jobs, nbytes = [], 0
        for label, fmt, N, K, W, x in self.data:
            r = min(rows, N)
            start = (N - r) // 2
            chunk = max(1, math.ceil(r / self.threads))
            for _ in range(self.batch):
                for a in range(start, start + r, chunk):
                    jobs.append((fmt, x, W, N, K, a, min(start + r, a + chunk)))
            nbytes += synth.packed_bytes(fmt, r, K) + self.batch * (2 * K + 4 * r)
        t0 = time.perf_counter()
        list(self.pool.map(lambda j: self.oracle.gemv(*j), jobs))
        dt = time.perf_counter() - t0
        sample = "middle rows of each GEMV: " + ", ".join(
            f"{min(rows, d[2])} of {d[0]} {d[2]}x{d[3]}" for d in self.data)
        return nbytes / dt / 1e9, dt, sample

    def close(self):
        self.pool.shutdown()


def run_reference(args, gemvs, rank, world):
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    sampler = OracleSampler(gemvs, threads, batch=args.batch)
    per_step = max(0.01, 5.0 * args.cpu_seconds / max(1, args.steps + args.warmup))  # about a minute in all
    for _ in range(args.warmup):
        sampler.run(per_step)
    rates, total, sample = [], 0.0, ""
    for _ in range(args.steps):
        r, dt, sample = sampler.run(per_step)
        rates.append(r)
        total += dt
    sampler.close()
    value = statistics.median(rates)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "shapes": [f"{g[0]}:{synth.FORMAT_NAMES[g[1]]}:{g[2]}x{g[3]}"
                                                             for g in gemvs], "batch": args.batch},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"per step: {sample}"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ multi-rank host logic
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (all ranks take part; a single rank returns its own)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, steps: int, step_bytes: int, ms: float) -> float:
    """Weak scaling: every rank streams its own copy of the step; bytes of all ranks over the
    slowest rank's time."""
    return world * steps * step_bytes / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ GPU arm
def largest_divisor_le(k: int, cap: int) -> int:
    for d in range(min(k, cap), 0, -1):
        if k % d == 0:
            return d
    return 1


def run_profile_launches(args, gemvs):
    """Plain launches of the workload's launch units (one weight copy, no graph, no timing),
    for running under a profiler: `--profile-launches N [--only LABEL]`."""
    import torch

    from quantized_weight_dequant_gb300 import qgemv
    from quantized_weight_dequant_gb300.build import build_library

    build_library()
    h = qgemv.create(0)
    if args.pdl:
        qgemv.set_option(h, qgemv.OPT_PDL, 1)
    units = [u for u in launch_units(args.workload, gemvs) if args.only in (None, u[0])]
    if not units:
        raise SystemExit(f"--only {args.only}: no such launch in {args.workload}")
    grouped = set(GROUPS.get(args.workload, {}).values())
    for label, idx, sw in units:
        Ws, ys = [], []
        for gi in idx:
            _, fmt, N, K, _ = gemvs[gi]
            Ws.append(torch.from_numpy(synth.make_weights(fmt, N, K, WEIGHT_SEED + gi)).cuda())
            ys.append(torch.empty(N, dtype=torch.float32, device="cuda"))
        _, fmt, N, K, _ = gemvs[idx[0]]
        B = args.batch
        x = torch.from_numpy(np.stack([synth.make_x(fmt, K, WEIGHT_SEED + idx[0] + 7919 * m)
                                       for m in range(B)]).view(np.int16)).cuda()
        if B > 1:
            ys = [torch.empty((B, gemvs[gi][2]), dtype=torch.float32, device="cuda") for gi in idx]
        for _ in range(args.profile_launches):
            if label not in grouped and B > 1:
                qgemv.run_batch(h, fmt, x, B, Ws[0], N, K, ys[0])
            elif label not in grouped:
                qgemv.run(h, fmt, x, Ws[0], N, K, ys[0])
            elif sw:
                qgemv.run_group(h, x, K, [qgemv.problem(fmt, Ws[0], N, ys[0], packed_W_up=Ws[1], swiglu=True)])
            else:
                qgemv.run_group(h, x, K, [qgemv.problem(gemvs[gi][1], W, gemvs[gi][2], y)
                                          for gi, W, y in zip(idx, Ws, ys)])
        torch.cuda.synchronize()
        st = qgemv.check_error(h)
        if st != qgemv.OK:
            raise RuntimeError(f"qgemv error {qgemv.status_string(st)}")
        plan = (qgemv.describe(h, fmt, N, K) if B == 1 else f"batch of {B}") if label not in grouped else "grouped launch"
        print(f"{label}: {args.profile_launches} launches, {plan}", flush=True)
    h.close()
    return 0


def load_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def run_prefill(args, gemvs, rank, world):
    """`--prefill M`: the NVFP4 GEMM of M activation rows (qgemv_run_gemm, the tcgen05
    tensor-core kernel for M > 8) on the workload's NVFP4 matrices, timed with CUDA events
    over --steps launches after --warmup, weight copies rotated so that W and X together
    exceed L2 three times.  One JSON line: TFLOP/s against the dense bf16 tensor peak."""
    import torch

    from quantized_weight_dequant_gb300 import qgemv
    from quantized_weight_dequant_gb300.build import build_library

    shapes = [(lab, n, k) for lab, f, n, k, _ in gemvs if f == synth.NVFP4]
    if not shapes:
        raise SystemExit(f"--prefill: workload {args.workload} has no NVFP4 matrix")
    if world > 1 and rank != 0:
        return 0  # replicas only: rank 0 measures
    build_library()
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    h = qgemv.create(0)
    M = args.prefill
    stream = torch.cuda.Stream(device=dev)
    rows, total_flop, total_ms, launches = [], 0.0, 0.0, 0
    clocks = Clocks(0, str(getattr(props, "uuid", "")) or None)
    for lab, N, K in shapes:
        W = torch.from_numpy(synth.make_weights(synth.NVFP4, N, K, WEIGHT_SEED)).to(dev)
        X = torch.from_numpy(np.stack([synth.make_x(synth.NVFP4, K, 11 + 7919 * m) for m in range(M)])
                             .view(np.int16)).to(dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        copies = max(2, math.ceil(3 * l2 / (W.numel() + X.numel() * 2)))
        Ws = [W] + [W.clone() for _ in range(copies - 1)]
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                qgemv.run_gemm(h, synth.NVFP4, X, M, Ws[i % copies], N, K, Y, stream=stream)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                qgemv.run_gemm(h, synth.NVFP4, X, M, Ws[i % copies], N, K, Y, stream=stream)
            e1.record(stream)
        stream.synchronize()
        st = qgemv.check_error(h, stream)
        if st != qgemv.OK:
            raise RuntimeError(f"qgemv error {qgemv.status_string(st)}")
        ms = e0.elapsed_time(e1)
        flop = 2.0 * M * N * K * args.steps
        rows.append({"gemm": f"{lab}:NVFP4:{M}x{N}x{K}", "us": ms * 1e3 / args.steps,
                     "TFLOP/s": flop / (ms * 1e-3) / 1e12, "copies": copies})
        total_flop += flop
        total_ms += ms
        launches += args.steps
        del Ws, W, X, Y
    clk = clocks.stop()
    peak, kind = load_bf16_peak()
    value = total_flop / (total_ms * 1e-3) / 1e12
    line = {"metric": "NVFP4 W4A16 prefill GEMM TFLOP/s (qgemv_run_gemm)", "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "replicas only", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "impl": "ours",
            "config": {"workload": args.workload, "rows": M, "gemms": rows,
                       "timing": "CUDA events around --steps launches per matrix, rotating weight copies"},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                         "frac": value / peak, "peak_kind": f"bf16_tflops of {kind} (dense bf16 burst)",
                         "traffic": None},
            "gpu_launches": launches, "clocks": clk, "build": qgemv.build_marker(), "gpu": props.name}
    print(json.dumps(line), flush=True)
    h.close()
    return 0


def run_profile_prefill(args, gemvs):
    """`--prefill M --profile-launches N`: N plain GEMM launches per NVFP4 matrix, for a profiler."""
    import torch

    from quantized_weight_dequant_gb300 import qgemv
    from quantized_weight_dequant_gb300.build import build_library

    build_library()
    h = qgemv.create(0)
    M = args.prefill
    for lab, f, N, K, _ in gemvs:
        if f != synth.NVFP4 or args.only not in (None, lab):
            continue
        W = torch.from_numpy(synth.make_weights(f, N, K, WEIGHT_SEED)).cuda()
        X = torch.from_numpy(np.stack([synth.make_x(f, K, 11 + 7919 * m) for m in range(M)]).view(np.int16)).cuda()
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for _ in range(args.profile_launches):
            qgemv.run_gemm(h, f, X, M, W, N, K, Y)
        torch.cuda.synchronize()
        st = qgemv.check_error(h)
        if st != qgemv.OK:
            raise RuntimeError(f"qgemv error {qgemv.status_string(st)}")
        print(f"{lab}: {args.profile_launches} GEMM launches of {M}x{N}x{K}", flush=True)
    h.close()
    return 0


def graph_us(launch, copies: int, stream, R: int = 200, reps: int = 7) -> float:
    """Mean µs per launch: a CUDA graph of R launches cycling over `copies` weight copies,
    replayed `reps` times after one warm replay; median over the replays (CUDA events on the
    launch stream)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(R):
            launch(i % copies)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    samples = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        stream.synchronize()
        samples.append(a.elapsed_time(b) * 1e3 / R)
    del g
    return statistics.median(samples)


def flushed_single_us(launch, stream, l2: int, reps: int = 15) -> float:
    """Median µs of one launch with L2 flushed just before it: a buffer of twice the L2 size
    is written, then the launch alone is bracketed by CUDA events on its stream."""
    import torch
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=stream.device)
    samples = []
    for i in range(reps + 2):
        with torch.cuda.stream(stream):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(0)
            b.record(stream)
        stream.synchronize()
        if i >= 2:
            samples.append(a.elapsed_time(b) * 1e3)
    del flush
    return statistics.median(samples)


def run_configs(h, dev, stream, l2: int, pdl: int, peak: float):
    """Every GEMV of the benchmark configurations, one at a time: µs per call in the graph
    protocol (programmatic dependent launch as set), GB/s and fraction of the HBM peak, and
    the single-launch latency with L2 flushed (no dependent launch).  Config 4's mixed layer
    is also timed as a step of its 7 GEMVs.  Returns {config: {...}} and the launch count."""
    import torch

    from quantized_weight_dequant_gb300 import qgemv

    done, out, launches = {}, {}, 0
    for cname, gl in CONFIGS:
        rows = {}
        for label, fmt, N, K in gl:
            key = (fmt, N, K)
            if key not in done:
                W = torch.from_numpy(synth.make_weights(fmt, N, K, WEIGHT_SEED + N + K + fmt)).to(dev)
                copies = max(2, math.ceil(3 * l2 / W.numel()))
                Ws = [W] + [W.clone() for _ in range(copies - 1)]
                x = torch.from_numpy(synth.make_x(fmt, K, WEIGHT_SEED).view(np.int16).copy()).to(dev)
                y = torch.empty(N, dtype=torch.float32, device=dev)

                def launch(c, Ws=Ws, x=x, y=y, fmt=fmt, N=N, K=K):
                    qgemv.run(h, fmt, x, Ws[c], N, K, y, stream=stream)

                us = graph_us(launch, copies, stream)
                qgemv.set_option(h, qgemv.OPT_PDL, 0)
                us1 = flushed_single_us(launch, stream, l2)
                qgemv.set_option(h, qgemv.OPT_PDL, pdl)
                st = qgemv.check_error(h, stream)
                if st != qgemv.OK:
                    raise RuntimeError(f"qgemv error {qgemv.status_string(st)} on {key}")
                b = gemv_bytes(fmt, N, K)
                done[key] = {"shape": f"{synth.FORMAT_NAMES[fmt]} {N}x{K}", "us": round(us, 3),
                             "GB/s": round(b / (us * 1e-6) / 1e9, 1), "frac": round(b / (us * 1e-6) / 1e9 / peak, 4),
                             "us_single_l2_flushed": round(us1, 3), "MB": round(b / 1e6, 3)}
                launches += 200 * 8 + 17
                del Ws, W, x, y
            rows[label] = done[key]
        out[cname] = {"gemvs": rows}
    # the mixed layer as one step: 7 launches in order, x of the layer shared, down on its own x
    gl = dict(CONFIGS)["config4_layer_mixed"]
    Wl, xs, ys = [], {}, []
    step_w = sum(synth.packed_bytes(f, n, k) for _, f, n, k in gl)
    copies = max(2, math.ceil(3 * l2 / step_w))
    for i, (label, fmt, N, K) in enumerate(gl):
        W = torch.from_numpy(synth.make_weights(fmt, N, K, WEIGHT_SEED + i)).to(dev)
        Wl.append([W] + [W.clone() for _ in range(copies - 1)])
        xs.setdefault(K, torch.from_numpy(synth.make_x(fmt, K, WEIGHT_SEED + K).view(np.int16).copy()).to(dev))
        ys.append(torch.empty(N, dtype=torch.float32, device=dev))

    def step(c):
        for i, (label, fmt, N, K) in enumerate(gl):
            qgemv.run(h, fmt, xs[K], Wl[i][c], N, K, ys[i], stream=stream)

    us = graph_us(step, copies, stream, R=50)
    sb = sum(gemv_bytes(f, n, k) for _, f, n, k in gl)
    out["config4_layer_mixed"]["step"] = {"launches": len(gl), "us": round(us, 3),
                                          "GB/s": round(sb / (us * 1e-6) / 1e9, 1),
                                          "frac": round(sb / (us * 1e-6) / 1e9 / peak, 4)}
    launches += 50 * 8 * len(gl)
    del Wl, xs, ys
    torch.cuda.empty_cache()
    return out, launches


def run_ours(args, gemvs, rank, world):
    import torch

    from quantized_weight_dequant_gb300 import qgemv
    from quantized_weight_dequant_gb300.build import build_library

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build_library()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    h = qgemv.create(local)
    if args.pdl:
        qgemv.set_option(h, qgemv.OPT_PDL, 1)

    # Inputs: one seeded matrix per GEMV, cloned on the device into C rotating copies.
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    step_w_bytes = sum(synth.packed_bytes(f, n, k) for _, f, n, k, _ in gemvs)
    copies = max(2, math.ceil(3 * l2 / step_w_bytes))
    xs, Ws, ys = {}, [], []
    B = args.batch  # activation vectors per GEMV
    for gi, (label, fmt, N, K, xk) in enumerate(gemvs):
        seed = WEIGHT_SEED + gi + 100 * rank
        W = synth.make_weights(fmt, N, K, seed)
        Wd = torch.from_numpy(W).to(dev)
        Ws.append([Wd] + [Wd.clone() for _ in range(copies - 1)])
        if (xk, K, fmt) not in xs:
            xb = np.stack([synth.make_x(fmt, K, seed + 7919 * m) for m in range(B)])  # [B, K]
            xs[(xk, K, fmt)] = torch.from_numpy(xb.view(np.int16).copy()).to(dev)
        ys.append(torch.empty((B, N), dtype=torch.float32, device=dev))
        del W
    # Every x of a step in one device buffer and every output in another (views at 16-byte
    # offsets), so the end-to-end run moves a step's inputs and results with one copy each way.
    xoff, off = {}, 0
    for k in xs:
        xoff[k] = off
        off += (xs[k].numel() + 7) // 8 * 8
    xall = torch.zeros(off, dtype=torch.int16, device=dev)
    for k in list(xs):
        v = xall[xoff[k]:xoff[k] + xs[k].numel()].view(xs[k].shape)
        v.copy_(xs[k])
        xs[k] = v
    yoff, off = [], 0
    for y in ys:
        yoff.append(off)
        off += (y.numel() + 3) // 4 * 4
    yall = torch.empty(off, dtype=torch.float32, device=dev)
    ys = [yall[o:o + y.numel()].view(y.shape) for o, y in zip(yoff, ys)]
    units = launch_units(args.workload, gemvs)
    grouped = set(GROUPS.get(args.workload, {}).values())
    for label, idx, sw in units:
        if sw:
            ys[idx[1]] = None  # the up matrix of a SwiGLU pair has no output of its own
    step_bytes = sum(unit_bytes(gemvs, idx, sw, B) for _, idx, sw in units)
    stream = torch.cuda.Stream(device=dev)

    # A second set of x / y buffers, for the end-to-end run's double buffering.
    xall2 = xall.clone()
    xs2 = {k: xall2[xoff[k]:xoff[k] + v.numel()].view(v.shape) for k, v in xs.items()}
    yall2 = torch.empty_like(yall)
    ys2 = [None if y is None else yall2[o:o + y.numel()].view(y.shape) for o, y in zip(yoff, ys)]
    bufs = [(xs, ys), (xs2, ys2)]

    def launch(ui, c, s, bs=0):
        """Launch unit ui on weight copy c, with buffer set bs."""
        label, idx, sw = units[ui]
        _, fmt, N, K, xk = gemvs[idx[0]]
        xv, yv = bufs[bs]
        x = xv[(xk, K, fmt)]
        if label not in grouped and B > 1:
            qgemv.run_batch(h, fmt, x, B, Ws[idx[0]][c], N, K, yv[idx[0]], stream=s)
        elif label not in grouped:
            qgemv.run(h, fmt, x, Ws[idx[0]][c], N, K, yv[idx[0]], stream=s)
        elif sw:
            qgemv.run_group(h, x, K, [qgemv.problem(fmt, Ws[idx[0]][c], N, yv[idx[0]], packed_W_up=Ws[idx[1]][c],
                                                    swiglu=True)], stream=s)
        else:
            qgemv.run_group(h, x, K, [qgemv.problem(gemvs[i][1], Ws[i][c], gemvs[i][2], yv[i]) for i in idx], stream=s)

    def step(i, s, bs=0):
        c = i % copies
        for ui in range(len(units)):
            launch(ui, c, s, bs)

    # sanity: one step, checked for errors, before anything is captured
    with torch.cuda.stream(stream):
        step(0, stream)
    stream.synchronize()
    st = qgemv.check_error(h, stream)
    if st != qgemv.OK:
        raise RuntimeError(f"qgemv error {qgemv.status_string(st)}")

    spg = largest_divisor_le(args.steps, args.graph_steps)
    reps = args.steps // spg
    g = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.graph(g, stream=stream):
        for i in range(spg):
            step(i, stream)
    launches_per_step = len(units)  # one kernel per launch unit (split-K adds its column sums in-kernel)

    # warm-up: at least W steps
    warm_reps = max(1, math.ceil(args.warmup / spg))
    with torch.cuda.stream(stream):
        for _ in range(warm_reps):
            g.replay()
    stream.synchronize()

    clocks = Clocks(local, str(getattr(props, "uuid", "")) or None) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = e0.elapsed_time(e1)
    clk = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    st = qgemv.check_error(h, stream)
    if st != qgemv.OK:
        raise RuntimeError(f"qgemv error after timing: {qgemv.status_string(st)}")

    value = whole_job_gbs(world, args.steps, step_bytes, elapsed_ms)
    ms_per_step = elapsed_ms / args.steps

    # Per-launch duration (CUDA events around graph replays of R launches of one unit).
    per_call = {}
    for ui, (label, idx, sw) in enumerate(units):
        R = 200
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=stream):
            for i in range(R):
                launch(ui, i % copies, stream)
        with torch.cuda.stream(stream):
            gg.replay()
        stream.synchronize()
        samples = []
        for _ in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                gg.replay()
                b.record(stream)
            stream.synchronize()
            samples.append(a.elapsed_time(b) * 1e3 / R)
        us = statistics.median(samples)
        shape = " + ".join(f"{synth.FORMAT_NAMES[gemvs[i][1]]} {gemvs[i][2]}x{gemvs[i][3]}" for i in idx)
        per_call[label] = {"us": us, "GB/s": unit_bytes(gemvs, idx, sw, B) / (us * 1e-6) / 1e9,
                           "shape": shape + (" (SwiGLU pair)" if sw else "")}
        if label not in grouped:
            per_call[label]["plan"] = qgemv.describe(h, gemvs[idx[0]][1], gemvs[idx[0]][2], gemvs[idx[0]][3])
        del gg
    if args.dense_context and B == 1:
        # Context only (a library, not this product): the same GEMV with dense bf16 weights
        # through cuBLAS (torch.mv), same protocol (graph of 200 launches over rotating copies
        # that exceed L2), and the speed-up of the packed format over it.
        for ui, (label, idx, sw) in enumerate(units):
            if label in grouped:
                continue
            _, fmt, N, K, _ = gemvs[idx[0]]
            dc = max(2, math.ceil(3 * l2 / (2 * N * K)))
            Wb = [torch.randn(N, K, device=dev, dtype=torch.bfloat16) * 0.02 for _ in range(dc)]
            xb = torch.randn(K, device=dev, dtype=torch.bfloat16)
            with torch.cuda.stream(stream):
                torch.mv(Wb[0], xb)  # cuBLAS sets up its handle outside the capture
            stream.synchronize()
            R = 200
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=stream):
                for i in range(R):
                    torch.mv(Wb[i % dc], xb)
            with torch.cuda.stream(stream):
                gg.replay()
            stream.synchronize()
            samples = []
            for _ in range(7):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    gg.replay()
                    b.record(stream)
                stream.synchronize()
                samples.append(a.elapsed_time(b) * 1e3 / R)
            dus = statistics.median(samples)
            per_call[label]["dense_bf16_cublas_us"] = dus
            per_call[label]["speedup_over_dense_bf16"] = dus / per_call[label]["us"]
            del gg, Wb
    dom = max(units, key=lambda u_: unit_bytes(gemvs, u_[1], u_[2], B))[0]
    peak, peak_kind = load_peaks()
    achieved = per_call[dom]["GB/s"]
    dom_idx = [u_ for u_ in units if u_[0] == dom][0][1]
    tkey = ("+".join(f"{synth.FORMAT_NAMES[gemvs[i][1]]}_{gemvs[i][2]}x{gemvs[i][3]}" for i in dom_idx)
            + ("_group" if dom in grouped else "") + (f"_batch{B}" if B > 1 else ""))
    traffic, traffic_cmd = load_traffic(qgemv.build_marker(), tkey)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic,
                "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one {tkey} launch of this "
                                   f"build (profiles/roofline_traffic.json): {traffic_cmd}") if traffic is not None
                else (traffic_cmd or f"no ncu record of {tkey} for this build"),
                "kernel": f"{'group_kernel' if dom in grouped else 'batch_kernel' if B > 1 else 'stream_kernel'} "
                          f"{per_call[dom]['shape']}" + (f" x {B} vectors" if B > 1 else ""),
                "peak_kind": f"hbm_gbs of {peak_kind} (copy bandwidth)",
                "achieved_how": "algorithmic bytes per launch / mean launch duration over graph replays of 200 "
                                "launches rotating weight copies (CUDA events on the launch stream)"}

    # End to end through the public API: the step's packed x from pinned host memory to the
    # device (one copy), one qgemv call per launch unit, the packed outputs back (one copy).
    # Steps are pipelined as a serving loop runs independent requests: step i's input copy and
    # step i - 1's result copy run on copy streams while step i - 1 / i compute, with two
    # device buffer sets (step i uses set i % 2).  Events keep each buffer safe: a step's
    # compute waits for its input copy and for the result copy that last read its y buffer;
    # an input copy waits for the compute that last read its x buffer.
    e2e_steps = min(args.steps, 2000)
    hx = torch.empty(xall.shape, dtype=torch.int16).pin_memory()
    hx.copy_(xall.cpu())
    hys = [torch.empty(yall.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    xalls, yalls = [xall, xall2], [yall, yall2]
    h2d = 2 * xall.numel()
    d2h = 4 * yall.numel()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_steps_run(n):
        """n pipelined steps on `stream` (compute), s_in and s_out (copies); joined at the end."""
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        computed = [None, None]  # event: the last compute that used buffer set p
        copied_out = [None, None]  # event: the last result copy of buffer set p
        for i in range(n):
            p = i % 2
            if computed[p] is not None:
                s_in.wait_event(computed[p])
            with torch.cuda.stream(s_in):
                xalls[p].copy_(hx, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            if copied_out[p] is not None:
                stream.wait_event(copied_out[p])
            step(i, stream, p)
            computed[p] = torch.cuda.Event()
            computed[p].record(stream)
            s_out.wait_event(computed[p])
            with torch.cuda.stream(s_out):
                hys[p].copy_(yalls[p], non_blocking=True)
            copied_out[p] = torch.cuda.Event()
            copied_out[p].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    # The steps are recorded in a CUDA graph, as a decode loop would run them: every replayed
    # step still copies its inputs in and its results out (memcpy nodes), without the host's
    # per-call launch cost.  If the copies cannot be captured the steps run eagerly.
    e2e_spg = largest_divisor_le(e2e_steps, 100)
    with torch.cuda.stream(stream):
        e2e_steps_run(5)
    stream.synchronize()
    ge = None
    try:
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            e2e_steps_run(e2e_spg)
        with torch.cuda.stream(stream):
            ge.replay()
        stream.synchronize()
    except RuntimeError:
        ge = None
        torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if ge is not None:
            for _ in range(e2e_steps // e2e_spg):
                ge.replay()
        else:
            e2e_steps_run(e2e_steps)
        b.record(stream)
    stream.synchronize()
    e2e_ms = a.elapsed_time(b)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e = {"value": whole_job_gbs(world, e2e_steps, step_bytes, e2e_ms), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "ms_per_step": e2e_ms / e2e_steps,
           "how": ("CUDA graph of %d steps, replayed" % e2e_spg if ge is not None else "eager, stream-ordered")
                  + ": per step one pinned H2D copy of the step's packed x, one qgemv_run / qgemv_run_group / "
                  "qgemv_run_batch per launch unit, one D2H copy of the packed outputs; weights resident; "
                  "copies on two copy streams overlap the neighbouring steps' compute (two device buffer sets, "
                  "event-ordered)"}

    configs = None
    if rank == 0 and not args.no_configs and B == 1:
        configs, _ = run_configs(h, dev, stream, l2, args.pdl, peak)
        configs["how"] = ("each GEMV alone: µs per call = a CUDA graph of 200 launches over rotating weight copies "
                          "(> 3x L2), programmatic dependent launch %s, CUDA events; us_single_l2_flushed = one "
                          "launch after writing a buffer of twice the L2 size, no dependent launch, median of 15; "
                          "frac against hbm_gbs of MEASURED_PEAKS.json" % ("on" if args.pdl else "off"))

    cpu = cpu1 = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        sampler = OracleSampler(gemvs, threads, batch=B)
        rates, spent = [], 0.0
        while spent < args.cpu_seconds or len(rates) < 3:  # repeated bounded samples, median rate
            rate, dt, sample = sampler.run(max(0.5, args.cpu_seconds / 5))
            rates.append(rate)
            spent += dt
        sampler.close()
        cpu = {"value": statistics.median(rates), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{sample}; median of {len(rates)} samples, {spent:.1f} s wall in total"}
        sampler1 = OracleSampler(gemvs, 1, batch=B)  # the same oracle on one thread
        rates1, spent1 = [], 0.0
        while spent1 < args.cpu_seconds / 2 or len(rates1) < 3:
            rate, dt, sample1 = sampler1.run(max(0.3, args.cpu_seconds / 10))
            rates1.append(rate)
            spent1 += dt
        sampler1.close()
        cpu1 = {"value": statistics.median(rates1), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{sample1}; median of {len(rates1)} samples, {spent1:.1f} s wall in total"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": args.workload,
                           "shapes": [f"{g_[0]}:{synth.FORMAT_NAMES[g_[1]]}:{g_[2]}x{g_[3]}" for g_ in gemvs],
                           "bytes_per_step": step_bytes,
                           "l2": f"inputs larger than L2: {copies} rotating weight copies = "
                                 f"{copies * step_w_bytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB",
                           "timing": f"CUDA graph of {spg} steps replayed {reps}x, CUDA events",
                           "batch": B,
                           "launches": [f"{u_[0]}:{'+'.join(gemvs[i][0] for i in u_[1])}"
                                        + (":swiglu" if u_[2] else "") for u_ in units],
                           "pdl": bool(args.pdl)},
                "roofline": roofline, "cpu_baseline": cpu, "cpu_baseline_1_thread": cpu1, "e2e": e2e,
                "configs": configs,
                "gpu_launches": launches_per_step * args.steps, "clocks": clk,
                "us_per_call": per_call, "impl": "ours", "build": qgemv.build_marker(),
                "gpu": props.name}
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--graph-steps", type=int, default=200)
    ap.add_argument("--pdl", type=int, default=1,
                    help="1 (default): launch with programmatic dependent launch, as a decode loop would")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="only run this many plain launches of each GEMV (for a profiler) and exit")
    ap.add_argument("--only", default=None, help="with --profile-launches: the one GEMV label to run")
    ap.add_argument("--batch", type=int, default=1,
                    help="activation vectors per GEMV (1..8; > 1 runs qgemv_run_batch, ungrouped workloads only)")
    ap.add_argument("--dense-context", action="store_true",
                    help="also time each GEMV with dense bf16 weights through cuBLAS (context only)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="M > 0: time the NVFP4 GEMM of M activation rows (the prefill path) instead of the GEMV")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing every GEMV of the five benchmark configurations")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 1 <= args.batch <= 8:
        ap.error("--batch must be in 1..8")
    if args.batch > 1 and GROUPS.get(args.workload):
        ap.error("--batch > 1 applies to workloads without grouped launches")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    gemvs = WORKLOADS[args.workload]
    if args.prefill < 0:
        ap.error("--prefill must be >= 0")
    if args.prefill and args.profile_launches:
        return run_profile_prefill(args, gemvs)
    if args.profile_launches:
        return run_profile_launches(args, gemvs)
    if args.prefill:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--prefill has no oracle arm: the oracle is a GEMV"}))
            return 0
        return run_prefill(args, gemvs, rank, world)
    if args.impl == "reference":
        return run_reference(args, gemvs, rank, world)
    return run_ours(args, gemvs, rank, world)


if __name__ == "__main__":
    sys.exit(main())
