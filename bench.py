#!/usr/bin/env python3
"""Benchmark of the FP32 row-reduction hot path on one GB300 (or N replicas).

Metric: achieved HBM GB/s (algorithmic bytes / time) and microseconds per op.
Default workload: softmax, RMSNorm and LayerNorm at 768 x 6144 (x ~ N(0,1),
weight ~ U(0.5,1.5), bias ~ N(0,0.1), eps 1e-5, seed 2), each under the
unordered and the ordered (OT-1024) policy: one step = these 6 launches, each
on its own input and output buffers. Inputs are resident in HBM when timing
starts; rotating buffer sets keep every launch's data out of L2.

Timed regions (CUDA events on the launching stream, one nvidia-smi clock
record around all of them):
  1. the headline `value`: CUDA graphs of exactly --steps unrolled steps;
  2. every kernel of the step alone: a graph of 200 back-to-back launches,
     replayed 9 times, the median replay (the roofline kernel is the slowest);
  3. `per_op`: the same protocol for every configuration of the workload list
     (cross-entropy 4096x50257, the long-row sweep, the small shapes);
  4. synchronized single calls (GPU time between events, and host wall time
     through the C-ABI including the synchronisation), median of 30.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--suite] [--no-per-op]

``--impl reference`` times the CPU oracle (serial FP64 definitions and the
OT-1024 emulation) on a bounded row sample of the same workload.
``--suite`` prints one line per workload (every configuration) and exits.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "achieved HBM GB/s and µs/op per op×shape on 1 GB300 (fraction of ~8 TB/s)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# workload name -> list of (op, synth workload, order)
TRIO = [("softmax", "softmax_768x6144"), ("rmsnorm", "rmsnorm_768x6144"), ("layernorm", "layernorm_768x6144")]
WORKLOADS = {
    "trio_768x6144": [(op, w, o) for o in ("unordered", "ordered") for op, w in TRIO],
}
for _name, _w in synth.WORKLOADS.items():
    WORKLOADS[_name] = [(_w["op"], _name, "unordered")]
    if _name.endswith("768x6144"):
        WORKLOADS[_name + "_ordered"] = [(_w["op"], _name, "ordered")]
        if _w["op"] in ("softmax", "rmsnorm", "layernorm", "row_sum", "row_minmax"):
            for _f in ("fold_left", "fold_right"):
                WORKLOADS[f"{_name}_{_f}"] = [(_w["op"], _name, _f)]
DEFAULT_WORKLOAD = "trio_768x6144"


def alg_bytes(op, rows, cols):
    """Algorithmic bytes of one launch: every input read once, every output written once."""
    e = rows * cols
    return {"softmax": 8 * e, "rmsnorm": 8 * e + 4 * cols, "layernorm": 8 * e + 8 * cols,
            "cross_entropy": 4 * e + 12 * rows,
            # fused residual norms: x and r read, y and h = x + r written
            "add_rmsnorm": 16 * e + 4 * cols, "add_layernorm": 16 * e + 8 * cols,
            # standalone row reductions: x read, one (two) values per row written
            "row_sum": 4 * e + 4 * rows, "row_max": 4 * e + 4 * rows, "row_min": 4 * e + 4 * rows,
            "row_minmax": 4 * e + 8 * rows,
            # reductions over axis 0: x read, one (two) values per column written
            "axis_sum": 4 * e + 4 * cols, "axis_max": 4 * e + 4 * cols, "axis_min": 4 * e + 4 * cols,
            "axis_minmax": 4 * e + 8 * cols,
            # backward passes: inputs read once, dx (and the column gradients) written once
            "softmax_bwd": 12 * e, "cross_entropy_bwd": 8 * e + 12 * rows,
            "rmsnorm_bwd": 12 * e + 8 * cols, "layernorm_bwd": 12 * e + 12 * cols}[op]


# The sources that define, select or launch the default step's kernels (the
# unordered row kernels and the ordered tree of softmax, RMSNorm, LayerNorm):
# a committed traffic record counts only while none of them has changed.
STEP_SOURCES = ["k_softmax.cu", "k_rmsnorm.cu", "k_layernorm.cu", "k_ordered.cu", "tr_dispatch.cuh",
                "tr_split_kernels.cuh", "tr_row_kernels.cuh", "tr_device.cuh", "tr_internal.h", "tr_api.cu", "tr_ot.cuh",
                "tr_plan.cpp", "tr_plan.h", "tr_wave_kernels.cuh", "k_wave.cu", "k_wave_ordered.cu"]

# The configurations whose kernels `per_op` reports beside the step's: every
# workload of the benchmark's list (op, synthetic workload, policy).
PER_OP_CONFIGS = [
    ("softmax", "softmax_37x1537", "unordered"),
    ("rmsnorm", "rmsnorm_256x3072", "unordered"), ("layernorm", "layernorm_256x3072", "unordered"),
    ("rmsnorm", "rmsnorm_64x12289", "unordered"), ("layernorm", "layernorm_64x12289", "unordered"),
    ("cross_entropy", "cross_entropy_4096x50257", "unordered"),
    ("softmax", "softmax_16x65536", "unordered"), ("softmax", "softmax_16x262144", "unordered"),
    ("softmax", "softmax_16x1048576", "unordered"), ("softmax", "softmax_65536x128", "unordered"),
    ("layernorm", "layernorm_16x65536", "unordered"), ("layernorm", "layernorm_16x262144", "unordered"),
    ("layernorm", "layernorm_16x1048576", "unordered"), ("layernorm", "layernorm_65536x128", "unordered"),
]
KERNEL_LAUNCHES = 200   # back-to-back launches per timed graph
KERNEL_ROUNDS = 9       # replays of that graph; the median is reported
SINGLE_CALLS = 30       # synchronized single calls per kernel


def kernel_source_hash():
    csrc = os.path.join(ROOT, "fp32_row_reduction_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(STEP_SOURCES):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        v = float(json.load(open(p))["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(key):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p))
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    ent = rec.get("launches", {}).get(key)
    return None if ent is None else ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]) if f[3] not in ("[N/A]", "") else 0.0, f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        maxp = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * maxp] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded), "power_w_max": maxp}


# ----------------------------------------------------------------- our arm

class Launch:
    """One launch of the step: op, policy, its input/output buffer sets."""

    def __init__(self, op, workload, order, sets, device):
        import fp32_row_reduction_gb300 as tr
        self.tr = tr
        self.op, self.workload, self.order = op, workload, order
        w = synth.WORKLOADS[workload]
        self.rows, self.cols = w["rows"], w["cols"]
        base = synth.workload_inputs(workload, device=device)
        if op == "softmax_bwd":  # y = the forward output, by this library's softmax
            base = {"y": tr.softmax(base["x"]), "dy": base["dy"]}
        self.inputs = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(sets - 1)]
        if op == "cross_entropy" or op.startswith("row_"):
            self.outputs = [torch.empty(self.rows, device=device) for _ in range(sets)]
        elif op.startswith("axis_"):
            self.outputs = [torch.empty(self.cols, device=device) for _ in range(sets)]
        else:
            self.outputs = [torch.empty_like(base["x"] if "x" in base else base["y"]) for _ in range(sets)]
        # fused residual norms also write h = x + r
        self.h = [torch.empty_like(base["x"]) for _ in range(sets)] if op.startswith("add_") else None
        if op == "row_minmax":  # the maxima (the minima go to outputs)
            self.h = [torch.empty(self.rows, device=device) for _ in range(sets)]
        if op == "axis_minmax":
            self.h = [torch.empty(self.cols, device=device) for _ in range(sets)]
        # norm backward passes: the column gradients and one workspace per buffer set
        self.aux = None
        if op in ("rmsnorm_bwd", "layernorm_bwd"):
            nws = tr.norm_backward_workspace_bytes(self.rows, self.cols)
            self.aux = [{"dw": torch.empty(self.cols, device=device), "db": torch.empty(self.cols, device=device),
                         "ws": torch.empty(nws, dtype=torch.uint8, device=device)} for _ in range(sets)]
        self.bytes = alg_bytes(op, self.rows, self.cols)
        self.key = f"{op}/{self.order}/{self.rows}x{self.cols}"

    def __call__(self, s, stream=None):
        d = self.inputs[s]
        if self.op == "softmax_bwd":
            self.tr.softmax_backward(d["y"], d["dy"], out=self.outputs[s], order=self.order, stream=stream)
        elif self.op == "cross_entropy_bwd":
            self.tr.cross_entropy_backward(d["x"], d["labels"], d["dloss"], out=self.outputs[s], order=self.order,
                                           stream=stream)
        elif self.op == "rmsnorm_bwd":
            a = self.aux[s]
            self.tr.rmsnorm_backward(d["x"], d["w"], d["dy"], order=self.order, dx=self.outputs[s], dw=a["dw"],
                                     workspace=a["ws"], stream=stream)
        elif self.op == "layernorm_bwd":
            a = self.aux[s]
            self.tr.layernorm_backward(d["x"], d["w"], d["dy"], order=self.order, dx=self.outputs[s],
                                       dgamma=a["dw"], dbeta=a["db"], workspace=a["ws"], stream=stream)
        else:
            self.tr.run_op(self.op, d, out=self.outputs[s], order=self.order, stream=stream,
                           h_out=None if self.h is None else self.h[s])

    def plan(self):
        if self.op.endswith("_bwd"):
            return {"kind": "backward", "block_threads": 256,
                    "slots": next((k for k in (1, 2, 4, 6, 8) if self.cols <= 1024 * k), 0)}
        if self.op.startswith("axis_"):
            sm = torch.cuda.get_device_properties(0).multi_processor_count
            splits, tiles = self.tr.axis_launch_shape(self.op[len("axis_"):], 1, self.rows, self.cols, sm, self.order)
            return {"kind": "axis", "splits": splits, "tiles": tiles, "block_threads": 256,
                    "grid_ctas": splits * tiles}
        return self.tr.plan_for(self.op, self.rows, self.cols, self.order)


def pick_sets(launches_bytes, l2=126 << 20):
    per_set = sum(launches_bytes)
    return max(2, math.ceil(2 * l2 / per_set))


def build_graph(launches, steps, sets, first_set, timing):
    """Capture `steps` unrolled steps; returns (graph, events[step][k]) with per-launch events."""
    g = torch.cuda.CUDAGraph()
    evs = []
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    # one eager call of each launch on the capture stream first: split-row
    # plans allocate their per-stream workspace on a stream's first call
    with torch.cuda.stream(stream):
        for ln in launches:
            ln(first_set % sets)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            s = (first_set + i) % sets
            row = []
            for ln in launches:
                if timing:
                    e = torch.cuda.Event(enable_timing=True, external=True)
                    e.record()
                    row.append(e)
                ln(s)
            if timing:
                e = torch.cuda.Event(enable_timing=True, external=True)
                e.record()
                row.append(e)
            evs.append(row)
    return g, evs


def max_over_ranks(ms, device):
    """The slowest rank's time: every replica waits for it (all-reduce MAX)."""
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, steps, step_bytes, elapsed_ms):
    """Whole-job throughput: every replica's steps over the slowest rank's time."""
    return world * steps * step_bytes / (elapsed_ms * 1e-3) / 1e9


def workload_config(specs, sets=None):
    """The `config` object of both arms: the workload and what a step launches."""
    return {"workload": specs["name"], "launches_per_step": len(specs["launches"]),
            "shapes": sorted({f"{synth.WORKLOADS[w]['rows']}x{synth.WORKLOADS[w]['cols']}"
                              for _, w, _ in specs["launches"]}),
            "policies": sorted({o for _, _, o in specs["launches"]}),
            "l2": "inputs larger than L2: rotating buffer sets, every launch reads data not used since "
                  "more than twice the L2 size was touched"}


def timed_graph_us(ln, sets, n=KERNEL_LAUNCHES, rounds=KERNEL_ROUNDS):
    """Median microseconds per launch of `rounds` replays of a graph of `n`
    back-to-back launches of one kernel (its rotating buffer sets)."""
    g = build_graph([ln], n, sets, 0, timing=False)[0]
    g.replay()
    torch.cuda.synchronize()
    samples = []
    for _ in range(rounds):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        g.replay()
        t1.record()
        t1.synchronize()
        samples.append(1e3 * t0.elapsed_time(t1) / n)
    del g
    return statistics.median(samples), samples


def timed_segments_us(entries, n=KERNEL_LAUNCHES, rounds=KERNEL_ROUNDS):
    """Per-launch microseconds of several kernels from ONE graph: for each
    (launch, buffer sets) entry a segment of `n` back-to-back launches, with a
    timing event at every segment boundary; the graph is replayed `rounds`
    times and each segment's median is reported. (On this driver, every CUDA
    graph instantiated after a process's second runs each kernel node about
    0.4 us slower, a plain torch.mul included; one graph for all the per-kernel
    timings keeps them in the state of the step graph that `value` times.)"""
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    # one eager call of each launch on the capture stream first (split plans
    # allocate their per-stream workspace on a stream's first call)
    with torch.cuda.stream(stream):
        for ln, sets in entries:
            ln(0)
    torch.cuda.synchronize()
    evs = []
    with torch.cuda.graph(g, stream=stream):
        for ln, sets in entries:
            e = torch.cuda.Event(enable_timing=True, external=True)
            e.record()
            evs.append(e)
            for i in range(n):
                ln(i % sets)
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        evs.append(e)
    g.replay()
    torch.cuda.synchronize()
    samples = [[] for _ in entries]
    for _ in range(rounds):
        g.replay()
        torch.cuda.synchronize()
        for k in range(len(entries)):
            samples[k].append(1e3 * evs[k].elapsed_time(evs[k + 1]) / n)
    del g
    return [(statistics.median(sm), sm) for sm in samples]


def single_call_us(ln, sets, reps=SINGLE_CALLS):
    """Synchronized single calls: GPU time between events around one call, and
    host wall time of the call through the C-ABI plus the synchronisation
    (medians; the buffer sets rotate, so every call reads cold data)."""
    gpu, host = [], []
    for i in range(reps):
        s = i % sets
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record()
        ln(s)
        e1.record()
        e1.synchronize()
        host.append(1e6 * (time.perf_counter() - t0))
        gpu.append(1e3 * e0.elapsed_time(e1))
    return statistics.median(gpu), statistics.median(host)


def op_entry(ln, us, samples, peak, single=None):
    e = {"us": round(us, 3), "gbs": round(ln.bytes / (us * 1e3), 1),
         "frac_of_peak": round(ln.bytes / (us * 1e3) / peak, 4),
         "frac_of_8tbs": round(ln.bytes / (us * 1e3) / 8000.0, 4),
         "us_rounds": [round(v, 3) for v in samples], "alg_bytes": ln.bytes, "plan": ln.plan()}
    if single is not None:
        e["single_call_gpu_us"], e["single_call_e2e_us"] = round(single[0], 3), round(single[1], 3)
    return e


def run_ours(args, rank, world):
    import fp32_row_reduction_gb300 as tr
    tr.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    specs = WORKLOADS[args.workload]
    probe = [alg_bytes(op, synth.WORKLOADS[w]["rows"], synth.WORKLOADS[w]["cols"]) for op, w, _ in specs]
    # enough buffer sets that a step, and also each kernel alone (timed region 2),
    # cycles through more than twice the L2 before reusing a buffer
    sets = max([pick_sets(probe)] + [pick_sets([b]) for b in probe])
    launches = [Launch(op, w, o, sets, dev) for op, w, o in specs]
    step_bytes = sum(ln.bytes for ln in launches)
    torch.cuda.synchronize()

    # warm-up (eager: also fills the plan cache before capture)
    for i in range(max(args.warmup, 1)):
        for ln in launches:
            ln(i % sets)
    torch.cuda.synchronize()

    K = args.steps
    U = min(K, args.unroll)
    rem = K % U
    # timed region 1 (the step throughput): graphs of unrolled steps with no
    # nodes between the launches, so back-to-back launches overlap as they would
    # in an application (programmatic dependent launch)
    g_main = build_graph(launches, U, sets, 0, timing=False)[0]
    g_rem = build_graph(launches, rem, sets, U % sets, timing=False)[0] if rem else None
    for g in (g_main,) + ((g_rem,) if g_rem is not None else ()):
        g.replay()  # graph warm-up
    torch.cuda.synchronize()

    def timed(replays):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        replays()
        t1.record()
        t1.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return t0.elapsed_time(t1)

    def main_steps():
        for _ in range(K // U):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()

    peak, peak_kind = measured_peak()
    with ClockSampler(dev.index) as clk:
        elapsed_ms = timed(main_steps)
        del g_main, g_rem
        # timed regions 2 and 3: each kernel of the step, and every other
        # configuration of the list, alone: segments of 200 back-to-back
        # launches of one kernel on its own rotating buffers, all in one graph
        # (timed_segments_us), median of 9 replays
        extra = []
        if rank == 0 and not args.no_per_op and args.workload == DEFAULT_WORKLOAD:
            for op, w, o in PER_OP_CONFIGS:
                b = alg_bytes(op, synth.WORKLOADS[w]["rows"], synth.WORKLOADS[w]["cols"])
                xs = pick_sets([b])
                ln = Launch(op, w, o, xs, dev)
                for i in range(3):
                    ln(i % xs)
                extra.append((ln, xs))
            torch.cuda.synchronize()
        segs = timed_segments_us([(ln, sets) for ln in launches] + extra)
        per = segs[:len(launches)]
        per_us = [p[0] for p in per]
        # timed region 4: synchronized single calls
        singles = [single_call_us(ln, sets) for ln in launches]
        per_op = {ln.key: op_entry(ln, per[k][0], per[k][1], peak, singles[k]) for k, ln in enumerate(launches)}
        for (ln, xs), (us, samples) in zip(extra, segs[len(launches):]):
            per_op[ln.key] = op_entry(ln, us, samples, peak, single_call_us(ln, xs, reps=10))
        del extra
        torch.cuda.empty_cache()

    if world > 1:
        elapsed_ms = max_over_ranks(elapsed_ms, dev)

    e2e = measure_e2e(launches, args, dev) if rank == 0 else None
    cpu = cpu_baseline(launches, args) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank != 0:
        return None

    dom = max(range(len(launches)), key=lambda k: per_us[k])
    dl = launches[dom]
    achieved = dl.bytes / (per_us[dom] * 1e-6) / 1e9
    value = job_gbs(world, K, step_bytes, elapsed_ms)
    config = workload_config({"name": args.workload, "launches": specs})
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config,
        "timing": {"value": "CUDA graphs of exactly `steps` unrolled steps, CUDA events on the launching stream",
                   "per_kernel": f"per kernel, a segment of {KERNEL_LAUNCHES} back-to-back launches on its "
                                 f"rotating buffer sets, every kernel's segment in one CUDA graph with events "
                                 f"at the segment boundaries, replayed {KERNEL_ROUNDS} times; median replay "
                                 f"(us_rounds lists all)",
                   "single_call": "median of synchronized single calls: GPU time between events around the call, "
                                  "and host wall time of the call through the C-ABI plus the synchronisation",
                   "buffer_sets": sets,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dl.key, "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_8tbs": round(achieved / 8000.0, 4),
                     "traffic": traffic_record(dl.key), "alg_bytes_per_launch": dl.bytes,
                     "launch_us": round(per_us[dom], 3)},
        "per_op": per_op,
        "e2e": e2e,
        "gpu_launches": K * len(launches),
        "per_kernel_timing": {"launches_per_kernel": KERNEL_LAUNCHES * KERNEL_ROUNDS,
                              "sum_of_kernels_ms_per_step": round(sum(per_us) / 1e3, 6)},
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def measure_e2e(launches, args, dev):
    """Same metric through the public API with pinned HOST buffers: H2D of each
    launch's inputs, the launches, D2H of the outputs, all inside the timed region.

    Three streams: host-to-device copies, the launches, device-to-host copies.
    A launch waits for its inputs' copy; the copy of its output waits for the
    launch; a copy into a device buffer set waits until the launch that last read
    it has finished, and a launch waits until its output buffer has been copied
    out. Steps alternate over the device buffer sets, so the copies of one launch
    overlap the compute of another, and H2D overlaps D2H on the full-duplex link."""
    host_in = [{k: v.cpu().pin_memory() for k, v in ln.inputs[0].items()} for ln in launches]
    host_out = [ln.outputs[0].cpu().pin_memory() for ln in launches]
    h2d = sum(t.numel() * t.element_size() for d in host_in for t in d.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    steps = max(3, min(args.e2e_steps, args.steps))
    nsets = len(launches[0].inputs)
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [[torch.cuda.Event() for _ in range(nsets)] for _ in launches]
    in_ready, done, out_done = ev(), ev(), ev()

    def one(i):
        s = i % nsets
        for k, ln in enumerate(launches):
            s_in.wait_event(done[k][s])
            with torch.cuda.stream(s_in):
                for name, t in host_in[k].items():
                    ln.inputs[s][name].copy_(t, non_blocking=True)
            in_ready[k][s].record(s_in)
            s_comp.wait_event(in_ready[k][s])
            s_comp.wait_event(out_done[k][s])
            ln(s, stream=s_comp)
            done[k][s].record(s_comp)
            s_out.wait_event(done[k][s])
            with torch.cuda.stream(s_out):
                host_out[k].copy_(ln.outputs[s], non_blocking=True)
            out_done[k][s].record(s_out)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    step_bytes = sum(ln.bytes for ln in launches)
    return {"value": round(steps * step_bytes / dt / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(1e3 * dt / steps, 4),
            "streams": "H2D, compute and D2H on three streams, ordered by events"}


# ------------------------------------------------------------ the oracle

def oracle_fn(op, order):
    import oracle
    if order in ("fold_left", "fold_right"):
        d = "left" if order == "fold_left" else "right"
        return {"softmax": lambda h: oracle.fold_softmax(h["x"], d),
                "rmsnorm": lambda h: oracle.fold_rmsnorm(h["x"], h["w"], 1e-5, d),
                "layernorm": lambda h: oracle.fold_layernorm(h["x"], h["w"], h["b"], 1e-5, d),
                "cross_entropy": lambda h: oracle.fold_cross_entropy(h["x"], h["labels"], d),
                "row_sum": lambda h: oracle.fold_row_sum(h["x"], d),
                "row_minmax": lambda h: (oracle.fold_row_min(h["x"], d), oracle.fold_row_max(h["x"], d))}[op]
    if order == "ordered":
        return {"softmax": lambda h: oracle.ot_softmax(h["x"]),
                "rmsnorm": lambda h: oracle.ot_rmsnorm(h["x"], h["w"], 1e-5),
                "layernorm": lambda h: oracle.ot_layernorm(h["x"], h["w"], h["b"], 1e-5),
                "cross_entropy": lambda h: oracle.ot_cross_entropy(h["x"], h["labels"]),
                "add_rmsnorm": lambda h: oracle.ot_add_rmsnorm(h["x"], h["r"], h["w"], 1e-5),
                "add_layernorm": lambda h: oracle.ot_add_layernorm(h["x"], h["r"], h["w"], h["b"], 1e-5),
                "row_sum": lambda h: oracle.ot_row_sum(h["x"]), "row_max": lambda h: oracle.ot_row_max(h["x"]),
                "row_min": lambda h: oracle.ot_row_min(h["x"]),
                "row_minmax": lambda h: (oracle.ot_row_min(h["x"]), oracle.ot_row_max(h["x"])),
                "softmax_bwd": lambda h: oracle.ot_softmax_backward(h["y"], h["dy"]),
                "cross_entropy_bwd": lambda h: oracle.ot_cross_entropy_backward(h["x"], h["labels"], h["dloss"]),
                "rmsnorm_bwd": lambda h: oracle.ot_rmsnorm_backward(h["x"], h["w"], h["dy"], 1e-5),
                "layernorm_bwd": lambda h: oracle.ot_layernorm_backward(h["x"], h["w"], h["dy"], 1e-5),
                "axis_sum": lambda h: oracle.ot_axis_sum(h["x"], 0),
                "axis_minmax": lambda h: (oracle.ot_axis_min(h["x"], 0), oracle.ot_axis_max(h["x"], 0))}[op]
    return {"softmax": lambda h: oracle.softmax(h["x"]),
            "rmsnorm": lambda h: oracle.rmsnorm(h["x"], h["w"], 1e-5),
            "layernorm": lambda h: oracle.layernorm(h["x"], h["w"], h["b"], 1e-5),
            "cross_entropy": lambda h: oracle.cross_entropy(h["x"], h["labels"]),
            "add_rmsnorm": lambda h: oracle.add_rmsnorm(h["x"], h["r"], h["w"], 1e-5),
            "add_layernorm": lambda h: oracle.add_layernorm(h["x"], h["r"], h["w"], h["b"], 1e-5),
            "row_sum": lambda h: oracle.row_sum(h["x"]), "row_max": lambda h: oracle.row_max(h["x"]),
            "row_min": lambda h: oracle.row_min(h["x"]),
            "row_minmax": lambda h: (oracle.row_min(h["x"]), oracle.row_max(h["x"])),
            "softmax_bwd": lambda h: oracle.softmax_backward(h["y"], h["dy"]),
            "cross_entropy_bwd": lambda h: oracle.cross_entropy_backward(h["x"], h["labels"], h["dloss"]),
            "rmsnorm_bwd": lambda h: oracle.rmsnorm_backward(h["x"], h["w"], h["dy"], 1e-5),
            "layernorm_bwd": lambda h: oracle.layernorm_backward(h["x"], h["w"], h["dy"], 1e-5),
            "axis_sum": lambda h: oracle.axis_sum(h["x"], 0),
            "axis_minmax": lambda h: (oracle.axis_min(h["x"], 0), oracle.axis_max(h["x"], 0))}[op]


def host_sample(op, workload, rows):
    w = synth.WORKLOADS[workload]
    d = synth.make_inputs(op, min(rows, w["rows"]), w["cols"], w["seed"], var=w.get("var"),
                          row_offset=w.get("row_offset", False))
    h = {k: v.numpy() for k, v in d.items()}
    if op == "softmax_bwd":
        import oracle
        h = {"y": oracle.ot_softmax(h["x"]), "dy": h["dy"]}
    return h


def sample_shape(h):
    """(rows, cols) of a host sample (the softmax backward's matrix is y)."""
    return (h["x"] if "x" in h else h["y"]).shape


ROW_KEYS = ("x", "y", "dy", "labels", "dloss", "r")  # per-row inputs; the rest are column vectors


def cpu_info():
    """Host core count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform
    return {"cpu_count": os.cpu_count() or 1, "cpu_model": model or platform.machine()}


def row_chunks(h, n):
    """Split a host sample into n contiguous row ranges (column vectors shared)."""
    rows = sample_shape(h)[0]
    bounds = [rows * i // n for i in range(n + 1)]
    return [{k: (v[a:b] if k in ROW_KEYS else v) for k, v in h.items()}
            for a, b in zip(bounds, bounds[1:]) if b > a]


def time_oracle(specs, rows_per_launch, budget_s=None, repeats=1, threads=1):
    """Run the oracle over `rows_per_launch` rows of every launch of the step,
    row-parallel on `threads` host threads (the C oracle runs with the
    interpreter lock released, one contiguous row range per thread)."""
    samples = [(oracle_fn(op, o), host_sample(op, w, rows_per_launch), op, w) for op, w, o in specs]
    pool = None
    if threads > 1:
        import concurrent.futures as cf
        pool = cf.ThreadPoolExecutor(max_workers=threads)
        samples = [(fn, h, op, w, row_chunks(h, threads)) for fn, h, op, w in samples]
    done_bytes, t_total, reps = 0, 0.0, 0
    try:
        while True:
            t0 = time.perf_counter()
            for smp in samples:
                if pool is None:
                    smp[0](smp[1])
                else:
                    list(pool.map(smp[0], smp[4]))
            t_total += time.perf_counter() - t0
            reps += 1
            done_bytes += sum(alg_bytes(smp[2], *sample_shape(smp[1])) for smp in samples)
            if budget_s is None and reps >= repeats:
                break
            if budget_s is not None and t_total >= budget_s:
                break
    finally:
        if pool is not None:
            pool.shutdown()
    return done_bytes, t_total, reps


def cpu_baseline(launches, args):
    specs = [(ln.op, ln.workload, ln.order) for ln in launches]
    rows = min(ln.rows for ln in launches)
    info = cpu_info()
    cores = info["cpu_count"]
    serial_rows = min(rows, args.cpu_rows)
    b1, t1, r1 = time_oracle(specs, serial_rows, budget_s=args.cpu_seconds / 2)
    par_rows = rows
    bp, tp, rp = time_oracle(specs, par_rows, budget_s=args.cpu_seconds / 2, threads=cores)
    return {"value": round(bp / tp / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": info["cpu_model"],
            "sample": f"{par_rows} rows of each of the {len(specs)} launches' inputs, row-parallel on {cores} "
                      f"threads, {rp} passes, {tp:.1f} s (serial FP64 C oracle / OT-1024 C emulation per row range)",
            "serial": {"value": round(b1 / t1 / 1e9, 4), "cores": 1,
                       "sample": f"{serial_rows} rows of each launch's inputs, {r1} passes, {t1:.1f} s, one thread"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    specs = WORKLOADS[args.workload]
    info = cpu_info()
    cores = info["cpu_count"]
    # size each step so the whole --warmup + --steps run stays within ~2 minutes
    b1, t1, _ = time_oracle(specs, 1, repeats=1)
    per_row = max(t1, 1e-5) / max(1, min(cores, 8))
    rows = int(max(1, min(768, 120.0 / (args.steps + args.warmup) / per_row)))
    samples = [(oracle_fn(op, o), host_sample(op, w, rows), op) for op, w, o in specs]
    import concurrent.futures as cf
    chunks = [(fn, row_chunks(h, cores)) for fn, h, _ in samples]
    step_bytes = sum(alg_bytes(op, *sample_shape(h)) for _, h, op in samples)
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        def step():
            for fn, ch in chunks:
                list(pool.map(fn, ch))
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        dt = time.perf_counter() - t0
    value = args.steps * step_bytes / dt / 1e9
    sample = (f"{rows} rows of each of the {len(specs)} launches' inputs per step, row-parallel on {cores} threads "
              f"(serial C oracle per row range)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config({"name": args.workload, "launches": specs}),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu_model": info["cpu_model"], "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_suite(args):
    """One line per workload: µs/op (median of 9 graphs of 200 back-to-back
    launches), GB/s, single-call latency and plan."""
    import fp32_row_reduction_gb300 as tr
    tr.load()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    names = [n for n in WORKLOADS if n != DEFAULT_WORKLOAD] if args.workload == DEFAULT_WORKLOAD \
        else [args.workload]
    for name in names:
        specs = WORKLOADS[name]
        op, w, order = specs[0]
        b = alg_bytes(op, synth.WORKLOADS[w]["rows"], synth.WORKLOADS[w]["cols"])
        sets = pick_sets([b])
        ln = Launch(op, w, order, sets, dev)
        for i in range(args.warmup):
            ln(i % sets)
        torch.cuda.synchronize()
        us, samples = timed_graph_us(ln, sets)
        e = op_entry(ln, us, samples, peak, single_call_us(ln, sets, reps=10))
        print(json.dumps(dict(workload=name, op=op, order=order, rows=ln.rows, cols=ln.cols, us_per_op=e["us"],
                              gbs=e["gbs"], frac_of_peak=e["frac_of_peak"], frac_of_8tbs=e["frac_of_8tbs"],
                              single_call_gpu_us=e["single_call_gpu_us"], single_call_e2e_us=e["single_call_e2e_us"],
                              alg_bytes=b, l2=f"{sets} rotating buffer sets", plan=e["plan"])), flush=True)
        del ln
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--unroll", type=int, default=100, help="steps per captured graph")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-rows", type=int, default=96)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--suite", action="store_true", help="one line per workload, then exit")
    ap.add_argument("--no-per-op", action="store_true", help="report only the step's kernels in per_op")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        if args.suite:
            run_suite(args)
            return
        line = run_ours(args, rank, world)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
