#!/usr/bin/env python
"""Benchmark of the FP8 mixed-granularity linear-layer hot path on GB300.

One step = the forward and backward of the four Llama-3.1-8B layer linears at
M = 8192 training tokens (QKV 4096→6144, O 4096→4096, gate/up 4096→28672,
down 14336→4096) through the jetfp8 C ABI:
  RMSNorm+1×128 quant (QKV and gate/up inputs) or 1×128 quant (O and down),
  128×128 weight quant with the transposed payload, FProp, dual gradient
  quant, DGrad, 1×128→128×1 requantise-transpose, WGrad.
Inputs are seeded synthetic bf16 tensors with the distributions of the Jet-RL
workloads; together they exceed the 129 MB L2 many times over, so no L2 flush
is needed between steps.

metric  FP8 block-scaled GEMM TFLOP/s: the step's GEMM FLOPs (3 × 2·M·N·K per
        linear) divided by the whole step's time (quantisers included), summed
        over ranks.
Also reported: each kernel family's own TFLOP/s or GB/s (the median of every
launch over the timed steps, from CUDA events on the launching stream), the
roofline of the dominant kernel, the CPU oracle on a bounded sample, the same
metric end to end from pinned host memory, and, after the headline step, the
other workloads: Qwen3-8B decode FProp at 64/128/256 tokens (CUDA-graph replay,
fraction of HBM), the 32B-class layer step at 16384 tokens with the weight
requantisation after an update, and the gated-MLP block chain at 16384 tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same single-GPU step on its own
GPU (replicas: the path needs no collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 block-scaled GEMM TFLOP/s (% dense-FP8 peak); quant kernels GB/s (% HBM)"
WORKLOAD = "llama3.1-8b-training-linears"
REF_ROWS, REF_COLS = 128, 1024       # CPU sample: 128 tokens × 1024 output features per linear
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one gate/up FProp launch
# (8192 x 28672 x 4096) from a single-pass ncu capture, and the SHA-256 (first 16 hex
# digits) of the GEMM sources it was captured on.  When the sources differ from that
# digest the figure no longer describes the kernel and `traffic` is reported as null.
GATEUP_FPROP_DRAM_BYTES = 607120896
GATEUP_FPROP_DRAM_SRC = "fef81d3071166beb"
GEMM_SOURCES = ("gemm_tcgen05.cu", "jetfp8_common.cuh", "jetfp8_internal.h")

# algorithmic bytes per element of each quantiser (inputs read + outputs written)
QUANT_BYTES = {
    "quant_act": 2 + 1 + 4 / 128,
    "rmsnorm_quant": 2 + 1 + 4 / 128,
    "quant_weight": 2 + 1 + 1 + 4 / 16384,
    "quant_grad_dual": 2 + 2 * (1 + 4 / 128),
    "requant": 1 + 4 / 128 + 1 + 4 / 128,
    # per element of h [M, I]: gate and up read (2 + 2 B), codes and scales written
    "swiglu_quant": 2 + 2 + 1 + 4 / 128,
    # per element of ∇h [M, I]: gate, up and ∇h read, ∇gate and ∇up written
    "swiglu_bwd": 5 * 2,
    # per element: x and ∇y read, ∇x written (γ, r and ∇γ are per row or column)
    "rmsnorm_bwd": 3 * 2,
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the decode, 32B-class and MLP-chain workloads after the headline step")
    p.add_argument("--case", choices=sorted(CASES), default=None,
                   help="time one kernel alone (for profiling) instead of the layer step")
    p.add_argument("--shape", default="8192,28672,4096", help="M,N,K for --case")
    p.add_argument("--gemm-path", type=int, choices=[0, 1, 2], default=0,
                   help="with --case: GEMM kernel choice (0 automatic, 1 single-CTA tiles, 2 CTA-pair "
                        "tiles where the shape allows)")
    p.add_argument("--graph", action="store_true",
                   help="with --case: capture the timed launches in a CUDA graph and time its replay "
                        "(kernel time without the per-call host work, as a serving loop runs decode)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank contributes its own time and all
    receive the maximum (a no-op for one rank).  `device` is where the
    collective runs (the rank's GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, ms: float, scale: float = 1e12) -> float:
    """Whole-job throughput: the units all replicas processed in the slowest
    rank's time (weak scaling: every rank runs the same workload)."""
    return units_per_rank * world / (ms * 1e-3) / scale


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle reasons;
    only samples taken inside the timed window are summarised."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t_begin: float, t_end: float):
        self.window = (t_begin, t_end)

    @staticmethod
    def _epoch(ts: str):
        try:
            return time.mktime(time.strptime(ts.strip().split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                float("0." + ts.strip().split(".")[1]) if "." in ts else 0.0
        except (ValueError, IndexError):
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = rows
        if self.window is not None:
            t0, t1 = self.window
            stamped = [(self._epoch(r[0]), r) for r in rows]
            inside = [r for t, r in stamped if t is not None and t0 <= t <= t1]
            if not inside:   # timed window shorter than the sampling interval: nearest sample
                mid = 0.5 * (t0 + t1)
                inside = [min(((abs(t - mid), r) for t, r in stamped if t is not None),
                              key=lambda x: x[0], default=(0, rows[-1]))[1]]
        sm = [float(r[1]) for r in inside]
        smax = max(float(r[2]) for r in inside)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(inside), "power_w_max": max(float(r[3]) for r in inside)}


# ---------------------------------------------------------------------------
# CPU oracle sample (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_sample_step(lins, seed=0):
    """The whole path for a 128-token × 1024-output-feature slice of every
    linear, on the CPU oracle.  Returns the GEMM FLOPs it performed."""
    from fp8_mixed_granularity_gb300 import workloads as W
    from oracle import jetfp8_oracle as O
    flops = 0
    for i, lin in enumerate(lins):
        m, n, k = REF_ROWS, min(REF_COLS, lin.N), lin.K
        x = W.bf16_values(W.activations(m, k, seed=seed, stream=10 + i))
        w = W.bf16_values(W.weights(n, k, seed=seed, stream=20 + i))
        dy = W.bf16_values(W.gradients(m, n, seed=seed, stream=30 + i))
        xq, sx = O.quant_act_1x128(x)
        wq, sw, wqT = O.quant_weight_128x128(w)
        O.gemm_fprop(xq, sx, wq, sw)
        dq, ds, dqT, dsT = O.quant_grad_dual(dy)
        O.gemm_dgrad(dq, ds, wqT, sw)
        xqT, sxT = O.requant_rowgrp_to_colgrp(xq, sx)
        O.gemm_wgrad(dqT, dsT, xqT, sxT)
        flops += 3 * 2 * m * n * k
    return flops


def blas_threads():
    """Threads the oracle's BLAS calls may use (the numpy matmuls): from
    threadpoolctl where it is installed, else from the thread-count variables
    the BLAS libraries read, else their default of one thread per usable core."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "").strip()
        if v.isdigit() and int(v) > 0:
            return int(v)
    return host_cores()


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count()


def time_oracle(lins, steps):
    t0 = time.perf_counter()
    flops = 0
    for s in range(steps):
        flops += oracle_sample_step(lins, seed=s)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, flops


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, timed as it stands
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from fp8_mixed_granularity_gb300 import workloads as W
    lins = W.llama8b_training()
    for s in range(args.warmup):
        oracle_sample_step(lins, seed=1000 + s)
    value, dt, flops = time_oracle(lins, args.steps)
    sample = (f"per step: the full path (quantisers + FProp/DGrad/WGrad) for {REF_ROWS} tokens × "
              f"{REF_COLS} output features of each of the 4 linears")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": 8192, "linears": [l.name for l in lins],
                   "l2": "inputs larger than L2"},
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": "TFLOP/s", "cores": host_cores(),
                         "blas_threads": blas_threads(), "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def gemm_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "fp8_mixed_granularity_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def launch_medians(events_per_step):
    """{(linear, kind): median launch ms} over the timed steps.  Each step's
    launches are a list of (linear, kind, ms)."""
    per = {}
    for evs in events_per_step:
        for lname, kind, ms in evs:
            per.setdefault((lname, kind), []).append(ms)
    return {k: float(np.median(v)) for k, v in per.items()}, {k: len(v) for k, v in per.items()}


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__ as g
    if rank == 0:
        g.build()
    if world > 1:
        torch.distributed.barrier()
    g.build()
    from fp8_mixed_granularity_gb300 import jetfp8 as J
    from fp8_mixed_granularity_gb300 import workloads as W
    from fp8_mixed_granularity_gb300.linear import EventLog, LinearBuffers, quant_weights_grouped

    lins = W.llama8b_training()
    norm_fed = {"qkv", "gate_up"}
    bufs, inputs = [], []
    for i, lin in enumerate(lins):
        b = LinearBuffers(lin, dev, rmsnorm=lin.name in norm_fed)
        x = W.device_activations(lin.M, lin.K, dev, seed=100 + i + 10 * rank)
        w = W.device_normal((lin.N, lin.K), 0.02, dev, seed=200 + i + 10 * rank)
        dy = W.device_normal((lin.M, lin.N), 1e-3, dev, seed=300 + i + 10 * rank)
        gamma = W.device_uniform((lin.K,), 0.5, 1.5, dev, seed=400 + i) if b.rmsnorm else None
        bufs.append(b)
        inputs.append((x, w, dy, gamma))
    gemm_flops = sum(3 * l.gemm_flops for l in lins)

    def step(events=None):
        # the four weights quantised in one grouped launch (149 vs 171 µs for
        # four launches, graph-timed), then forward and backward of each linear,
        # its WGrad as a launch of its own (four single WGrads measure faster
        # than the grouped launch of the four: 1.97 vs 2.10 ms).  With `events`
        # (a list), every launch is bracketed by CUDA events on its stream.
        ev = None if events is None else type(events)()
        n = quant_weights_grouped(bufs, [inp[1] for inp in inputs], events=ev)
        if events is not None:
            events.extend((GROUPED, kind, s, e) for kind, s, e in ev)
        for b, (x, w, dy, gamma) in zip(bufs, inputs):
            ev = None if events is None else type(events)()
            n += b.forward(x, None, gamma, events=ev)
            n += b.backward(dy, events=ev)
            if events is not None:
                events.extend((b.lin.name, kind, s, e) for kind, s, e in ev)
        return n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    J.jetfp8_get_last_device_error()
    # the step captured once as a CUDA graph (every launch of the step, none
    # skipped), replayed in the headline's timed region as a training loop in
    # steady state would; the eager steps that follow give the per-launch times
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            per_step = step()
    torch.cuda.current_stream().wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    J.jetfp8_get_last_device_error()

    # --- timed region: K graph replays of the whole step, CUDA events on the stream ---
    sampler = ClockSampler(local)
    events_per_step = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    host_t0 = time.time()
    t0.record()
    for _ in range(args.steps):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    host_t1 = time.time()
    launches = per_step * args.steps
    # --- then the breakdown: the step captured again with a CUDA event-record
    # node around every launch, replayed K times (each replay's times read before
    # the next); where this torch cannot put events in a graph, K eager steps
    # with CUDA events around every launch ---
    breakdown_how = "graph"
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        breakdown_how = "eager"
    if breakdown_how == "graph":
        graph_ev = torch.cuda.CUDAGraph()
        captured = EventLog()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph_ev, stream=cap):
                step(captured)
        torch.cuda.current_stream().wait_stream(cap)
        graph_ev.replay()
        torch.cuda.synchronize()
        for _ in range(args.steps):
            graph_ev.replay()
            torch.cuda.synchronize()
            events_per_step.append([(ln, kind, s.elapsed_time(e)) for ln, kind, s, e in captured])
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    eager_events = []
    for _ in range(args.steps):
        ev = []
        step(ev)
        eager_events.append(ev)
    e1.record()
    torch.cuda.synchronize()
    if breakdown_how == "eager":
        events_per_step = [[(ln, kind, s.elapsed_time(e)) for ln, kind, s, e in ev] for ev in eager_events]
    sampler.mark(host_t0, time.time())
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    J.jetfp8_get_last_device_error()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    eager_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    # --- per-launch medians over the timed steps ---
    med, counts = launch_medians(events_per_step)
    by_name = {l.name: l for l in lins}
    gemm_kinds = ("gemm_fprop", "gemm_dgrad", "gemm_wgrad")
    gemm_ms = {k: sum(v for (ln, kk), v in med.items() if kk == k) for k in gemm_kinds}
    gemm_total_ms = sum(gemm_ms.values())
    layer_flops = sum(l.gemm_flops for l in lins)
    peaks = measured_peaks()
    # dense FP8 = 2 × bf16 (the nominal 4.5/2.25 ratio); the burst figure, because
    # each launch runs inside a timed region of well under a second at full clocks
    fp8_peak = 2.0 * peaks["bf16"]
    quant = {}
    for kind in QUANT_KINDS:
        # a grouped launch (recorded under GROUPED) covers every linear of the step
        parts = [(ln, v) for (ln, kk), v in med.items() if kk in (kind, kind + "_grouped")]
        if not parts:
            continue
        nb = lambda ln: sum(quant_bytes(kind, l) for l in (lins if ln == GROUPED else [by_name[ln]]))  # noqa: E731
        nbytes = sum(nb(ln) for ln, _ in parts)
        qms = sum(v for _, v in parts)
        gbs = nbytes / (qms * 1e-3) / 1e9
        quant[kind] = {"gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "ms_per_step": qms,
                       "launches_timed": sum(counts[k] for k in counts if k[0] in dict(parts)
                                             and k[1] in (kind, kind + "_grouped")),
                       "per_linear_gbs": {ln: nb(ln) / (v * 1e-3) / 1e9 for ln, v in parts}}
    # the dominant single launch: the gate/up FProp
    dom = by_name["gate_up"]
    dom_ms = med[("gate_up", "gemm_fprop")]
    dom_tflops = dom.gemm_flops / (dom_ms * 1e-3) / 1e12
    gemm_tflops = gemm_flops / (gemm_total_ms * 1e-3) / 1e12
    value = job_value(gemm_flops, world, ms)
    same_src = gemm_sources_digest() == GATEUP_FPROP_DRAM_SRC

    # --- end to end from pinned host memory ---
    e2e = None if args.no_e2e else run_e2e(bufs, inputs, args, torch, gemm_flops, world)
    del bufs, inputs
    torch.cuda.empty_cache()

    # --- the other workloads (parity cases of their own; timed here, outside the headline) ---
    configs = {} if args.no_configs else run_configs(args, torch, J, W, dev, peaks)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": 8192, "linears": {l.name: [l.K, l.N] for l in lins},
                   "step": ("fwd+bwd of the 4 linears incl. all quantisers (one grouped launch for the four "
                            "weights, one WGrad launch per linear), captured once as a CUDA graph and replayed"),
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (no flush)"},
        "roofline": {
            "kernel": f"k_gemm_e4m3_blockscaled gate/up FProp {dom.M}x{dom.N}x{dom.K}",
            "bound": "tensor", "achieved": dom_tflops,
            "peak": fp8_peak, "unit": "TFLOP/s", "frac": dom_tflops / fp8_peak,
            "traffic": GATEUP_FPROP_DRAM_BYTES if same_src else None,
            "traffic_note": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one such launch"
                             if same_src else "null: the GEMM sources changed since the DRAM capture"),
            "algorithmic_flops": dom.gemm_flops, "launch_ms": dom_ms,
            "peak_note": (f"2 x {peaks['source']} burst bf16 cuBLAS ({peaks['bf16']} TFLOP/s), of {peaks['source']}"),
            "all_gemm_launches": {"achieved": gemm_tflops, "frac": gemm_tflops / fp8_peak},
        },
        "breakdown": {
            "timing": ("median of each launch over K replays of the step captured as a CUDA graph with an "
                       "event-record node around every launch" if breakdown_how == "graph" else
                       "median of each launch over K eager steps (CUDA events on the launching stream "
                       "around every launch)"),
            "eager_ms_per_step": eager_ms,
            "gemm_tflops": {k: layer_flops / (v * 1e-3) / 1e12 for k, v in gemm_ms.items()},
            "gemm_frac": {k: layer_flops / (v * 1e-3) / 1e12 / fp8_peak for k, v in gemm_ms.items()},
            "gemm_ms_per_step": gemm_total_ms,
            "quant": quant,
            "hbm_peak_gbs": peaks["hbm_gbs"],
            "configs": configs,
        },
        "clocks": clocks,
        "gpu_launches": launches,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cv, cdt, cfl = time_oracle(lins, 5)
        line["cpu_baseline"] = {
            "value": cv, "unit": "TFLOP/s", "cores": host_cores(), "blas_threads": blas_threads(),
            "kind": "oracle",
            "sample": (f"5 steps of the full path on {REF_ROWS} tokens × {REF_COLS} output features of "
                       f"each of the 4 linears ({cfl / 1e9:.1f} GFLOP in {cdt:.1f} s)")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


QUANT_KINDS = ("rmsnorm_quant", "quant_act", "quant_weight", "quant_grad_dual", "requant")
GROUPED = "all_four"   # the name under which a launch for all four linears is recorded


def quant_bytes(kind, lin):
    """Algorithmic bytes of one quantiser launch of linear `lin`."""
    M, K, N = lin.M, lin.K, lin.N
    if kind == "rmsnorm_quant":
        return M * K * QUANT_BYTES[kind] + 2 * K + 4 * M
    if kind == "quant_act":
        return M * K * QUANT_BYTES[kind]
    if kind == "quant_weight":
        return N * K * QUANT_BYTES[kind]
    if kind == "quant_grad_dual":
        return M * N * QUANT_BYTES[kind]
    if kind == "requant":
        return M * K * QUANT_BYTES[kind]
    raise KeyError(kind)


# ---------------------------------------------------------------------------
# the other workloads, timed after the headline step
# ---------------------------------------------------------------------------
def _graph_ms(torch, fn, reps=5):
    """Median ms of one replay of a CUDA graph holding fn()'s launches."""
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        graph.replay()
        e.record()
        torch.cuda.synchronize()
        out.append(s.elapsed_time(e))
    return float(np.median(out))


def _events_ms(torch, fn, steps, warmup=3):
    """Median ms of fn() (a step of many launches), CUDA events per step."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        evs.append((s, e))
    torch.cuda.synchronize()
    return float(np.median([s.elapsed_time(e) for s, e in evs]))


def decode_config(torch, J, W, dev, peaks, layers=4):
    """Qwen3-8B decode FProp at M ∈ {64, 128, 256}: the four linears of `layers`
    distinct layers (their weights together exceed L2, as in a model's forward),
    replayed from a CUDA graph as a serving loop would.  HBM bytes per FProp =
    X̂ + Ŵ + both scale sets + bf16 Y."""
    out = {}
    shapes = W.qwen3_8b_decode(1)
    wsets = []
    for l in range(layers):
        ws = []
        for i, lin in enumerate(shapes):
            w = W.device_normal((lin.N, lin.K), 0.02, dev, seed=900 + 10 * l + i)
            wq = torch.empty(lin.N, lin.K, dtype=torch.uint8, device=dev)
            sw = torch.empty(lin.N // 128, lin.K // 128, dtype=torch.float32, device=dev)
            J.jetfp8_quant_weight_128x128(w, wq, sw)
            ws.append((wq, sw))
            del w
        wsets.append(ws)
    for M in (64, 128, 256):
        xs = []
        for i, lin in enumerate(shapes):
            x = W.device_channel_outlier_activations(M, lin.K, dev, seed=700 + i)
            xq, sx = J.empty_rowgroup_quant(M, lin.K, dev)
            J.jetfp8_quant_act_1x128(x, xq, sx)
            y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
            xs.append((xq, sx, y))

        def fwd():
            for ws in wsets:
                for (wq, sw), (xq, sx, y) in zip(ws, xs):
                    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
        ms = _graph_ms(torch, fwd) / layers
        flops = sum(2 * M * lin.N * lin.K for lin in shapes)
        nbytes = sum(M * lin.K + lin.N * lin.K + 4 * (lin.K // 128) * J.round_up4(M)
                     + 4 * (lin.N // 128) * (lin.K // 128) + 2 * M * lin.N for lin in shapes)
        gbs = nbytes / (ms * 1e-3) / 1e9
        # each linear alone (same graph method) for the narrow / wide split
        per = {}
        for i, lin in enumerate(shapes):
            def one(i=i):
                for ws in wsets:
                    wq, sw = ws[i]
                    xq, sx, y = xs[i]
                    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
            lms = _graph_ms(torch, one) / layers
            lb = M * lin.K + lin.N * lin.K + 4 * (lin.K // 128) * J.round_up4(M) \
                + 4 * (lin.N // 128) * (lin.K // 128) + 2 * M * lin.N
            per[lin.name] = {"us": lms * 1e3, "gbs": lb / (lms * 1e-3) / 1e9,
                             "frac_hbm": lb / (lms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        out[f"M{M}"] = {"ms_per_layer_fwd": ms, "tflops": flops / (ms * 1e-3) / 1e12, "gbs": gbs,
                        "frac_hbm": gbs / peaks["hbm_gbs"], "per_linear": per}
        del xs
    out["method"] = (f"CUDA-graph replay; {layers} layers' distinct weights per replay (> L2); "
                     "bytes = X̂ + Ŵ + scales + bf16 Y per FProp")
    return out


def b32_config(torch, J, W, dev, peaks, steps):
    """32B-class layer linears at M = 16384: forward + backward of the four
    linears (all quantisers, one WGrad launch per linear), and the 128×128 requantisation of
    all four weights after the update W += N(0, 1e-4)."""
    from fp8_mixed_granularity_gb300.linear import LinearBuffers, quant_weights_grouped
    lins = W.dense32b_training()
    bufs, inputs = [], []
    for i, lin in enumerate(lins):
        b = LinearBuffers(lin, dev)
        x = W.device_activations(lin.M, lin.K, dev, seed=500 + i)
        w = W.device_normal((lin.N, lin.K), 0.02, dev, seed=510 + i)
        dy = W.device_normal((lin.M, lin.N), 1e-3, dev, seed=520 + i)
        bufs.append(b)
        inputs.append((x, w, dy))

    def step():
        quant_weights_grouped(bufs, [inp[1] for inp in inputs])
        for b, (x, w, dy) in zip(bufs, inputs):
            b.forward(x, None)
            b.backward(dy)
    ms = _events_ms(torch, step, steps)
    flops = sum(3 * l.gemm_flops for l in lins)
    # weight update and requantisation (the update is setup, not timed)
    for i, (b, (x, w, dy)) in enumerate(zip(bufs, inputs)):
        w += W.device_normal(tuple(w.shape), 1e-4, dev, seed=530 + i)

    def requant_all():
        quant_weights_grouped(bufs, [inp[1] for inp in inputs])
    rq_ms = _events_ms(torch, requant_all, steps)
    n_w = sum(l.N * l.K for l in lins)
    rq_gbs = n_w * QUANT_BYTES["quant_weight"] / (rq_ms * 1e-3) / 1e9
    return {"tokens": 16384, "linears": {l.name: [l.K, l.N] for l in lins},
            "ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "weight_requant": {"elements": n_w, "ms": rq_ms, "gbs": rq_gbs,
                               "frac_hbm": rq_gbs / peaks["hbm_gbs"]}}


def mlp_config(torch, J, W, dev, peaks, steps, M=16384, H=4096, I=14336):
    """The gated-MLP block chain at M tokens: RMSNorm + 1×128 quant → gate/up
    FProp → SwiGLU + quant → down FProp, then the backward: dual gradient
    quant → down DGrad, requant of h → SwiGLU backward → dual quant → gate/up
    DGrad, requant of the norm output → RMSNorm backward, both WGrads; both
    weights quantised (with transposes) every step."""
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
    x = W.device_activations(M, H, dev, seed=600)
    gamma = W.device_uniform((H,), 0.5, 1.5, dev, seed=601)
    w_gu = W.device_normal((2 * I, H), 0.02, dev, seed=602)
    w_d = W.device_normal((H, I), 0.02, dev, seed=603)
    dy = W.device_normal((M, H), 1e-3, dev, seed=604)
    xq, sx = J.empty_rowgroup_quant(M, H, dev)
    rstd = e(M, dt=f32)
    wq_gu, sw_gu, wqT_gu = e(2 * I, H, dt=u8), e(2 * I // 128, H // 128, dt=f32), e(H, 2 * I, dt=u8)
    wq_d, sw_d, wqT_d = e(H, I, dt=u8), e(H // 128, I // 128, dt=f32), e(I, H, dt=u8)
    gu = e(M, 2 * I, dt=bf)
    hq, hs = J.empty_rowgroup_quant(M, I, dev)
    out = e(M, H, dt=bf)
    dyq, sdy = J.empty_rowgroup_quant(M, H, dev)
    dyqT, sdyT = J.empty_rowgroup_quant(H, M, dev)
    dh = e(M, I, dt=bf)
    hqT, hsT = J.empty_rowgroup_quant(I, M, dev)
    dw_d = e(H, I, dt=bf)
    dgu = e(M, 2 * I, dt=bf)
    dguq, sdgu = J.empty_rowgroup_quant(M, 2 * I, dev)
    dguqT, sdguT = J.empty_rowgroup_quant(2 * I, M, dev)
    dxn = e(M, H, dt=bf)
    xqT, sxT = J.empty_rowgroup_quant(H, M, dev)
    dw_gu = e(2 * I, H, dt=bf)
    dx = e(M, H, dt=bf)
    dgamma = e(H, dt=f32)
    ws = e(J.jetfp8_rmsnorm_bwd_workspace_bytes(M, H), dt=u8)

    def step():
        J.jetfp8_quant_weight_grouped([(w_gu, wq_gu, sw_gu, wqT_gu), (w_d, wq_d, sw_d, wqT_d)])
        J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, xq, sx, rstd)
        J.jetfp8_gemm_fprop(xq, sx, wq_gu, sw_gu, gu)
        J.jetfp8_swiglu_quant(gu, hq, hs)
        J.jetfp8_gemm_fprop(hq, hs, wq_d, sw_d, out)
        J.jetfp8_quant_grad_dual(dy, dyq, sdy, dyqT, sdyT)
        J.jetfp8_gemm_dgrad(dyq, sdy, wqT_d, sw_d, dh)
        J.jetfp8_requant_rowgrp_to_colgrp(hq, hs, hqT, hsT)
        J.jetfp8_swiglu_bwd(gu, dh, dgu)
        J.jetfp8_quant_grad_dual(dgu, dguq, sdgu, dguqT, sdguT)
        J.jetfp8_gemm_dgrad(dguq, sdgu, wqT_gu, sw_gu, dxn)
        J.jetfp8_requant_rowgrp_to_colgrp(xq, sx, xqT, sxT)
        J.jetfp8_rmsnorm_bwd(x, gamma, rstd, dxn, dx, dgamma, ws)
        J.jetfp8_gemm_wgrad(dyqT, sdyT, hqT, hsT, dw_d)
        J.jetfp8_gemm_wgrad(dguqT, sdguT, xqT, sxT, dw_gu)
    ms = _events_ms(torch, step, steps)
    flops = 3 * 2 * M * (2 * I * H + H * I)
    return {"tokens": M, "hidden": H, "intermediate": I, "ms_per_step": ms,
            "tflops": flops / (ms * 1e-3) / 1e12, "launches_per_step": 15}


def nvfp4_config(torch, J, W, dev, peaks, steps, M=8192):
    """The FP4 variant of the flow on the Llama-3.1-8B forward linears at M
    tokens: the row quantiser of the activation and the block-scaled FProp of
    each linear (weights quantised once, outside the timed launches), against
    the FP4 dense peak taken as the measured bf16 burst figure times the
    nominal FP4/BF16 ratio (13.5 / 2.25 = 6)."""
    peak = 6.0 * peaks["bf16"]
    res = {"peak_tflops": peak, "peak_note": f"6 x {peaks['source']} burst bf16 (nominal FP4/BF16 ratio), of {peaks['source']}"}
    lins = {"qkv": (4096, 6144), "o": (4096, 4096), "gate_up": (4096, 28672), "down": (14336, 4096)}
    per = {}
    total_ms, total_flops = 0.0, 0.0
    for name, (K, N) in lins.items():
        x = W.device_activations(M, K, dev, seed=700)
        w = W.device_normal((N, K), 0.02, dev, seed=701)
        xq, xsf, gx = J.empty_nvfp4(M, K, dev)
        wq, wsf, gw = J.empty_nvfp4(N, K, dev)
        J.jetfp8_quant_nvfp4(w, wq, wsf, gw)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        qms = _events_ms(torch, lambda: J.jetfp8_quant_nvfp4(x, xq, xsf, gx), steps)
        gms = _events_ms(torch, lambda: J.jetfp8_gemm_fprop_nvfp4(xq, xsf, gx, wq, wsf, gw, y), steps)
        f = 2.0 * M * N * K
        qbytes = M * K * (2 + 0.5 + 1 / 16) + 4 * M
        per[name] = {"fprop_us": gms * 1e3, "fprop_tflops": f / (gms * 1e-3) / 1e12,
                     "fprop_frac": f / (gms * 1e-3) / 1e12 / peak, "quant_us": qms * 1e3,
                     "quant_gbs": qbytes / (qms * 1e-3) / 1e9}
        total_ms += gms
        total_flops += f
        del x, w, xq, xsf, gx, wq, wsf, gw, y
    res["per_linear"] = per
    res["fprop_tflops_all"] = total_flops / (total_ms * 1e-3) / 1e12
    res["tokens"] = M
    return res


def run_configs(args, torch, J, W, dev, peaks):
    steps = max(5, min(args.steps, 10))
    out = {"decode_qwen3_8b": decode_config(torch, J, W, dev, peaks)}
    torch.cuda.empty_cache()
    out["dense32b_training"] = b32_config(torch, J, W, dev, peaks, steps)
    torch.cuda.empty_cache()
    out["gated_mlp_chain"] = mlp_config(torch, J, W, dev, peaks, steps)
    torch.cuda.empty_cache()
    out["nvfp4_variant_fprop"] = nvfp4_config(torch, J, W, dev, peaks, steps)
    torch.cuda.empty_cache()
    J.jetfp8_get_last_device_error()
    return out


def run_e2e(bufs, inputs, args, torch, gemm_flops, world):
    """Same metric through the public API with host buffers: every step copies
    its bf16 inputs (x, W, ∇Y and γ of each linear) from pinned host memory to
    the device and reads Y, ∇X and ∇W back, all inside the timed region.  Copies
    in, compute and copies out run on three streams.  The device inputs are
    double-buffered (step k uses set k mod 2), so a step's copies in never wait
    for the previous step's compute; each step copies its four weights first
    (the grouped weight quantiser needs all four) and then each linear's x, ∇Y
    and γ, and each linear's results leave while the next linear computes.
    Events keep every buffer's uses in order (a set is refilled once the compute
    two steps back has read it; a linear's compute waits until the previous read-
    back of its outputs is done)."""
    from fp8_mixed_granularity_gb300.linear import quant_weights_grouped
    host_in = [tuple(None if t is None else t.cpu().pin_memory() for t in inp) for inp in inputs]
    host_out = [tuple(torch.empty_like(b.t[k], device="cpu").pin_memory() for k in ("y", "dx", "dw"))
                for b in bufs]
    dev_in = [inputs, [tuple(None if t is None else torch.empty_like(t) for t in inp) for inp in inputs]]
    h2d = sum(t.numel() * t.element_size() for inp in host_in for t in inp if t is not None)
    d2h = sum(t.numel() * t.element_size() for outs in host_out for t in outs)
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n = len(bufs)
    ev = lambda: [torch.cuda.Event() for _ in range(n)]  # noqa: E731
    in_ready = [ev(), ev()]
    w_ready = [torch.cuda.Event(), torch.cuda.Event()]
    set_free = [torch.cuda.Event(), torch.cuda.Event()]
    out_ready, out_free = ev(), ev()
    count = [0]

    def step():
        k = count[0]
        p = k % 2
        dset = dev_in[p]
        if k >= 2:
            s_in.wait_event(set_free[p])   # step k-2's compute has read this set
        with torch.cuda.stream(s_in):
            for hi, di in zip(host_in, dset):
                di[1].copy_(hi[1], non_blocking=True)
            w_ready[p].record(s_in)
            for i, (hi, di) in enumerate(zip(host_in, dset)):
                for j, (hsrc, ddst) in enumerate(zip(hi, di)):
                    if hsrc is not None and j != 1:
                        ddst.copy_(hsrc, non_blocking=True)
                in_ready[p][i].record(s_in)
        s_comp.wait_event(w_ready[p])
        quant_weights_grouped(bufs, [di[1] for di in dset], stream=s_comp)
        for i, (b, di, ho) in enumerate(zip(bufs, dset, host_out)):
            s_comp.wait_event(in_ready[p][i])
            if k >= 1:
                s_comp.wait_event(out_free[i])
            x, w, dy, gamma = di
            b.forward(x, None, gamma, stream=s_comp)
            b.backward(dy, stream=s_comp)
            out_ready[i].record(s_comp)
            s_out.wait_event(out_ready[i])
            with torch.cuda.stream(s_out):
                for kk, hdst in zip(("y", "dx", "dw"), ho):
                    hdst.copy_(b.t[kk], non_blocking=True)
            out_free[i].record(s_out)
        set_free[p].record(s_comp)
        count[0] += 1

    cur = torch.cuda.current_stream()
    for s_ in (s_in, s_comp, s_out):
        s_.wait_stream(cur)
    step()
    torch.cuda.synchronize()
    steps = max(2, args.steps // 2)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for s_ in (s_in, s_comp, s_out):
        s_.wait_stream(cur)
    for _ in range(steps):
        step()
    for s_ in (s_in, s_comp, s_out):
        cur.wait_stream(s_)
    t1.record(cur)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, world, bufs[0].device)
    return {"value": job_value(gemm_flops, world, ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "overlap": ("copies in, compute and copies out on three streams; device inputs double-buffered "
                        "across steps, results read back per linear")}


# ---------------------------------------------------------------------------
# single-kernel cases (profiling aid): one kernel, one shape, W + K launches
# ---------------------------------------------------------------------------
CASES = {"fprop", "dgrad", "wgrad", "quant_act", "rmsnorm_quant", "quant_weight",
         "quant_grad_dual", "requant", "swiglu_quant", "swiglu_bwd", "fprop_quant", "fprop_then_quant",
         "rmsnorm_bwd", "decoder_layer", "wgrad_grouped", "wgrad_separate", "fp8_library_probe",
         "fprop_nvfp4", "quant_nvfp4", "quant_weight_grouped"}


def run_case(args):
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__ as g
    g.build()
    from fp8_mixed_granularity_gb300 import jetfp8 as J
    from fp8_mixed_granularity_gb300 import workloads as W
    from fp8_mixed_granularity_gb300.linear import LinearBuffers
    M, N, K = (int(v) for v in args.shape.split(","))
    J.jetfp8_test_set_gemm_path(args.gemm_path)
    if args.case == "decoder_layer":
        # a Llama-3.1-8B-shaped decoder layer (BF16 attention core), forward +
        # backward, on M tokens = M/1024 sequences of 1024; the rate counts the
        # four linear layers' GEMM FLOPs (6·M·N·K each) over the whole layer time
        from fp8_mixed_granularity_gb300.decoder_layer import DecoderLayerFP8, llama8b
        shape = llama8b()
        S = 1024
        Bq = max(1, M // S)
        T = Bq * S
        D, I = shape.hidden, shape.intermediate
        w = {"wqkv": W.device_normal((shape.qkv_width, D), 0.02, dev, seed=11),
             "wo": W.device_normal((D, shape.attn_width), 0.02, dev, seed=12),
             "wgu": W.device_normal((2 * I, D), 0.02, dev, seed=13),
             "wd": W.device_normal((D, I), 0.02, dev, seed=14),
             "gamma1": W.device_uniform((D,), 0.5, 1.5, dev, seed=15),
             "gamma2": W.device_uniform((D,), 0.5, 1.5, dev, seed=16)}
        x = W.device_activations(T, D, dev, seed=17)
        dy = W.device_normal((T, D), 1e-3, dev, seed=18)
        layer = DecoderLayerFP8(shape, w, dev)

        def fwd_bwd():
            layer.forward(x, Bq, S)
            layer.backward(dy)
        flops = sum(6 * m * n * k for _, m, n, k in shape.linears(T))
        _time_case(args, fwd_bwd, flops, "TFLOP/s", [T, D, D])
        return
    if args.case == "fp8_library_probe":
        # context for the roofline only (not this library's path): the PyTorch /
        # cuBLASLt dense E4M3 GEMM with per-tensor scales on M x N x K, bf16 out
        a8 = (torch.randn(M, K, device=dev) * 0.5).to(torch.float8_e4m3fn)
        b8 = (torch.randn(N, K, device=dev) * 0.5).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        fn = lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)  # noqa: E731
        _time_case(args, fn, 2 * M * N * K, "TFLOP/s", [M, N, K])
        return
    if args.case in ("wgrad_grouped", "wgrad_separate"):
        # the WGrads of a Llama-3.1-8B layer's four linears on M tokens: one
        # grouped launch, or four launches one after another
        from fp8_mixed_granularity_gb300.linear import wgrad_grouped
        lins = W.llama8b_training(M)
        bufs = []
        for i, lin in enumerate(lins):
            b = LinearBuffers(lin, dev)
            b.forward(W.device_activations(M, lin.K, dev, seed=1 + i), W.device_normal((lin.N, lin.K), 0.02, dev, seed=5 + i))
            b.backward(W.device_normal((M, lin.N), 1e-3, dev, seed=9 + i), wgrad=False)
            bufs.append(b)
        if args.case == "wgrad_grouped":
            fn = lambda: wgrad_grouped(bufs)  # noqa: E731
        else:
            def fn():
                for b in bufs:
                    t = b.t
                    J.jetfp8_gemm_wgrad(t["dyqT"], t["sdyT"], t["xqT"], t["sxT"], t["dw"])
        _time_case(args, fn, sum(l.gemm_flops for l in lins), "TFLOP/s", [M, 0, 0])
        return
    if args.case == "quant_weight_grouped":
        # the four Llama-3.1-8B layer weights (with transposes) in one grouped launch
        from fp8_mixed_granularity_gb300.linear import quant_weights_grouped
        lins = W.llama8b_training(128)
        bufs = [LinearBuffers(lin, dev) for lin in lins]
        ws = [W.device_normal((lin.N, lin.K), 0.02, dev, seed=5 + i) for i, lin in enumerate(lins)]
        nbytes = sum(lin.N * lin.K * QUANT_BYTES["quant_weight"] for lin in lins)
        _time_case(args, lambda: quant_weights_grouped(bufs, ws), nbytes, "GB/s", [0, 0, 0])
        return
    if args.case == "rmsnorm_bwd":
        # RMSNorm backward on an [M, H] = [M, K] activation with its forward's r
        x = W.device_activations(M, K, dev, seed=1)
        gamma = W.device_uniform((K,), 0.5, 1.5, dev, seed=4)
        dy = W.device_normal((M, K), 1e-3, dev, seed=3)
        xq, sx = J.empty_rowgroup_quant(M, K, dev)
        rstd = torch.empty(M, dtype=torch.float32, device=dev)
        J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, xq, sx, rstd)
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dg = torch.empty(K, dtype=torch.float32, device=dev)
        ws = torch.empty(J.jetfp8_rmsnorm_bwd_workspace_bytes(M, K), dtype=torch.uint8, device=dev)
        fn = lambda: J.jetfp8_rmsnorm_bwd(x, gamma, rstd, dy, dx, dg, ws)  # noqa: E731
        _time_case(args, fn, M * K * QUANT_BYTES[args.case], "GB/s", [M, N, K])
        return
    if args.case in ("fprop_nvfp4", "quant_nvfp4"):
        # FP4 variant: the row quantiser of X [M, K] (bf16 in; codes, block and
        # row scales out), or the block-scaled FProp Y = X̂ Ŵᵀ [M, N]
        x = W.device_activations(M, K, dev, seed=1)
        xq, xsf, gx = J.empty_nvfp4(M, K, dev)
        if args.case == "quant_nvfp4":
            fn = lambda: J.jetfp8_quant_nvfp4(x, xq, xsf, gx)  # noqa: E731
            _time_case(args, fn, M * K * (2 + 0.5 + 1 / 16) + 4 * M, "GB/s", [M, N, K])
            return
        w = W.device_normal((N, K), 0.02, dev, seed=2)
        wq, wsf, gw = J.empty_nvfp4(N, K, dev)
        J.jetfp8_quant_nvfp4(x, xq, xsf, gx)
        J.jetfp8_quant_nvfp4(w, wq, wsf, gw)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        fn = lambda: J.jetfp8_gemm_fprop_nvfp4(xq, xsf, gx, wq, wsf, gw, y)  # noqa: E731
        _time_case(args, fn, 2.0 * M * N * K, "TFLOP/s", [M, N, K])
        return
    if args.case in ("swiglu_quant", "swiglu_bwd"):
        # SwiGLU of an [M, 2I] gate/up output, I = N / 2 (N = the gate/up width)
        I = N // 2
        gu = W.device_normal((M, 2 * I), 1.0, dev, seed=5)
        dh = W.device_normal((M, I), 1e-3, dev, seed=6)
        hq, hs = J.empty_rowgroup_quant(M, I, dev)
        dgu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev)
        if args.case == "swiglu_quant":
            fn = lambda: J.jetfp8_swiglu_quant(gu, hq, hs)
        else:
            fn = lambda: J.jetfp8_swiglu_bwd(gu, dh, dgu)
        _time_case(args, fn, M * I * QUANT_BYTES[args.case], "GB/s", [M, N, K])
        return
    lin = W.Linear("case", M, K, N)
    b = LinearBuffers(lin, dev, rmsnorm=args.case == "rmsnorm_quant")
    x = W.device_activations(M, K, dev, seed=1)
    w = W.device_normal((N, K), 0.02, dev, seed=2)
    dy = W.device_normal((M, N), 1e-3, dev, seed=3)
    gamma = W.device_uniform((K,), 0.5, 1.5, dev, seed=4)
    b.forward(x, w, gamma)
    if args.case not in ("fprop", "fprop_quant", "fprop_then_quant", "quant_act", "rmsnorm_quant",
                         "quant_weight") or M % 128 == 0:
        b.backward(dy)   # the backward quantisers need M to be a multiple of 128
    t = b.t
    yq, ys = J.empty_rowgroup_quant(M, N, dev)

    def fprop_then_quant():
        J.jetfp8_gemm_fprop(t["xq"], t["sx"], t["wq"], t["sw"], t["y"])
        J.jetfp8_quant_act_1x128(t["y"], yq, ys)

    calls = {
        "fprop": (lambda: J.jetfp8_gemm_fprop(t["xq"], t["sx"], t["wq"], t["sw"], t["y"]), 2 * M * N * K, "TFLOP/s"),
        # FProp whose epilogue also emits the 1×128-quantised output, against
        # FProp followed by the separate quantiser on its bf16 output
        "fprop_quant": (lambda: J.jetfp8_gemm_fprop_quant(t["xq"], t["sx"], t["wq"], t["sw"], yq, ys, t["y"]),
                        2 * M * N * K, "TFLOP/s"),
        "fprop_then_quant": (fprop_then_quant, 2 * M * N * K, "TFLOP/s"),
        "dgrad": (lambda: J.jetfp8_gemm_dgrad(t["dyq"], t["sdy"], t["wqT"], t["sw"], t["dx"]), 2 * M * N * K, "TFLOP/s"),
        "wgrad": (lambda: J.jetfp8_gemm_wgrad(t["dyqT"], t["sdyT"], t["xqT"], t["sxT"], t["dw"]), 2 * M * N * K, "TFLOP/s"),
        "quant_act": (lambda: J.jetfp8_quant_act_1x128(x, t["xq"], t["sx"]), M * K * QUANT_BYTES["quant_act"], "GB/s"),
        "rmsnorm_quant": (lambda: J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, t["xq"], t["sx"], t["rstd"]),
                          M * K * QUANT_BYTES["rmsnorm_quant"] + 2 * K + 4 * M, "GB/s"),
        "quant_weight": (lambda: J.jetfp8_quant_weight_128x128(w, t["wq"], t["sw"], t["wqT"]),
                         N * K * QUANT_BYTES["quant_weight"], "GB/s"),
        "quant_grad_dual": (lambda: J.jetfp8_quant_grad_dual(dy, t["dyq"], t["sdy"], t["dyqT"], t["sdyT"]),
                            M * N * QUANT_BYTES["quant_grad_dual"], "GB/s"),
        "requant": (lambda: J.jetfp8_requant_rowgrp_to_colgrp(t["xq"], t["sx"], t["xqT"], t["sxT"]),
                    M * K * QUANT_BYTES["requant"], "GB/s"),
    }
    fn, work, unit = calls[args.case]
    _time_case(args, fn, work, unit, [M, N, K])


def _time_case(args, fn, work, unit, shape):
    import torch
    from fp8_mixed_granularity_gb300 import jetfp8 as J
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    if args.graph:
        # one graph of `steps` launches, replayed `steps` times; per-launch time
        stream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()   # warm the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(args.steps):
                    fn()
        graph.replay()
        torch.cuda.synchronize()
        ms = []
        for _ in range(5):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(); graph.replay(); e.record()
            torch.cuda.synchronize()
            ms.append(s.elapsed_time(e) / args.steps)
        J.jetfp8_get_last_device_error()
        ms.sort()
        med = ms[len(ms) // 2]
    else:
        evs = []
        for _ in range(args.steps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(); fn(); e.record()
            evs.append((s, e))
        torch.cuda.synchronize()
        J.jetfp8_get_last_device_error()
        ms = sorted(s.elapsed_time(e) for s, e in evs)
        med = ms[len(ms) // 2]
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    print(json.dumps({"case": args.case, "shape": shape, "median_ms": med, "min_ms": ms[0],
                      "value": work / (med * 1e-3) / scale, "unit": unit, "graph": bool(args.graph),
                      "gemm_path": args.gemm_path}),
          flush=True)


def main():
    args = parse_args()
    if args.case is not None:
        run_case(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
