#!/usr/bin/env python3
"""Throughput of the autotuned tcgen05 GEMM on one workload; prints one JSON line.

Default workload: bf16 C = gelu(A·B + bias), M = N = 1000, K = 8192 (the
under-filled shape of "Compilers and Kernel Languages", where a fixed 128x128
tile leaves most SMs idle).  One step = one GEMM on each of R rotating input
sets (R chosen so the sets together exceed twice the L2, so no step is served
from L2); the plan is tuned on first use and cached (that is the method), and
steps reuse it.  The timed region replays a CUDA graph of one step K times.

Also reported: the roofline of the GEMM kernel against MEASURED_PEAKS.json,
the fixed 128x128 tile on the same protocol (tuned-vs-fixed speedup), the
tuner's rank agreement and search cost, an end-to-end number through the
host-buffer entry point (copies inside the timed region), the CPU oracle on
the host cores, and SM clocks sampled during the timed region.

  python bench.py [--steps K] [--warmup W] [--workload NAME] [--impl reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); value = work of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (or GB/s) per shape, % of roofline; tuned vs fixed-128x128 speedup"
DEFAULT_WORKLOAD = "bf16_gelu_1000x1000x8192"
# Timed beside the headline in the same run: the correctness-sized fp32 case,
# the large square multiply and the 16-token decode (the targets are set on the
# last two: >= 70% of the dense bf16 tensor peak and >= 80% of HBM bandwidth).
PER_WORKLOAD = ["fp32_relu_256", "bf16_relu_8192", "bf16_decode_16x8192x28672"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of CPU work for the oracle baseline (our arm)")
    ap.add_argument("--cpu-budget", type=float, default=120.0,
                    help="total seconds of CPU work for the reference arm's steps")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fixed", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload block (the 256^3 fp32, 8192^3 and 16-token decode workloads)")
    ap.add_argument("--eager", action="store_true", help="launch from Python instead of a CUDA graph")
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload (the four headline shapes and the 30-shape sweep): one "
                         "JSON line per shape with tuned and fixed-tile throughput and roofline share")
    ap.add_argument("--workloads", default=None,
                    help="with --sweep: comma-separated workload names instead of the full list")
    ap.add_argument("--search-quality", action="store_true",
                    help="model-guided top-k vs random-k at equal measurement budgets, from one "
                         "exhaustive tuning table per workload (one JSON line per workload)")
    ap.add_argument("--operands", choices=["none", "B", "AB"], default="none",
                    help="operands declared independent of the previous GEMM: none (the default) makes every "
                         "launch wait for the previous kernel; B as the weights of a layer chain, whose A is "
                         "the previous layer's output; AB for independent GEMMs")
    ap.add_argument("--config", default=None,
                    help="explicit tile config bm,bn,bk,stages,raster,group,split_k,cta_group,swap_ab "
                         "(skips tuning; used to profile one configuration)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def elt_sizes(dtype):
    """(operand bytes, bytes of C and bias): FP8 operands give a bf16 C."""
    return {"bf16": (2, 2), "fp8": (1, 2), "mxfp8": (1, 2)}.get(dtype, (4, 4))


def peak_ratio(dtype):
    """Dense tensor peak of `dtype` relative to bf16 (the nominal ratios:
    tf32 1.1, bf16 2.25, fp8 4.5 PFLOP/s; block-scaled FP8 runs at the FP8 rate)."""
    return {"bf16": 1.0, "fp8": 2.0, "mxfp8": 2.0}.get(dtype, 0.5)


def scale_bytes_of(w):
    """Block-scaled FP8: one E8M0 byte per 32 elements of K, for A and for B."""
    if w.dtype != "mxfp8":
        return 0
    kb = (w.K + 31) // 32
    return (w.M + w.N) * kb


def work_of(w):
    """FLOPs and compulsory bytes of one GEMM (a gated C is half the fused width)."""
    from autotuning_tcgen05_tmem_gb300 import inputs
    elt, eo = elt_sizes(w.dtype)
    flops = 2.0 * w.M * w.N * w.K
    bytes_ = (w.M * w.K + w.K * w.N) * elt + scale_bytes_of(w) + (w.N * eo if w.epi != "none" else 0) + \
        w.M * inputs.out_cols(w) * eo
    return flops, bytes_, elt


def set_bytes_of(w):
    from autotuning_tcgen05_tmem_gb300 import inputs
    elt, eo = elt_sizes(w.dtype)
    return (w.M * w.K + w.K * w.N) * elt + scale_bytes_of(w) + (w.N + w.M * inputs.out_cols(w)) * eo


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 100 ms.  Each sample is placed in time by
    nvidia-smi's own timestamp (its output reaches the pipe in bursts, so the
    time it is read says little), and `mark` brackets the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()
        deadline = time.time() + 5
        while not self.samples and time.time() < deadline:
            time.sleep(0.02)

    def _reader(self):
        import datetime
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except (ValueError, IndexError):
                t = time.time()
            self.samples.append((t, f))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self):
        if self.proc is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        return self.summary_between(self.t0, self.t1)

    def summary_between(self, t0, t1):
        if self.proc is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        inside = [s for t, s in list(self.samples) if t0 is not None and t1 is not None and t0 <= t <= t1]
        near = inside or [s for _t, s in list(self.samples)]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in near if len(s) > 1 and num(s[1]) is not None]
        mx = [num(s[2]) for s in near if len(s) > 2 and num(s[2]) is not None]
        pw = [num(s[3]) for s in near if len(s) > 3 and num(s[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in near:
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons),
                "samples_in_timed_region": len(inside),
                "samples_total": len(self.samples),
                "window": "timed region" if inside else "whole run (no sample fell inside the timed region)"}


# ---------------------------------------------------------------------------
# CPU oracle (rank 0, N = 1 only) — the reported CPU baseline
# ---------------------------------------------------------------------------

def oracle_slab(w, threads):
    """The oracle of workload w as a function of a row count (the first rows of
    the product), and the thread count it uses."""
    from autotuning_tcgen05_tmem_gb300 import inputs
    from oracle import gemm as og
    epi = {"none": 0, "bias": 1, "relu": 2, "gelu": 3}[w.epi]
    if w.dtype == "mxfp8":
        from oracle import mx
        A, SA, B, SB, bias = inputs.make_mx_workload(w, seed=0)
        # (numpy's fp64 matrix product: its BLAS threads, one per core by default)
        return (lambda rows: mx.mx_gemm(A[:rows], SA[:rows], B, SB, bias, epi)), threads
    og.build()
    A, B, bias = inputs.make_workload(w, seed=0)
    return (lambda rows: og.gemm(A[:rows], B, bias, epi, threads=threads)), threads


def cpu_oracle_run(w, seconds: float, total_budget_s: float | None = None, threads: int | None = None):
    """Time the fp64 oracle on a slab of rows of the workload (on every host
    core, or on `threads`); returns (TFLOP/s, threads, sample text, seconds)."""
    from oracle import gemm as og
    run, threads = oracle_slab(w, threads or og.default_threads())
    cal = min(w.M, max(1, threads))
    t0 = time.perf_counter()
    run(cal)
    per_row = max((time.perf_counter() - t0) / cal, 1e-7)
    rows = int(min(w.M, max(cal, seconds / per_row)))
    passes = 0
    t0 = time.perf_counter()
    while True:           # whole passes over the slab until `seconds` of CPU work
        run(rows)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds or dt >= 30.0:
            break
    flops = 2.0 * rows * w.N * w.K * passes
    sample = (f"rows 0..{rows - 1} of {w.M} (all {w.N} columns, full K={w.K}), fp64 oracle, "
              f"{threads} threads, {passes} pass(es)")
    return flops / dt / 1e12, threads, sample, dt


def reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import gemm as og
    run, threads = oracle_slab(w, og.default_threads())
    cal = min(w.M, max(1, threads))
    t0 = time.perf_counter()
    run(cal)
    per_row = max((time.perf_counter() - t0) / cal, 1e-7)
    budget = args.cpu_budget / max(1, args.steps + args.warmup)   # seconds of CPU work per step
    rows = int(min(w.M, max(1, budget / per_row)))
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    value = flops * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": w.epi,
                       "step": f"rows 0..{rows - 1} of the product (bounded sample)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{rows} of {w.M} rows per step, fp64, {threads} threads"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def make_sets(w, nsets, device):
    """Rotating input sets, drawn on the device from seeded generators:
    (A, B, bias, C), or for block-scaled FP8 (A, SA, B, SB, bias, C) with the
    scales packed once, outside any timed region, as a weight's would be."""
    import torch
    import autotuning_tcgen05_tmem_gb300 as g
    from autotuning_tcgen05_tmem_gb300 import inputs
    sets = []
    for s in range(nsets):
        C = torch.empty(w.M, inputs.out_cols(w), dtype=inputs.out_torch_dtype(w.dtype), device=device)
        if w.dtype == "mxfp8":
            A, SA, B, SB, bias = inputs.make_mx_workload(w, seed=100 + 10 * s, device=device)
            sets.append((A, g.mx_pack_scales(SA, w.M, w.K, False), B, g.mx_pack_scales(SB, w.N, w.K, True),
                         bias, C))
        else:
            A, B, bias = inputs.make_workload(w, seed=100 + 10 * s, device=device)
            sets.append((A, B, bias, C))
    return sets


def run_set(plan, s, stream):
    """One GEMM of `plan` on input set `s` (see make_sets)."""
    if len(s) == 6:
        A, SA, B, SB, bias, C = s
        plan.run_mx(A, SA, B, SB, bias, C, None, stream)
    else:
        A, B, bias, C = s
        plan.run(A, B, bias, C, stream)


def time_plan(plan, sets, steps, warmup, eager=False):
    """Average seconds per step (one GEMM per rotating set) over `steps`
    replays of a CUDA graph of one step; returns (sec_per_step, mode, stream)."""
    import torch
    stream = torch.cuda.Stream()

    def one_step():
        for s in sets:
            run_set(plan, s, stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one_step()
    torch.cuda.synchronize()
    mode = "eager"
    graph = None
    if not eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for s in sets:
                    run_set(plan, s, torch.cuda.current_stream())
            mode = "cuda_graph"
        except Exception:
            graph = None
            torch.cuda.synchronize()
    run = (lambda: graph.replay()) if graph is not None else one_step
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
    torch.cuda.synchronize()
    return run, mode, stream


OPERAND_NOTES = {
    "none": "every launch waits for the previous kernel before touching memory",
    "B": "B declared independent (the weights of a layer chain): each launch copies its first stages of B "
         "while the previous GEMM drains, and A after it has finished",
    "AB": "A and B declared independent (independent GEMMs): operand copies and MMAs run ahead of the previous "
          "GEMM's drain, and tiles that leave SMs idle fill them with the next GEMM; C stores still wait",
}


def declared(operands: str) -> str:
    """The operand string a plan takes for a --operands choice."""
    return "" if operands == "none" else operands


def region_gemm_seconds(plan, sets, steps, warmup, eager=False) -> float:
    """Seconds per GEMM over `steps` steps of `plan` (CUDA events on its stream)."""
    import torch
    run, _mode, stream = time_plan(plan, sets, steps, max(3, warmup // 4), eager)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            run()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps / len(sets)


def combine_ranks(elapsed: float, pg=None) -> float:
    """Max of the ranks' timed regions (the slowest replica bounds the job)."""
    if pg is None:
        return elapsed
    import torch
    t = torch.tensor([elapsed], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_gemm: float, gemms_per_step: int, steps: int, world: int, elapsed: float) -> float:
    """Whole-job TFLOP/s: the work of every replica over the max rank time."""
    return flops_per_gemm * gemms_per_step * steps * world / elapsed / 1e12


def time_gemm(plan, sets, steps, warmup):
    """Seconds per GEMM of `plan` over rotating sets (graph replay, CUDA events)."""
    import torch
    run, mode, stream = time_plan(plan, sets, steps, warmup)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            run()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps / len(sets)


def captured_traffic(name, cfg):
    """DRAM bytes of one launch of this workload's kernel in this configuration,
    from the committed ncu summaries (profiles/traffic.json), or None when no
    capture of the current build exists for it."""
    from autotuning_tcgen05_tmem_gb300 import _build
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        ents = json.load(f).get(name) or []
    for ent in ents if isinstance(ents, list) else [ents]:
        if ent.get("source_digest") == _build._sources_digest() and ent.get("config") == list(cfg):
            return ent.get("dram_bytes_per_launch")
    return None


def power_capped(clocks_summary) -> bool:
    """Whether the GPU ran under its power cap during a timed region: the
    sustained tensor peak is then the fair denominator, else the burst one."""
    if not clocks_summary:
        return False
    mhz, mx = clocks_summary.get("sm_mhz"), clocks_summary.get("sm_max_mhz")
    return "sw_power_cap" in clocks_summary.get("reasons", []) or bool(mhz and mx and mhz < 0.95 * mx)


def rotating_sets(w, l2_bytes, cap=512):
    """How many input sets a step rotates over: enough that together they
    exceed twice the L2 (so no timed GEMM is served from L2), at most `cap`."""
    return int(min(cap, max(1, math.ceil(2 * l2_bytes / set_bytes_of(w)))))


def measure_workload(w, devp, peaks, peak_src, operands="none", clocks=None, target_s=0.5,
                     tune_report=False):
    """The tuned plan of workload w and the fixed 128x128 tile, each timed over
    rotating input sets (graph replay, CUDA events, about `target_s` seconds of
    GEMMs); returns a dict with the value in the bound's unit, the roofline
    share of the GEMM kernel, tuned vs fixed, the tuned configuration and the
    SM clocks sampled during the tuned timing."""
    import torch
    import autotuning_tcgen05_tmem_gb300 as g
    flops, cbytes, _elt = work_of(w)
    nsets = rotating_sets(w, devp.l2_bytes)
    sets = make_sets(w, nsets, torch.device("cuda", torch.cuda.current_device()))
    t0 = time.perf_counter()
    plan = g.plan(w.M, w.N, w.K, w.dtype, w.epi)
    tune_s = time.perf_counter() - t0
    try:
        plan.set_independent_operands(declared(operands))
        est = time_gemm(plan, sets, 2, 2)                     # calibrate the step count
        steps = int(min(20000, max(3, target_s / max(est * nsets, 1e-7))))
        if clocks is not None:
            clocks.mark("t0")
        t_tuned = time_gemm(plan, sets, steps, 5)
        if clocks is not None:
            clocks.mark("t1")
        assert plan.status() == 0, g.last_error()
        shape_clocks = clocks.summary() if clocks is not None else None
        fixed = g.fixed_config(w.dtype, devp)
        with g.plan_with_config(w.M, w.N, w.K, w.dtype, w.epi, fixed) as fp:
            fp.set_independent_operands(declared(operands))
            t_fixed = time_gemm(fp, sets, max(3, steps // 2), 5)
            assert fp.status() == 0, g.last_error()
        t_decl = {}
        for decl in ("none", "B", "AB"):
            if decl != operands:
                plan.set_independent_operands(declared(decl))
                t_decl[decl] = time_gemm(plan, sets, max(3, steps // 4), 5) * 1e6
        plan.set_independent_operands(declared(operands))
        cfg = list(plan.config.astuple())
        info = plan.launch_info
    finally:
        plan.close()
    # Under the power cap (seen in the clocks sampled during the timing) the
    # sustained tensor peak is the denominator; otherwise the burst one.
    region_s = t_tuned * steps * nsets
    sustained = power_capped(shape_clocks) if shape_clocks is not None else region_s > 1.0
    bf16_peak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops", 1900.0)
    tpeak = bf16_peak * peak_ratio(w.dtype)
    bw = peaks.get("hbm_gbs", 6800.0)
    tensor_bound = flops / (tpeak * 1e12) >= cbytes / (bw * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": flops / t_tuned / 1e12, "peak": tpeak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": cbytes / t_tuned / 1e9, "peak": bw, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = captured_traffic(w.name, cfg)
    roof["peak_source"] = (f"{peak_src} bf16 {'sustained' if sustained else 'burst'} x {peak_ratio(w.dtype)}"
                           if tensor_bound else f"{peak_src} HBM")
    out = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype, "epilogue": w.epi,
           "value": roof["achieved"], "unit": roof["unit"],
           "tflops": flops / t_tuned / 1e12, "gbs": cbytes / t_tuned / 1e9, "roofline": roof,
           "tuned_config": cfg, "tuned_us": t_tuned * 1e6, "fixed_us": t_fixed * 1e6,
           "tuned_vs_fixed": t_fixed / t_tuned, "operands": operands, "tuned_us_other_operands": t_decl,
           "splitk_route": g.SPLITK_ROUTES.get(info.splitk_route, str(info.splitk_route)),
           "plan_seconds": tune_s, "timed_region_s": region_s, "rotating_sets": nsets,
           "l2": (f"{nsets} sets of {set_bytes_of(w) / 1e6:.1f} MB rotate ({nsets * set_bytes_of(w) / 1e6:.0f} MB "
                  f"{'>' if nsets * set_bytes_of(w) > 2 * devp.l2_bytes else '<='} 2 x L2)"),
           "clocks": shape_clocks}
    if tune_report:
        tr = g.tune(w.M, w.N, w.K, w.dtype, w.epi, topk=int(os.environ.get("GEMM_TUNE_TOPK", "24")))
        st = tr.stats
        out["tune"] = {"candidates": st.n_candidates, "measured": st.n_measured, "kendall_tau": st.kendall_tau,
                       "top1_hit": st.top1_hit, "regret": st.regret, "search_seconds": st.tune_seconds}
    del sets
    torch.cuda.empty_cache()
    return out


def sweep(args):
    """One JSON line per workload: tuned vs fixed throughput and roofline share."""
    import autotuning_tcgen05_tmem_gb300 as g
    from autotuning_tcgen05_tmem_gb300 import _build, inputs
    _build.build()
    peaks, peak_src = load_peaks()
    os.environ.setdefault("GEMM_PEAK_BF16_TFLOPS", str(peaks.get("bf16_tflops", 1900.0)))
    os.environ.setdefault("GEMM_HBM_GBS", str(peaks.get("hbm_gbs", 6800.0)))
    devp = g.device_params_query()
    names = ["fp32_relu_256", "bf16_gelu_1000x1000x8192", "bf16_relu_8192", "bf16_decode_16x8192x28672"] + \
        [w.name for w in inputs.SWEEP] + ["fp8_gelu_1000x1000x8192", "fp8_relu_8192", "fp8_decode_16x8192x28672",
                                          "mxfp8_gelu_1000x1000x8192", "mxfp8_relu_8192",
                                          "mxfp8_decode_16x8192x28672"] + \
        [n for n in inputs.WORKLOADS if "_gate_up_t" in n and n.split("_")[1] in inputs.GATED]
    if args.workloads:
        names = [n for n in args.workloads.split(",")]
    clocks = ClockSampler(0)      # sampled through the sweep; each line summarises its tuned timing
    clocks.start()
    for name in names:
        w = inputs.WORKLOADS[name]
        # Host side of the selection alone: enumerate and rank by the model
        # (microseconds; "Autotuning & cost models" §5 weighs it against the
        # on-device search).
        t0 = time.perf_counter()
        cands = g.enumerate_configs(w.M, w.N, w.K, w.dtype, w.epi, devp)
        preds = [g.model_predict(w.M, w.N, w.K, w.dtype, w.epi, c_, devp).predicted_us for c_ in cands]
        host_rank_us = (time.perf_counter() - t0) * 1e6
        line = measure_workload(w, devp, peaks, peak_src, args.operands, clocks, target_s=0.3)
        line.update({"candidates": len(cands), "host_rank_us": host_rank_us,
                     "model_best_us": min(preds) if preds else None,
                     "bound": line["roofline"]["bound"], "roofline_frac": line["roofline"]["frac"]})
        print(json.dumps(line), flush=True)
    clocks.stop()
    return 0


def expected_random_best(measured, k):
    """E[best of k distinct uniform draws] as a fraction of the true best:
    with values sorted ascending, P(min = v_i) = C(n-i, k-1) / C(n, k)."""
    v = sorted(measured)
    n = len(v)
    if k >= n:
        return 1.0
    total = math.comb(n, k)
    return sum(math.comb(n - i, k - 1) / total * v[0] / v[i - 1] for i in range(1, n - k + 2))


def search_quality(args):
    import autotuning_tcgen05_tmem_gb300 as g
    from autotuning_tcgen05_tmem_gb300 import _build, inputs
    _build.build()
    peaks, _ = load_peaks()
    os.environ.setdefault("GEMM_PEAK_BF16_TFLOPS", str(peaks.get("bf16_tflops", 1900.0)))
    os.environ.setdefault("GEMM_HBM_GBS", str(peaks.get("hbm_gbs", 6800.0)))
    budgets = [1, 2, 4, 8, 16, 24, 32]
    names = ["bf16_gelu_1000x1000x8192", "bf16_relu_8192", "bf16_decode_16x8192x28672", "fp32_relu_256"] + \
        [w.name for w in inputs.SWEEP]
    tables = {}
    for name in names:
        w = inputs.WORKLOADS[name]
        r = g.tune_search(w.M, w.N, w.K, w.dtype, w.epi, g.SEARCH_EXHAUSTIVE, 0)
        rows = [row for row in r.rows if row.measured_us > 0]
        if w.dtype == "bf16":
            tables[name] = {row.config.astuple(): row.measured_us for row in rows}
        meas = [row.measured_us for row in rows]
        best = min(meas)
        by_model = sorted(rows, key=lambda row: row.model_rank)
        model_q = {k: best / min(row.measured_us for row in by_model[:k]) for k in budgets}
        random_q = {k: expected_random_best(meas, k) for k in budgets}
        print(json.dumps({"workload": name, "candidates": len(rows), "best_us": best,
                          "kendall_tau": r.stats.kendall_tau, "model_quality": model_q,
                          "random_quality_expected": random_q, "search_seconds": r.stats.tune_seconds}),
              flush=True)
    print(json.dumps({"shipped_set": shipped_set_report(tables)}), flush=True)
    return 0


def shipped_set_report(tables, sizes=(4, 8, 16, 30)):
    """Quality of a small shipped configuration set chosen greedily from the
    exhaustive tables (gemm_select_config_set): in sample, and leave-one-out
    (chosen without a workload, judged on it)."""
    import numpy as np
    import autotuning_tcgen05_tmem_gb300 as g
    names = sorted(tables)
    cols = sorted({c for t in tables.values() for c in t})
    idx = {c: j for j, c in enumerate(cols)}
    mat = np.zeros((len(names), len(cols)))
    for i, n in enumerate(names):
        for c, us in tables[n].items():
            mat[i, idx[c]] = us
    out = {"workloads": len(names), "configurations": len(cols)}
    for k in sizes:
        chosen, mean, worst = g.select_config_set(mat, k)
        loo = []
        for i in range(len(names)):
            rest = np.delete(mat, i, axis=0)
            pick, _, _ = g.select_config_set(rest, k)
            runs = [mat[i, j] for j in pick if mat[i, j] > 0]
            best = mat[i][mat[i] > 0].min()
            loo.append(min(runs) / best if runs else float("inf"))
        fin = lambda v: v if math.isfinite(v) else None   # null: some workload no member runs
        out[str(k)] = {"in_sample_mean": fin(mean), "in_sample_worst": fin(worst),
                       "leave_one_out_mean": fin(float(np.mean(loo))), "leave_one_out_worst": fin(float(np.max(loo))),
                       "configs": [list(cols[j]) for j in chosen]}
    return out


def main():
    args = parse_args()
    from autotuning_tcgen05_tmem_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w)
    if args.sweep:
        return sweep(args)
    if args.search_quality:
        return search_quality(args)

    import torch
    import autotuning_tcgen05_tmem_gb300 as g
    from autotuning_tcgen05_tmem_gb300 import _build
    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    os.environ.setdefault("GEMM_PEAK_BF16_TFLOPS", str(peaks.get("bf16_tflops", 1900.0)))
    os.environ.setdefault("GEMM_HBM_GBS", str(peaks.get("hbm_gbs", 6800.0)))
    flops, cbytes, elt = work_of(w)
    devp = g.device_params_query()
    set_bytes = set_bytes_of(w)
    nsets = rotating_sets(w, devp.l2_bytes)
    sets = make_sets(w, nsets, dev)

    # --- plan: tune once (cost model + measurement), cached by shape ---------
    t0 = time.perf_counter()
    if args.config:
        plan = g.plan_with_config(w.M, w.N, w.K, w.dtype, w.epi,
                                  g.make_config(*[int(x) for x in args.config.split(",")]))
    else:
        plan = g.plan(w.M, w.N, w.K, w.dtype, w.epi)
    plan_s = time.perf_counter() - t0
    cfg = plan.config
    # By default nothing is declared independent: every launch waits for the
    # previous kernel, as in any chain of GEMMs (--operands picks others).
    plan.set_independent_operands(declared(args.operands))
    launches_per_gemm = 1 + plan.launch_info.b_transposed   # (+ the transpose into a K-major B)

    run, mode, stream = time_plan(plan, sets, args.steps, args.warmup, args.eager)
    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark("t0")
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            run()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    if pg:
        pg.barrier()
    clocks.stop()
    assert plan.status() == 0, g.last_error()
    elapsed = combine_ranks(e0.elapsed_time(e1) / 1e3, pg)
    sec_per_step = elapsed / args.steps
    gemm_s = sec_per_step / nsets
    value = job_value(flops, nsets, args.steps, world, elapsed)

    # --- roofline of the GEMM kernel -----------------------------------------
    clock_summary = clocks.summary()
    sustained = power_capped(clock_summary)
    # another dtype's peak: the measured bf16 peak x the nominal dense ratio
    tpeak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops", 1900.0) * peak_ratio(w.dtype)
    bw = peaks.get("hbm_gbs", 6800.0)
    t_compute = flops / (tpeak * 1e12)
    t_memory = cbytes / (bw * 1e9)
    traffic = captured_traffic(w.name, cfg.astuple())
    if t_compute >= t_memory:
        roof = {"bound": "tensor", "achieved": flops / gemm_s / 1e12, "peak": tpeak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": cbytes / gemm_s / 1e9, "peak": bw, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic
    roof["peak_source"] = f"{peak_src} ({'sustained' if sustained and roof['bound'] == 'tensor' else 'burst'})"
    roof["algorithmic_per_launch"] = flops if roof["bound"] == "tensor" else cbytes
    roof["kernel"] = "gemm_tcgen05_kernel"

    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": sec_per_step * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
           "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "epilogue": w.epi,
                      "dtype": w.dtype, "tile_config": cfg.asdict(),
                      "splitk_route": g.SPLITK_ROUTES.get(plan.launch_info.splitk_route,
                                                          str(plan.launch_info.splitk_route)),
                      "step": f"{nsets} GEMMs, one per rotating input set",
                      "l2": f"inputs rotate over {nsets} sets ({nsets * set_bytes / 1e6:.0f} MB > 2 x L2 "
                            f"{devp.l2_bytes / 1e6:.0f} MB)" if nsets * set_bytes > 2 * devp.l2_bytes
                      else f"each set ({set_bytes / 1e6:.0f} MB) exceeds L2",
                      "launch": mode, "parallelism": f"replicas x{world}",
                      "operands": OPERAND_NOTES[args.operands]},
           "roofline": roof,
           "gpu_launches": args.steps * nsets * launches_per_gemm,
           "clocks": clock_summary,
           "plan_seconds": plan_s}

    # --- tuned vs fixed 128x128, and the tuner's own report -------------------
    if not args.no_fixed and rank == 0:
        fixed = g.fixed_config(w.dtype, devp)
        with g.plan_with_config(w.M, w.N, w.K, w.dtype, w.epi, fixed) as fp:
            fp.set_independent_operands(declared(args.operands))
            fixed_gemm_s = region_gemm_seconds(fp, sets, max(20, args.steps // 4), args.warmup, args.eager)
        out["fixed_config"] = fixed.asdict()
        out["fixed_value"] = flops / fixed_gemm_s / 1e12
        out["tuned_vs_fixed"] = fixed_gemm_s / gemm_s
        tr = g.tune(w.M, w.N, w.K, w.dtype, w.epi, topk=int(os.environ.get("GEMM_TUNE_TOPK", "24")))
        st = tr.stats
        saved_us = max(st.fixed_us - st.best_us, 0.0) if st.fixed_us > 0 else 0.0
        out["tune"] = {"candidates": st.n_candidates, "measured": st.n_measured,
                       "kendall_tau": st.kendall_tau, "spearman_rho": st.spearman_rho,
                       "top1_hit": st.top1_hit, "regret": st.regret, "search_seconds": st.tune_seconds,
                       "best_us": st.best_us, "fixed_us": st.fixed_us,
                       "break_even_calls": (st.tune_seconds / (saved_us * 1e-6)) if saved_us > 0 else None}

    # --- the other operand declarations, tuned and fixed tile ----------------
    if not args.no_fixed and rank == 0:
        alt = {}
        for decl in ("none", "B", "AB"):
            if decl == args.operands:
                continue
            plan.set_independent_operands(declared(decl))
            v = flops / region_gemm_seconds(plan, sets, max(20, args.steps // 4), args.warmup, args.eager) / 1e12
            with g.plan_with_config(w.M, w.N, w.K, w.dtype, w.epi, g.fixed_config(w.dtype, devp)) as fp:
                fp.set_independent_operands(declared(decl))
                fv = flops / region_gemm_seconds(fp, sets, max(20, args.steps // 4), args.warmup,
                                                 args.eager) / 1e12
            alt[decl] = {"value": v, "fixed_value": fv, "tuned_vs_fixed": v / fv, "note": OPERAND_NOTES[decl]}
        plan.set_independent_operands(declared(args.operands))
        out["other_operand_declarations"] = alt

    # --- end to end through the host-buffer entry point ------------------------
    if not args.no_e2e and rank == 0 and w.dtype == "mxfp8":
        out["e2e"] = None
        out["e2e_note"] = "the host-buffer entry point takes no scales; block-scaled FP8 runs from device buffers"
    elif not args.no_e2e and rank == 0:
        A, B, bias, _C = sets[0]
        hA, hB = A.cpu().pin_memory(), B.cpu().pin_memory()
        hb = bias.cpu().pin_memory() if bias is not None else None
        h2d = (w.M * w.K + w.K * w.N) * elt + (w.N * elt_sizes(w.dtype)[1] if bias is not None else 0)
        d2h = w.M * w.N * elt_sizes(w.dtype)[1]
        esteps = max(6, min(args.steps, 200))
        esteps += esteps % 2
        hC = [torch.empty(w.M, w.N, dtype=inputs.out_torch_dtype(w.dtype)).pin_memory() for _ in range(2)]
        hstream = torch.cuda.Stream()
        # (1) gemm_run_host_many, the library's pipelined host-buffer entry
        # point: every GEMM copies its inputs from pinned host memory and its
        # result back, inside the timed region; the library alternates two
        # streams (and two plans of the configuration) so one GEMM's copies
        # overlap the other's kernel, and reads both plans' status words.
        many = lambda n: plan.run_host_many([hA] * n, [hB] * n, None if hb is None else [hb] * n,
                                             [hC[i % 2] for i in range(n)], hstream)
        many(4)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        many(esteps)
        dt = (time.perf_counter() - t0) / esteps
        out["e2e"] = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "steps": esteps,
                      "path": "gemm_run_host_many (C ABI): pinned host buffers; per GEMM, copy A, B, bias in, "
                              "run, copy C out; two streams inside the library overlap one GEMM's copies with "
                              "the other's kernel; returns after every C is in host memory"}
        # (2) The synchronous host-buffer entry point, one call per step.
        for _ in range(3):
            plan.run_host(hA, hB, hb, hC[0], hstream)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(esteps):
            plan.run_host(hA, hB, hb, hC[0], hstream)
        dt = (time.perf_counter() - t0) / esteps
        assert plan.status() == 0, g.last_error()
        out["e2e_sync"] = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h, "steps": esteps,
                           "path": "gemm_run_host (C ABI: copies, one kernel, copy back, synchronise; per step)"}

    # --- the other workloads the targets are set on, timed in this run --------
    if not args.no_per_workload and rank == 0 and world == 1:
        pw_clocks = ClockSampler(local)
        pw_clocks.start()
        per = {}
        for name in PER_WORKLOAD:
            if name == w.name:
                continue
            r = measure_workload(inputs.WORKLOADS[name], devp, peaks, peak_src, args.operands, pw_clocks,
                                 target_s=1.5 if name == "bf16_relu_8192" else 0.5)
            per[name] = {k: r[k] for k in ("value", "unit", "roofline", "tuned_vs_fixed", "tuned_config",
                                           "tuned_us", "fixed_us", "splitk_route", "timed_region_s", "l2",
                                           "clocks")}
        pw_clocks.stop()
        out["per_workload"] = per

    # --- CPU oracle ------------------------------------------------------------
    if not args.no_cpu and rank == 0 and world == 1:
        v, cores, sample, secs = cpu_oracle_run(w, args.cpu_seconds)
        out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                               "sample": sample, "seconds": secs}
        if w.dtype != "mxfp8":      # (the block-scaled oracle's matrix product picks its own threads)
            v1, _c1, sample1, secs1 = cpu_oracle_run(w, min(3.0, args.cpu_seconds), threads=1)
            out["cpu_baseline"]["one_core"] = {"value": v1, "unit": "TFLOP/s", "cores": 1, "sample": sample1,
                                               "seconds": secs1}
    if rank == 0:
        print(json.dumps(out), flush=True)
    plan.close()
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
