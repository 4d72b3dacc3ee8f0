#!/usr/bin/env python3
"""Benchmark of the HiSparse swap-in resolution step on one GB300 (or N, one rank each).

A step is one hs_resolve call over every request of the high-concurrency long-context
workload (256 requests, one layer, context 131072, 4096 slots, k = 2048, 656-byte
entries -- 22 GB of pinned host KV -- 85 % of each selection kept, Zipf(1.05) refill):
hit test, LRU victims, page-table update and host->HBM fetch of the misses. Inputs (the
selection trace, the host KV history) are resident before timing; L2 is flushed between
timed steps.

The first pass over the trace after the store is created is timed on its own and
reported apart (key first_pass_after_create): the GPU's first reads of each host page
cost more than later ones. The headline is the steady state, the same steps again.

Prints one JSON line. Extra keys: per-kernel times and the roofline of the dominant
kernel, an end-to-end number through the host-buffer entry point, the CPU oracle on the
host cores, the DSA-style decode workload (32 requests) with its CUDA-graph, pooled,
policy, attention and append figures, the no-IO (all-hit) latency at 64 requests x
k = 2048, and the Quest-style layer-wise overlap; the gate figures come last.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "top-k resolutions/s; miss-fetch GB/s vs H2D peak; µs per layer-step"
UNIT = "resolutions/s"
FLUSH_BYTES = 512 << 20
ATTEND_HEADS = 128                # query heads of the attention consumer (DeepSeek-style MLA)
ATTEND_SCALE = 576 ** -0.5         # softmax scale over the 576-dim keys
H2D_PROBE_BYTES = 1 << 30


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long")
    ap.add_argument("--wait-limit-ms", type=float, default=None,
                    help="device wait limit of the attention context (hs_set_wait_limit); a profiler's "
                         "instrumented replays can run far slower than the default 20 ms allows")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the headline workload: no CPU, DSA, no-IO, attention or layer-wise legs")
    return ap.parse_args()


def workload_for_rank(name: str, rank: int):
    import tracegen
    w = tracegen.WORKLOADS[name]
    # weak scaling: every rank resolves its own requests (distinct streams per rank)
    return w if rank == 0 else replace(w, seed=w.seed + 7919 * rank)


def kernel_code_digest(path: str) -> str:
    """sha256 of a CUDA source with its comments and whitespace removed: it changes when
    the code changes, not when a comment does."""
    import hashlib
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return hashlib.sha256("".join(text.split()).encode()).hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """ncu figures recorded in profiles/<kernel>_<workload>.md, or None once the kernel
    code has changed since the capture (its digest is recorded beside them)."""
    import re
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "hierarchical_kv_cache_swap_gb300", "csrc", "hs_kernels.cu")
    try:
        text = open(path).read()
        digest = kernel_code_digest(src)
    except OSError:
        return None
    m = re.search(r"```json\n(.*?)```", text, re.S)
    if not m:
        return None
    fig = json.loads(m.group(1))
    return fig if fig.get("kernel_code_sha256") == digest else None


def reduce_max(values, dist, device):
    """Element-wise max of `values` over all ranks (identity without a process group)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def weak_scaling_value(world: int, per_rank_units: int, steps: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * per_rank_units * steps / (max_ms * 1e-3)


def describe(w) -> str:
    extra = f", {w.recent} most recent always selected" if w.recent else ""
    return (f"{w.name}: {w.B} requests x {w.L} layer(s), context {w.C}, {w.S} slots, k={w.k}, "
            f"{w.E}-byte entries, keep {w.keep_pct}%, Zipf({w.zipf_s}) refill{extra}")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.device)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ measurement helpers

def h2d_peak_gbs(torch) -> float:
    """Pinned host -> device cudaMemcpyAsync of 1 GiB, best of 10 (GB/s)."""
    src = torch.empty(H2D_PROBE_BYTES, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(H2D_PROBE_BYTES, dtype=torch.uint8, device="cuda")
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    for _ in range(10):
        s.record()
        dst.copy_(src, non_blocking=True)
        e.record()
        e.synchronize()
        best = max(best, H2D_PROBE_BYTES / (s.elapsed_time(e) * 1e-3) / 1e9)
    del src, dst
    return best


def resolve_hbm_bytes(w, miss) -> float:
    """Algorithmic HBM bytes of the resolution kernel for one step (miss: per-request counts).

    Per request: selections 4k, page-table probes 4k, hit stamps 4h, output 4k, and when
    there are misses a scan of the S last-use stamps 4S, slot-token reads 4m, page-table
    unmap + map 8m, stamps 4m, miss list 8m, the fetch's device copy of the answers 4m,
    plus the counters.
    """
    total = 0
    for m in miss:
        m = int(m)
        h = w.k - m
        b = 12 * w.k + 4 * h + 12
        if m:
            b += 4 * w.S + 28 * m
        total += b
    return float(total)


def bench_config(w, W: int, K: int) -> dict:
    """The `config` dict of both arms' lines (identical for the same workload and steps)."""
    return {"workload": describe(w), "per_rank_requests": w.B,
            "trace_steps": f"{W} warm-up + {K} timed (of one seeded trace)",
            "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB write); "
                  "the page table and slot buffer exceed L2 on this workload" if w.B * w.C * 4 > (129 << 20)
                  else f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB write)",
            "timing": "CUDA events around each hs_resolve call, summed (CPU arm: wall clock)"}


# ------------------------------------------------------------------ reference arm (CPU oracle)

def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    import tracegen
    import oracle
    tracegen.build()
    oracle.build()
    w = (tracegen.noio_workload(4096) if args.workload == "noio"
         else tracegen.WORKLOADS["dsa" if args.workload == "attend" else args.workload])
    T = args.warmup + args.steps
    cores = host_cores()
    value, dt = oracle_rate(w, T, args.warmup, cores)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": bench_config(w, args.warmup, args.steps),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"whole workload, steps {args.warmup}..{T - 1}, all {w.B} requests, "
                                   f"the single-threaded C oracle per request on {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def timed_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W: int, K: int, reset: bool = True) -> list:
    """(hs_reset,) the W warm-up steps, then K steps each bracketed by CUDA events with an
    L2 flush before it; returns the K step times in ms."""
    stream = torch.cuda.current_stream()
    if reset:
        ctx.reset()
    for t in range(W):
        ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        t = W + i
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def profiled_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W: int, K: int):
    """The same steps with events between the two kernels (which then run one after the
    other), so that each kernel's own duration is measured: (resolution ms, fetch ms)."""
    ctx.reset()
    for t in range(W):
        ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
    torch.cuda.synchronize()
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        t = W + i
        flush.fill_(i & 0xFF)
        ctx.resolve_profiled(sel_dev[t], out_dev[t], miss_dev[t], pev[i])
    torch.cuda.synchronize()
    return [e[0].elapsed_time(e[1]) for e in pev], [e[1].elapsed_time(e[2]) for e in pev]


def load_peaks() -> dict:
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return {}


def step_figures(w, step_ms, res_ms, gat_ms, miss, peak_h2d: float, K: int) -> dict:
    """Per-step and per-kernel figures of one workload's timed steps (miss: [K][B] counts).
    The kernels' own durations come from the serialised pass (hs_resolve_profiled)."""
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    hbm_src = "MEASURED_PEAKS.json hbm_gbs (of measured)" if "hbm_gbs" in peaks else "fallback 6.8 TB/s"
    total_ms, res_total, gat_total = sum(step_ms), sum(res_ms), sum(gat_ms)
    miss_bytes = float(miss.sum()) * w.E
    res_bytes = sum(resolve_hbm_bytes(w, miss[i]) for i in range(K))
    fetch_step = miss_bytes / (total_ms * 1e-3) / 1e9
    fetch_kernel = miss_bytes / (gat_total * 1e-3) / 1e9 if gat_total > 0 else None
    return {
        "us_per_layer_step": total_ms / K * 1e3,
        "us_per_layer_step_median": statistics.median(step_ms) * 1e3,
        "resolutions_per_s": w.B * K / (total_ms * 1e-3),
        "misses_per_step": float(miss.sum()) / K,
        "miss_bytes_per_step": miss_bytes / K,
        "miss_fetch_gbs": fetch_step,
        "miss_fetch_frac_of_h2d_peak": fetch_step / peak_h2d,
        "kernels": {
            "gather_kernel": {"launches": K, "us_avg": gat_total / K * 1e3,
                              "link_bytes_per_launch": miss_bytes / K, "link_gbs": fetch_kernel,
                              "link_frac_of_h2d_peak": fetch_kernel / peak_h2d if fetch_kernel else None,
                              "share_of_serialized_time": gat_total / (gat_total + res_total)},
            "resolve_kernel": {"launches": K, "us_avg": res_total / K * 1e3,
                               "hbm_bytes_per_launch": res_bytes / K,
                               "hbm_gbs": res_bytes / (res_total * 1e-3) / 1e9,
                               "hbm_frac": res_bytes / (res_total * 1e-3) / 1e9 / hbm_peak,
                               "hbm_peak_source": hbm_src},
            "overlap_saving_us_per_step": (res_total + gat_total - total_ms) / K * 1e3,
            "how": "each kernel's duration from the serialised pass (hs_resolve_profiled: events "
                   "before, between and after the two kernels)",
        },
    }


def roofline_of(w, fig: dict, peak_h2d: float) -> dict:
    """The roofline line of the dominant kernel (the longer of the two in the serialised pass)."""
    g, r = fig["kernels"]["gather_kernel"], fig["kernels"]["resolve_kernel"]
    if g["us_avg"] >= r["us_avg"]:
        prof = profiled_traffic("gather_kernel", w.name)
        per_launch = g["link_bytes_per_launch"]
        return {"bound": "h2d_link", "kernel": "gather_kernel", "achieved": g["link_gbs"], "peak": peak_h2d,
                "unit": "GB/s", "frac": g["link_gbs"] / peak_h2d,
                "traffic": prof and prof["dram_bytes_per_algorithmic_link_byte"] * per_launch,
                "link_traffic": prof and prof["link_bytes_per_algorithmic_link_byte"] * per_launch,
                "algorithmic_bytes_per_launch": per_launch,
                "traffic_source": f"profiles/gather_kernel_{w.name}.md (ncu, scaled to this run's mean misses)"
                if prof else None,
                "peak_source": "pinned cudaMemcpyAsync host->device, 1 GiB, best of 10, this run"}
    return {"bound": "hbm", "kernel": "resolve_kernel", "achieved": r["hbm_gbs"],
            "peak": r["hbm_gbs"] / r["hbm_frac"], "unit": "GB/s", "frac": r["hbm_frac"], "traffic": None,
            "peak_source": r["hbm_peak_source"]}


def run_ours(args, rank: int, world: int, dist) -> None:
    import numpy as np
    import torch

    import __graft_entry__
    import hierarchical_kv_cache_swap_gb300 as hs
    import tracegen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
        __graft_entry__.build()

    w = workload_for_rank(args.workload, rank)
    K, W = args.steps, args.warmup
    T = W + K
    sel = tracegen.trace(w, T=T)
    sel_dev = torch.from_numpy(sel).cuda()
    out_dev = torch.empty_like(sel_dev)
    miss_dev = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    ctx = hs.Context(w.B, w.C, w.S, w.E)
    create_s = time.perf_counter() - t0
    t0 = time.perf_counter()
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w)
    fill_s = time.perf_counter() - t0
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peak_h2d = h2d_peak_gbs(torch)

    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.3)
        # ---- pass 0: the first pass over the trace after the store was created and
        # filled: the GPU reads most of these host pages for the first time
        first_ms = timed_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K, reset=False)
        first_miss = miss_dev[W:].cpu().numpy()

        # ---- pass 1: the step as users run it (resolution -> fetch chained by PDL), the
        # same steps again from an empty cache: the steady state, the headline
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        step_ms = timed_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K)
        wall = time.perf_counter() - wall0
        status = ctx.status()
        miss = miss_dev[W:].cpu().numpy()
        assert np.array_equal(miss, first_miss), "the two passes resolved differently"

        # ---- pass 2: per-kernel durations (the kernels run one after the other)
        res_ms, gat_ms = profiled_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K)
        kpc = ctx.kernels_per_call()

        # ---- pass 3: end to end through the host-buffer entry point (pinned in/out)
        ctx.reset()
        for t in range(W):
            ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
        torch.cuda.synchronize()
        sel_pin = torch.from_numpy(sel).pin_memory()
        out_pin = torch.empty((w.B, w.k), dtype=torch.int32).pin_memory()
        miss_pin = torch.empty(w.B, dtype=torch.int32).pin_memory()
        sel_np, out_np, miss_np = sel_pin.numpy(), out_pin.numpy(), miss_pin.numpy()
        e2e_s = 0.0
        for i in range(K):
            t = W + i
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            ctx.resolve_host(sel_np[t], out_np, miss_np)
            e2e_s += time.perf_counter() - t0

        extras = {}
        if not args.no_extras and rank == 0:
            extras["cpu_baseline"] = cpu_baseline(w, T=max(T, 16), W=W, host=ctx.host_kv_address(),
                                                  stride=ctx.host_stride)
    clocks = sampler.summary()
    if not args.no_extras and rank == 0:
        ctx.close()  # the extras need the host memory
        ctx = None
        with ClockSampler(local) as extra_sampler:
            if w.name != "dsa":
                extras["dsa"] = measure_dsa(torch, hs, tracegen, flush, peak_h2d, W, K)
            extras["no_io"] = measure_noio(torch, hs, tracegen, flush)
            extras["sweep"] = measure_sweep(torch, hs, tracegen, flush, peak_h2d)
            extras["quest_layerwise"] = layerwise(torch, hs, tracegen, tracegen.WORKLOADS["quest"],
                                                  W=4, K=16, rank=0, flush=flush, peak_h2d=peak_h2d)
        extras["clocks_extras"] = extra_sampler.summary()
    if ctx is not None:
        ctx.close()

    total_ms, e2e_s = reduce_max([sum(step_ms), e2e_s], dist if world > 1 else None, "cuda")
    if rank != 0:
        return

    fig = step_figures(w, step_ms, res_ms, gat_ms, miss, peak_h2d, K)
    value = weak_scaling_value(world, w.B, K, total_ms)
    roofline = roofline_of(w, fig, peak_h2d)
    first = {"us_per_layer_step": sum(first_ms) / K * 1e3,
             "us_first_step": first_ms[0] * 1e3, "us_max_step": max(first_ms) * 1e3,
             "ratio_to_steady_state": sum(first_ms) / sum(step_ms),
             "how": "the same W warm-up + K timed steps run once right after hs_create and the host fill, "
                    "before the headline pass (which repeats them from an empty cache)",
             "hs_create_s": create_s, "host_fill_s": fill_s}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32", "data": "synthetic",
        "config": bench_config(w, W, K),
        "positions_per_s": value * w.k,
        "h2d_peak_gbs": peak_h2d,
        **fig,
        "first_pass_after_create": first,
        "roofline": roofline,
        "gpu_launches": K * kpc,
        "device_status": status,
        "clocks": clocks,
        "e2e": {"value": weak_scaling_value(world, w.B, K, e2e_s * 1e3), "unit": UNIT,
                "h2d_bytes_per_step": w.B * w.k * 4, "d2h_bytes_per_step": w.B * w.k * 4 + w.B * 4,
                "how": "hs_resolve_host with page-locked buffers: the kernels read the selections and "
                       "write out_slots + miss_counts in host memory in place; stream sync"},
        "wall_s_timed_region": wall,
    }
    line.update({k: v for k, v in extras.items()})
    dsa = extras.get("dsa") or (fig if w.name == "dsa" else None)
    noio = extras.get("no_io")
    quest = extras.get("quest_layerwise")
    g = fig["kernels"]["gather_kernel"]
    line["gates"] = {
        "fetch_kernel_link_frac": g["link_frac_of_h2d_peak"],
        "step_link_frac": fig["miss_fetch_frac_of_h2d_peak"],
        "dsa_fetch_kernel_link_frac": dsa and dsa["kernels"]["gather_kernel"]["link_frac_of_h2d_peak"],
        "dsa_step_link_frac": dsa and dsa["miss_fetch_frac_of_h2d_peak"],
        "link_target": 0.8,
        "no_io_us_per_layer_step_graph": noio and noio["us_per_layer_step_graph"],
        "no_io_target_us": 5.0,
        "quest_hidden_fraction": quest and quest["hidden_fraction_of_miss_overhead"],
    }
    print(json.dumps(line), flush=True)


def measure_dsa(torch, hs, tracegen, flush, peak_h2d: float, W: int, K: int) -> dict:
    """The DSA-style decode workload (32 requests, context 32768, 4096 slots, k = 2048):
    the same passes as the headline, plus its CUDA graph, pooled-context, policy,
    attention and append figures."""
    w = tracegen.WORKLOADS["dsa"]
    T = W + K
    sel = tracegen.trace(w, T=T)
    sel_dev = torch.from_numpy(sel).cuda()
    out_dev = torch.empty_like(sel_dev)
    miss_dev = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
    ctx = hs.Context(w.B, w.C, w.S, w.E)
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w)
    timed_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K, reset=False)  # first touch
    step_ms = timed_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K)
    miss = miss_dev[W:].cpu().numpy()
    res_ms, gat_ms = profiled_steps(torch, ctx, sel_dev, out_dev, miss_dev, flush, W, K)
    fig = step_figures(w, step_ms, res_ms, gat_ms, miss, peak_h2d, K)
    fig["workload"] = describe(w)
    fig["roofline"] = roofline_of(w, fig, peak_h2d)
    fig["graph"] = measure_graph(torch, ctx, w, sel_dev, out_dev, miss_dev, W, K)
    fig["pooled"] = measure_pooled(torch, hs, ctx, w, sel_dev, out_dev, miss_dev, flush, W, K)
    fig["policies"] = measure_policies(torch, hs, ctx, w, sel_dev, out_dev, miss_dev, flush, W, K)
    fig["attend"] = measure_attend(torch, ctx, w, out_dev[W + K - 1], flush)
    fig["append"] = measure_append(torch, ctx, w, flush, K)
    fig["device_status"] = ctx.status()
    ctx.close()
    return fig


def layerwise(torch, hs, tracegen, w, W: int, K: int, rank: int, flush, peak_h2d: float) -> dict:
    """w.L layers sharing one selection per step: the two-stream overlap of layer l+1's
    resolution with layer l's consumer, against the serial order and against the serial
    order without fetches (the miss overhead). The consumer is the sparse attention
    (hs_attend, 128 heads) for 656-byte DSA entries, else the checksum stand-in. The
    layers' contexts share one host store (timing only: bytes are opaque to the method)."""
    T = W + K
    B, L = w.B, w.L
    sel = torch.from_numpy(tracegen.trace(w, T=T)).cuda()
    lender = hs.Context(B, w.C, w.S, w.E)
    tracegen.fill_kv(lender.host_kv_address(), lender.host_stride, w)
    ctxs = [lender] + [hs.Context(B, w.C, w.S, w.E, share_host_with=lender) for _ in range(L - 1)]
    out = torch.empty((L, B, w.k), dtype=torch.int32, device="cuda")
    miss = torch.empty((T, L, B), dtype=torch.int32, device="cuda")
    sums = torch.empty((L, B), dtype=torch.int64, device="cuda")
    attention = w.E == 656
    if attention:
        H = ATTEND_HEADS
        g = torch.Generator(device="cuda").manual_seed(21)
        qs = [torch.randn((B, H, 576), generator=g, device="cuda").to(torch.bfloat16) for _ in range(L)]
        o_l = torch.empty((L, B, H, 512), dtype=torch.float32, device="cuda")
        lse_l = torch.empty((L, B, H), dtype=torch.float32, device="cuda")
        nbytes = ctxs[0].attend_workspace(B, H, w.k)
        wss = [torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") for _ in range(L)]

    def consume(layer, stream):
        if attention:
            ctxs[layer].attend(qs[layer], out[layer], o_l[layer], lse_l[layer], ATTEND_SCALE,
                               workspace=wss[layer] if nbytes else None, stream=stream)
        else:
            ctxs[layer].checksum_rows(out[layer], sums[layer], stream=stream)

    s_res, s_use = torch.cuda.Stream(), torch.cuda.Stream()

    def run(mode):
        for c in ctxs:
            c.reset()
            c.set_flags(hs.HS_FLAG_NO_COPY if mode == "serial_no_fetch" else 0)
        torch.cuda.synchronize()
        times = []
        for t in range(T):
            timed = t >= W
            flush.fill_(t & 0xFF)
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_res.wait_stream(torch.cuda.current_stream())
            s_use.wait_stream(torch.cuda.current_stream())
            a.record(s_res)
            for layer in range(L):
                ctxs[layer].resolve(sel[t], out[layer], miss[t, layer], stream=s_res)
                if mode == "overlap":
                    ev = torch.cuda.Event()
                    ev.record(s_res)
                    s_use.wait_event(ev)
                    consume(layer, s_use)
                else:
                    consume(layer, s_res)
            if mode == "overlap":
                s_res.wait_stream(s_use)
            z.record(s_res)
            torch.cuda.current_stream().wait_stream(s_res)
            if timed:
                times.append((a, z))
        torch.cuda.synchronize()
        return [x.elapsed_time(y) * 1e3 for x, y in times]

    run("serial")  # first touch of the host pages, untimed
    res = {m: run(m) for m in ("serial", "overlap", "serial_no_fetch")}
    status = lender.status()
    miss_rows = float(miss[W:].sum())
    for c in reversed(ctxs):
        c.set_flags(0)
        c.close()
    med = {m: statistics.median(v) for m, v in res.items()}
    tot = {m: sum(v) for m, v in res.items()}
    overhead = tot["serial"] - tot["serial_no_fetch"]
    return {
        "workload": describe(w) + f"; one selection shared by the {L} layers; the layers' contexts share "
                    "one host store (timing only)",
        "steps": K, "warmup": W,
        "us_per_step": {m: tot[m] / K for m in tot}, "us_per_step_median": med,
        "us_per_layer_step_overlapped": tot["overlap"] / K / L,
        "miss_overhead_us_per_step": overhead / K,
        "hidden_fraction_of_miss_overhead": (tot["serial"] - tot["overlap"]) / overhead if overhead > 0 else None,
        "miss_bytes_per_step": miss_rows * w.E / K,
        "miss_fetch_gbs_overlapped": miss_rows * w.E / (tot["overlap"] * 1e-6) / 1e9,
        "h2d_peak_gbs": peak_h2d,
        "consumer": (f"hs_attend: sparse MLA-style attention, {ATTEND_HEADS} heads, bf16 tensor-core "
                     "products" if attention else "hs_checksum_rows (reads every resolved row)"),
        "consumer_bytes_per_step": B * L * w.k * w.E,
        "consumer_flops_per_step": (2 * B * L * ATTEND_HEADS * w.k * (576 + 512)) if attention else None,
        "device_status": status,
    }


def run_layers(args, rank: int, world: int, dist) -> None:
    """The layer-wise overlap workloads (quest, dsa_layers) as the headline line."""
    import torch

    import __graft_entry__
    import hierarchical_kv_cache_swap_gb300 as hs
    import tracegen

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    __graft_entry__.build()
    w = workload_for_rank(args.workload, rank)
    K, W = args.steps, args.warmup
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peak_h2d = h2d_peak_gbs(torch)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as sampler:
        lw = layerwise(torch, hs, tracegen, w, W, K, rank, flush, peak_h2d)
    us_step = lw["us_per_step"]["overlap"]
    value = weak_scaling_value(world, w.B * w.L, K, us_step * K / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT + " (request-layer)", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": us_step / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": bench_config(w, W, K),
        "layerwise_prefetch": lw, "clocks": sampler.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


POLICIES = (("lru", 0), ("fifo", 1), ("random", 2))
POLICY_SEED = 0x5EED


def measure_policies(torch, hs, ctx, w, sel_dev, out_dev, miss_dev, flush, W: int, K: int) -> dict:
    """The timed steps again under each replacement policy (L2 flushed between steps,
    like the main pass), then the misses per step over buffer sizes S on the same
    trace (bookkeeping only: HS_FLAG_NO_COPY, the first, cold call left out)."""
    stream = torch.cuda.current_stream()
    step = {}
    for name, pol in POLICIES:
        ctx.set_policy(pol, POLICY_SEED)
        ctx.reset()
        for t in range(W):
            ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            ctx.resolve(sel_dev[W + i], out_dev[W + i], miss_dev[W + i])
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        us = [a.elapsed_time(b) * 1e3 for a, b in ev]
        step[name] = {"us_per_layer_step": statistics.mean(us), "us_median": statistics.median(us),
                      "misses_per_step": float(miss_dev[W:].sum()) / K}
    ctx.set_policy(0)
    T = min(W + K, 128)
    curve = {}
    for S in (w.k, w.k * 3 // 2, 2 * w.k, 3 * w.k, 4 * w.k):
        c = hs.Context(w.B, w.C, S, w.E, share_host_with=ctx)
        c.set_flags(hs.HS_FLAG_NO_COPY)
        m = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
        row = {}
        for name, pol in POLICIES:
            c.set_policy(pol, POLICY_SEED)
            c.reset()
            for t in range(T):
                c.resolve(sel_dev[t], out_dev[t], m[t])
            torch.cuda.synchronize()
            row[name] = float(m[1:].sum()) / (T - 1)
        c.close()
        curve[str(S)] = row
    return {"step": step, "misses_per_step_by_slots": curve, "trace_steps_for_curve": T,
            "seed": POLICY_SEED}


def measure_graph(torch, ctx, w, sel_dev, out_dev, miss_dev, W: int, K: int) -> dict:
    """Steps W..W+K-1 captured in one CUDA graph after the W warm-up steps and replayed once:
    µs per layer-step as a decode graph sees it (no flush between steps; every step is a
    distinct selection, so the state advances as it does eagerly)."""
    ctx.reset()
    for t in range(W):
        ctx.resolve(sel_dev[t], out_dev[t], miss_dev[t])
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(K):
                ctx.resolve(sel_dev[W + i], out_dev[W + i], miss_dev[W + i], stream=s)
    torch.cuda.current_stream().wait_stream(s)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    us = a.elapsed_time(b) * 1e3 / K
    misses = float(miss_dev[W:W + K].sum()) / K
    return {"us_per_layer_step": us, "resolutions_per_s": w.B / (us * 1e-6), "steps": K,
            "misses_per_step": misses, "miss_fetch_gbs": misses * w.E / (us * 1e-6) / 1e9,
            "how": "one replay of a graph holding the K timed steps, after the W warm-up steps eagerly"}


def measure_pooled(torch, hs, ctx, w, sel_dev, out_dev, miss_dev, flush, W: int, K: int) -> dict:
    """The timed steps through hs_create_pooled over the main context's host store seen as a
    pool of B * C rows, request b at the extent of request (7b + 3) mod B, every length C."""
    rows = w.B * w.C
    pc = hs.Context(w.B, w.C, w.S, w.E, pool=(ctx.host_kv_address(), rows, ctx.host_stride))
    pc.set_extents([((7 * b + 3) % w.B) * w.C for b in range(w.B)], [w.C] * w.B)
    stream = torch.cuda.current_stream()
    for t in range(W):
        pc.resolve(sel_dev[t], out_dev[t], miss_dev[t])
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        pc.resolve(sel_dev[W + i], out_dev[W + i], miss_dev[W + i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    status = pc.status()
    pc.close()
    return {"us_per_layer_step": statistics.mean(us), "us_median": statistics.median(us),
            "misses_per_step": float(miss_dev[W:].sum()) / K, "device_status": status,
            "how": "hs_create_pooled over the same pinned store, extents permuted across requests"}


def measure_attend(torch, ctx, w, out_slots, flush, n: int = 32) -> dict:
    """hs_attend over one step's resolved slots: 128 heads of bf16 queries, L2 flushed
    between calls; achieved = algorithmic FLOPs (2 H k (576 + 512) per request) / time."""
    H = ATTEND_HEADS
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((w.B, H, 576), generator=g, device="cuda").to(torch.bfloat16)
    o = torch.empty((w.B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, H), dtype=torch.float32, device="cuda")
    nbytes = ctx.attend_workspace(w.B, H, w.k)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    ctx.clear_status()
    for _ in range(3):
        ctx.attend(q, out_slots, o, lse, ATTEND_SCALE, workspace=ws)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        ctx.attend(q, out_slots, o, lse, ATTEND_SCALE, workspace=ws)
        evs[i][1].record()
    torch.cuda.synchronize()
    assert ctx.status() == 0
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    flops = 2.0 * w.B * H * w.k * (576 + 512)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        pass
    peak = peaks.get("bf16_tflops", 1900.0)
    tf = flops / (statistics.mean(us) * 1e-6) / 1e12
    return {"calls": n, "heads": H, "k": w.k, "requests": w.B, "us_per_call": statistics.mean(us),
            "us_per_call_median": statistics.median(us), "algorithmic_flops_per_call": flops,
            "kv_bytes_per_call": w.B * w.k * w.E,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_source": "MEASURED_PEAKS.json bf16_tflops (of measured)" if "bf16_tflops" in peaks
                         else "fallback 1.9 PFLOP/s"}}


def measure_append(torch, ctx, w, flush, n: int) -> dict:
    """hs_append of one E-byte row per request per call at uniform random positions
    (those that are resident, about S / C of them, also write their slot), L2 flushed
    between calls."""
    g = torch.Generator().manual_seed(11)
    pos = torch.randint(0, w.C, (n, w.B), generator=g, dtype=torch.int32).cuda()
    rows = torch.randint(0, 256, (n, w.B, w.E), generator=g, dtype=torch.uint8).cuda()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    ctx.clear_status()
    for i in range(n):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        ctx.append(rows[i], pos[i])
        evs[i][1].record()
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    assert ctx.status() == 0
    link = w.B * w.E
    return {"calls": n, "rows_per_call": w.B, "link_bytes_per_call": link,
            "us_per_call": statistics.mean(us), "us_per_call_median": statistics.median(us),
            "link_gbs": link / (statistics.mean(us) * 1e-6) / 1e9}


def measure_sweep(torch, hs, tracegen, flush, peak_h2d: float, W: int = 8, K: int = 16) -> dict:
    """The buffer/locality sweep: 64 requests, context 65536, k = 2048, S in {2048, 4096,
    6144} x keep in {50, 80, 95} %. Per point: misses per step and µs per layer-step with
    the fetch (L2 flushed before each call) and without it (HS_FLAG_NO_COPY: the
    bookkeeping alone, at that point's miss rate). The nine points share one host store
    (its bytes depend only on the workload's seed)."""
    lender = None
    out = {}
    ctxs = {}
    try:
        for S in (2048, 4096, 6144):
            w0 = tracegen.sweep_workload(S, 50)
            if lender is None:
                lender = hs.Context(w0.B, w0.C, S, w0.E)
                tracegen.fill_kv(lender.host_kv_address(), lender.host_stride, w0)
                ctxs[S] = lender
            else:
                ctxs[S] = hs.Context(w0.B, w0.C, S, w0.E, share_host_with=lender)
        stream = torch.cuda.current_stream()
        for keep in (50, 80, 95):
            for S in (2048, 4096, 6144):
                w = tracegen.sweep_workload(S, keep)
                T = W + K
                sd = torch.from_numpy(tracegen.trace(w, T=T)).cuda()
                o = torch.empty_like(sd)
                m = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
                ctx = ctxs[S]
                row = {}
                for mode, flags in (("fetch", 0), ("bookkeeping_only", hs.HS_FLAG_NO_COPY)):
                    ctx.set_flags(flags)
                    ctx.reset()
                    for t in range(W):
                        ctx.resolve(sd[t], o[t], m[t])
                    torch.cuda.synchronize()
                    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                          for _ in range(K)]
                    for i in range(K):
                        flush.fill_(i & 0xFF)
                        ev[i][0].record(stream)
                        ctx.resolve(sd[W + i], o[W + i], m[W + i])
                        ev[i][1].record(stream)
                    torch.cuda.synchronize()
                    row[mode] = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev)
                ctx.set_flags(0)
                misses = float(m[W:].sum()) / K
                out[f"S{S}_keep{keep}"] = {
                    "us_per_layer_step": row["fetch"], "us_per_layer_step_bookkeeping_only": row["bookkeeping_only"],
                    "misses_per_step": misses, "resolutions_per_s": w.B / (row["fetch"] * 1e-6),
                    "miss_fetch_frac_of_h2d_peak": misses * w.E / (row["fetch"] * 1e-6) / 1e9 / peak_h2d}
        status = 0
        for c in ctxs.values():
            status |= c.status()
    finally:
        for S in (6144, 4096, 2048):
            if S in ctxs:
                ctxs[S].close()
    return {"points": out, "steps": K, "warmup": W, "device_status": status,
            "workload": "64 requests x 1 layer, context 65536, k=2048, 656-byte entries, Zipf(1.1) refill, seed 2",
            "how": "per point: W warm-up + K timed steps from an empty cache, L2 flushed before each call; "
                   "then the same with HS_FLAG_NO_COPY"}


def run_attend(args, rank: int, world: int, dist) -> None:
    """The attention consumer as the headline: the DSA-style workload's resolved slots of one
    step (32 requests x k = 2048), 128 heads, L2 flushed before each call."""
    import torch

    import __graft_entry__
    import hierarchical_kv_cache_swap_gb300 as hs
    import tracegen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    w = tracegen.WORKLOADS["dsa"]
    T = 4
    sd = torch.from_numpy(tracegen.trace(w, T=T)).cuda()
    out = torch.empty_like(sd)
    miss = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
    ctx = hs.Context(w.B, w.C, w.S, w.E)
    if args.wait_limit_ms:
        ctx.set_wait_limit(int(args.wait_limit_ms * 1e6))
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w)
    for t in range(T):
        ctx.resolve(sd[t], out[t], miss[t])
    torch.cuda.synchronize()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    with ClockSampler(local) as sampler:
        att = measure_attend(torch, ctx, w, out[T - 1], flush, n=args.steps)
    ctx.close()
    us = att["us_per_call"]
    line = {
        "metric": METRIC, "value": weak_scaling_value(world, w.B, 1, us * 1e-3), "unit": UNIT + " (attention calls)",
        "n_gpus": world, "steps": args.steps, "warmup": 3, "ms_per_step": us * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(w) + f"; attention over one step's resolved slots, {ATTEND_HEADS} heads",
                   "l2": f"flushed before each call ({FLUSH_BYTES >> 20} MiB write)",
                   "timing": "CUDA events around each hs_attend call"},
        "attend": att, "roofline": att["roofline"], "clocks": sampler.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_noio(args, rank: int, world: int, dist) -> None:
    """The no-IO gate as the headline: 64 requests x k = 2048 over 4096 slots, every call all
    hits, back to back in a CUDA graph (and, apart, each call after an L2 flush)."""
    import torch

    import __graft_entry__
    import hierarchical_kv_cache_swap_gb300 as hs
    import tracegen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    with ClockSampler(local) as sampler:
        noio = measure_noio(torch, hs, tracegen, flush, N=args.steps)
    us = noio["us_per_layer_step_graph"]
    w = tracegen.noio_workload(4096)
    us_all = reduce_max([us], dist if world > 1 else None, "cuda")[0]
    line = {
        "metric": METRIC, "value": weak_scaling_value(world, w.B, 1, us_all * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": 1, "ms_per_step": us_all * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": noio["workload"],
                   "l2": "warm: back to back in one CUDA graph, as a decode graph runs them "
                         f"(the flushed figure is in no_io: {FLUSH_BYTES >> 20} MiB write before each call)",
                   "timing": "CUDA events around one replay of a graph of the timed calls"},
        "no_io": noio, "clocks": sampler.summary(),
        "gates": {"no_io_us_per_layer_step_graph": us, "no_io_target_us": 5.0},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_noio(torch, hs, tracegen, flush, N: int = 64) -> dict:
    w = tracegen.noio_workload(4096)
    sel = tracegen.trace(w, T=N + 1)
    sd = torch.from_numpy(sel).cuda()
    out = torch.empty_like(sd)
    miss = torch.empty((N + 1, w.B), dtype=torch.int32, device="cuda")
    ctx = hs.Context(w.B, w.C, w.S, w.E)
    ctx.resolve(sd[0], out[0], miss[0])  # cold call: every selection misses
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(N)]
    for i in range(N):
        flush.fill_(i & 0xFF)
        evs[i][0].record()
        ctx.resolve(sd[i + 1], out[i + 1], miss[i + 1])
        evs[i][1].record()
    torch.cuda.synchronize()
    flushed = [a.elapsed_time(b) * 1e3 for a, b in evs]
    assert int(miss[1:].sum()) == 0, "no-IO trace produced misses"
    # back to back inside one CUDA graph (warm L2), as in a decode graph
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(N):
                ctx.resolve(sd[i + 1], out[i + 1], miss[i + 1], stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    graph_us = a.elapsed_time(b) * 1e3 / N
    ctx.close()
    return {"workload": describe(w) + "; every call re-selects step 0's set (all hits)",
            "us_per_layer_step_flushed": statistics.mean(flushed),
            "us_per_layer_step_flushed_median": statistics.median(flushed),
            "us_per_layer_step_graph": graph_us, "calls": N}


def oracle_rate(w, T: int, W: int, threads: int, host: int | None = None, stride: int | None = None,
                B: int | None = None):
    """The CPU oracle over steps W..T-1 of the workload's trace, every request resolved by
    the same single-threaded C function; with threads > 1 the requests are split among
    that many threads (requests are independent; the C call releases the GIL). `host` /
    `stride`: the address and row stride of a [B][C][stride] store already holding the
    history (the GPU context's pinned store), else a new array is filled. `B`: only the
    first B requests. Returns (resolutions/s, seconds)."""
    import tracegen
    from concurrent.futures import ThreadPoolExecutor
    from oracle import Oracle
    B = w.B if B is None else B
    sel = tracegen.trace(w, T=T, B=B)
    keep = None
    if host is None:
        keep = host_array(B * w.C * w.E)
        tracegen.fill_kv(keep.ctypes.data, w.E, w, B=B)
        host, stride = keep.ctypes.data, w.E
    o = Oracle(B, w.C, w.S, w.E)
    row = w.C * stride

    def run(requests, t0, t1):
        for t in range(t0, t1):
            for b in requests:
                o.resolve_request(b, host + b * row, stride, sel[t, b])

    groups = [list(range(i, B, threads)) for i in range(min(threads, B))]
    with ThreadPoolExecutor(len(groups)) as ex:
        list(ex.map(lambda g: run(g, 0, W), groups))
        t0 = time.perf_counter()
        list(ex.map(lambda g: run(g, W, T), groups))
        dt = time.perf_counter() - t0
    del keep
    return B * (T - W) / dt, dt


def host_array(nbytes: int):
    """A zeroed uint8 array for a host KV store, backed by transparent huge pages where
    the kernel offers them (a 22 GB store is 5.4 M faults with 4 KiB pages)."""
    import mmap
    import numpy as np
    m = mmap.mmap(-1, max(nbytes, 1))
    if hasattr(mmap, "MADV_HUGEPAGE"):
        try:
            m.madvise(mmap.MADV_HUGEPAGE)
        except OSError:
            pass
    return np.frombuffer(m, dtype=np.uint8, count=nbytes)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(w, T: int, W: int, host: int | None = None, stride: int | None = None,
                 min_cpu_s: float = 10.0, max_reps: int = 6) -> dict:
    """The CPU oracle on this host's cores (one thread per core, requests split among them)
    over steps W..T-1 of the same workload's trace, repeated from a fresh oracle until the
    timed part holds at least `min_cpu_s` seconds of CPU work (at most `max_reps` times);
    and on one core over up to 32 of those steps for a quarter of the requests (at least
    one)."""
    cores = host_cores()
    n, secs, reps = 0, 0.0, 0
    while reps < max_reps and (reps == 0 or secs * cores < min_cpu_s):
        rate, dt = oracle_rate(w, T, W, cores, host, stride)
        n += round(rate * dt)
        secs += dt
        reps += 1
    b1 = max(1, w.B // 4)
    t1 = min(T, W + 32)
    one, dt1 = oracle_rate(w, t1, W, 1, host, stride, B=b1)
    return {"value": n / secs, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "single_core_value": one, "seconds": secs, "single_core_seconds": dt1,
            "sample": f"steps {W}..{T - 1} (after {W} untimed) x all {w.B} requests of the same workload "
                      f"over the GPU context's pinned store, {reps} time(s) from a fresh oracle, the "
                      f"single-threaded C oracle per request on {cores} threads ({secs * cores:.1f} s of CPU "
                      f"work); single core: {t1 - W} steps x {b1} requests"}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.workload in ("quest", "dsa_layers"):
            run_layers(args, rank, world, dist)
        elif args.workload == "noio":
            run_noio(args, rank, world, dist)
        elif args.workload == "attend":
            run_attend(args, rank, world, dist)
        else:
            run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
