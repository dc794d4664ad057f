#!/usr/bin/env python
"""Benchmark of the relative-position attention forward path on GB300.

One step = one forward pass of the hot path over one batch of synthetic input:
at the headline workload (iRPE contextual-K attention at the DeiT-S shape,
B=64, 6 heads, 14x14 grid, d=64, bf16) that is one rpe_attn_fwd launch, which
derives bucket ids from the offset table, forms QR = Q R^K^T, QK^T, the
softmax and PV in one fused kernel. The offset table is built once outside
the timed region (the iRPE page: ids are computed once per grid and reused).

Timing: W warm-up steps, then exactly K steps captured in CUDA graphs and
timed with CUDA events on the launching stream, bracketed by a barrier and a
device synchronisation. Inputs rotate over enough copies to exceed 3x the L2
size, so no step finds its inputs in L2 (no flush is needed). Throughput is
query tokens per second (B*N per step, heads not multiplied in).

Prints one JSON line. ``--impl reference`` instead times the oracle (the CPU
reference of this path) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "RPE-attention fwd tokens/s and TFLOP/s (% of bf16 TC peak) at DeiT-S iRPE-K, 1 GB300"
HEADLINE = "irpe_k_deit_s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 * 1024 * 1024


# ---------------------------------------------------------------- workload arithmetic

def work_of(cfg):
    """(algorithmic flops, algorithmic bytes, query tokens) of one step of cfg."""
    from vision_transformer_attention_gb300.workloads import SwinConfig
    if isinstance(cfg, SwinConfig):
        units = cfg.num_windows * cfg.heads
        flops = units * 4.0 * cfg.n ** 2 * cfg.d
        elem = 2 if cfg.dtype == "bf16" else 4
        nbytes = 4.0 * units * cfg.n * cfg.d * elem
        return flops, nbytes, cfg.num_windows * cfg.n
    S = cfg.B * cfg.heads
    nterms = bin(cfg.flags).count("1")
    flops = S * (4.0 * cfg.N ** 2 * cfg.d + nterms * 2.0 * cfg.N * cfg.num_buckets * cfg.d)
    nbytes = 4.0 * S * cfg.N * cfg.d * 2
    return flops, nbytes, cfg.B * cfg.N


def workload_config(cfg):
    from vision_transformer_attention_gb300.workloads import SwinConfig
    if isinstance(cfg, SwinConfig):
        out = {"workload": cfg.name, "num_windows": cfg.num_windows, "heads": cfg.heads,
               "window": cfg.M, "n": cfg.n, "d": cfg.d}
        if cfg.fmap:
            out["feature_map"] = list(cfg.fmap) + [cfg.heads * cfg.d]
        return out
    terms = "".join(t for t, f in (("Q", 2), ("K", 1), ("V", 4)) if cfg.flags & f)
    return {"workload": cfg.name, "B": cfg.B, "heads": cfg.heads, "grid": [cfg.H, cfg.W],
            "N": cfg.N, "d": cfg.d, "terms": terms or "none", "num_buckets": cfg.num_buckets,
            "cls_token": cfg.cls,
            "index_fn": {"alpha": cfg.ratio, "beta": 2 * cfg.ratio, "gamma": 8 * cfg.ratio}}


# The kernel that dominates each workload's step, the roofline that bounds it,
# and its DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum
# from an ncu capture of the kernel as it stands; None when not measured).
DOMINANT = {
    "swin_t_stage1": ("swin_bf16_kernel<7,32>", "hbm", 57838336 + 1461504),
    "swin_t_stage1_fmap": ("swin_bf16_kernel<7,32,fmap>", "hbm", 57843712 + 1441024),
    "irpe_k_deit_s": ("rpe_pingpong_kernel<14,5,K>", "hbm", 28996864 + 0),
    "irpe_qkv_deit_s": ("rpe_pingpong_kernel<14,5,K,Q,V>", "hbm", 29055232 + 0),
    "irpe_k_56x56": ("rpe_pingpong_kernel<56,1,K,split>", "tensor", 58280192 + 2207232),
    "irpe_k_r2_deit_s": ("rpe_pingpong_kernel<14,5,K,128 buckets>", "hbm", None),
    "irpe_k_deit_s_cls": ("rpe_pingpong_kernel<14,5,K,cls>", "hbm", None),
}


def roofline_of(cfg, flops, nbytes, per_step_s, peaks, peak_src):
    kernel, bound, traffic = DOMINANT.get(cfg.name, ("?", "hbm", None))
    if bound == "tensor":
        achieved = flops / per_step_s / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = nbytes / per_step_s / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
            "kernel": kernel, "alg_bytes_per_launch": nbytes, "alg_flops_per_launch": flops}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, fl in zip(names, flags)
                          if fl.lower() == "active"})
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- GPU arm

def make_step(cfg, sets):
    """Returns step(i) running the hot path on input set i % len(sets)."""
    from vision_transformer_attention_gb300 import api
    from vision_transformer_attention_gb300.workloads import SwinConfig
    if isinstance(cfg, SwinConfig) and cfg.fmap:
        def step(i):
            s = sets[i % len(sets)]
            api.swin_window_attn_fwd_fmap(s["q"], s["k"], s["v"], s["table"], cfg.M,
                                          out=s["out"])
    elif isinstance(cfg, SwinConfig):
        def step(i):
            s = sets[i % len(sets)]
            api.swin_window_attn_fwd(s["q"], s["k"], s["v"], s["table"], cfg.M, out=s["out"])
    else:
        def step(i):
            s = sets[i % len(sets)]
            api.rpe_attn_fwd(s["q"], s["k"], s["v"], s["lut"], cfg.num_buckets, cfg.H, cfg.W,
                             cfg.flags, cls_token=cfg.cls, table_q=s["tab_q"], table_k=s["tab_k"],
                             table_v=s["tab_v"], out=s["out"])
    return step


def device_sets(cfg, dev, nbytes_step):
    from vision_transformer_attention_gb300 import api, workloads
    base = workloads.config_inputs(cfg)
    base = {k: (None if t is None else t.to(dev)) for k, t in base.items()}
    if isinstance(cfg, workloads.IrpeConfig):
        a, b, g = workloads.index_constants(cfg.ratio)
        lut, _, _ = api.rpe_build_bucket_ids(cfg.H, cfg.W, a, b, g, device=dev)
        base["lut"] = lut
    nsets = max(2, math.ceil(3 * L2_BYTES / nbytes_step))
    sets = []
    for r in range(nsets):
        s = dict(base)
        if r > 0:
            for key in ("q", "k", "v"):
                s[key] = base[key].clone()
        s["out"] = torch.empty_like(base["q"])
        sets.append(s)
    return sets


def time_graphs(step, K, W, group):
    """Warm up W steps eagerly on the capture stream (a stream's first call
    sets up what the library keeps per stream, which a capture cannot),
    capture `group` steps per CUDA graph, replay once untimed; returns the
    graphs, which together run exactly K steps."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    graphs = []
    idx = W
    with torch.cuda.stream(s):
        remaining = K
        while remaining > 0:
            n = min(group, remaining)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for j in range(n):
                    step(idx + j)
            graphs.append(g)
            idx += n
            remaining -= n
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for g in graphs:  # one untimed replay
        g.replay()
    torch.cuda.synchronize()
    return graphs


def replay_timed(graphs, barrier):
    stream = torch.cuda.current_stream()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for g in graphs:
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end)


def e2e_run(cfg, dev, steps, barrier):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device, runs the path and reads the result back.
    The steps are pipelined over three streams (uploads, compute, downloads)
    with two device buffer sets, so step i + 1's inputs go up while step i runs
    and step i - 1's result comes down; each step still moves its own bytes."""
    from vision_transformer_attention_gb300 import api, workloads
    base = workloads.config_inputs(cfg)
    host = {k: t.pin_memory() for k, t in base.items() if t is not None and k in ("q", "k", "v")}
    dq = [{k: torch.empty_like(t, device=dev) for k, t in host.items()} for _ in range(2)]
    tabs = {k: (None if base.get(k) is None else base[k].to(dev))
            for k in ("tab_q", "tab_k", "tab_v", "table")}
    out_host = torch.empty_like(base["q"]).pin_memory()
    lut = None
    if isinstance(cfg, workloads.IrpeConfig):
        a, b, g = workloads.index_constants(cfg.ratio)
        lut, _, _ = api.rpe_build_bucket_ids(cfg.H, cfg.W, a, b, g, device=dev)
    outs = [torch.empty_like(dq[0]["q"]) for _ in range(2)]
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded, computed, downloaded = ([ev() for _ in range(2)] for _ in range(3))
    used = [False, False]

    def one(i):
        j = i % 2
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(computed[j])   # step i - 2 has read this input set
            for k in ("q", "k", "v"):
                dq[j][k].copy_(host[k], non_blocking=True)
            uploaded[j].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(uploaded[j])
            if used[j]:
                s_run.wait_event(downloaded[j])  # step i - 2's result has left this buffer
            x = dq[j]
            if lut is not None:
                api.rpe_attn_fwd(x["q"], x["k"], x["v"], lut, cfg.num_buckets, cfg.H, cfg.W,
                                 cfg.flags, cls_token=cfg.cls, table_q=tabs["tab_q"],
                                 table_k=tabs["tab_k"], table_v=tabs["tab_v"], out=outs[j])
            elif cfg.fmap:
                api.swin_window_attn_fwd_fmap(x["q"], x["k"], x["v"], tabs["table"], cfg.M,
                                              out=outs[j])
            else:
                api.swin_window_attn_fwd(x["q"], x["k"], x["v"], tabs["table"], cfg.M, out=outs[j])
            computed[j].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[j])
            out_host.copy_(outs[j], non_blocking=True)
            downloaded[j].record(s_out)
        used[j] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(main)
    for st in (s_in, s_run, s_out):
        st.wait_event(start)
    for i in range(steps):
        one(3 + i)
    main.wait_stream(s_out)
    end.record(main)
    torch.cuda.synchronize()
    barrier()
    ms = start.elapsed_time(end)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()
    return ms, h2d, d2h


def oracle_runner(cfg):
    """(run(slices, out), S, tokens per slice, out buffer) for timing the oracle
    on cfg: run computes the picked (batch, head) or (window, head) slices into
    out. Inputs are converted to float64 and the iRPE id map is built once,
    here, outside any timed region (as the GPU path builds its offset table
    once per grid)."""
    import oracle
    from vision_transformer_attention_gb300 import workloads
    oracle.build()
    inp = workloads.config_inputs(cfg)
    f64 = {k: oracle._f64(t) for k, t in inp.items() if t is not None}
    out = np.zeros_like(f64["q"])
    if isinstance(cfg, workloads.SwinConfig):
        S = cfg.num_windows * cfg.heads

        def run(sl):
            oracle.swin_attention(f64["q"], f64["k"], f64["v"], f64["table"], cfg.M, slices=sl,
                                  out=out)
        return run, S, cfg.n / cfg.heads, out
    a, b, g = workloads.index_constants(cfg.ratio)
    ids, K = oracle.product_bucket_ids(cfg.H, cfg.W, a, b, g)
    if cfg.cls:
        ids, K = oracle.add_cls_bucket(ids, K)
    S = cfg.B * cfg.heads

    def run(sl):
        oracle.irpe_attention_ids(f64["q"], f64["k"], f64["v"], ids, K, cfg.flags,
                                  tab_q=f64.get("tab_q"), tab_k=f64.get("tab_k"),
                                  tab_v=f64.get("tab_v"), slices=sl, out=out)
    return run, S, cfg.N / cfg.heads, out


def cpu_baseline(cfg, budget_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload, its
    (batch, head) slices spread over every host core."""
    import oracle
    run, S, per_slice_tokens, _ = oracle_runner(cfg)
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    run(np.array([0]))
    one = max(time.perf_counter() - t0, 1e-4)  # one slice on one core
    n = int(min(S, max(cores, budget_s * cores / one)))
    t0 = time.perf_counter()
    used = oracle.parallel_slices(run, np.arange(n), cores)
    dt = time.perf_counter() - t0
    return {"value": n * per_slice_tokens / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{n} of {S} (batch, head) slices of {cfg.name}, fp64 C, id map built once "
                      f"before timing, slices split over {used} threads",
            "seconds": round(dt, 3), "single_core_tokens_per_s": per_slice_tokens / one}


def rank_helpers(dist, dev):
    """Replica coordination: a barrier, and the maximum of a per-rank float over
    all ranks (the slowest replica's time). No-ops for a single process."""
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)

    def max_over_ranks(x):
        if not dist:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def job_throughput(world, units_per_rank, seconds_per_step):
    """Whole-job units/s: every rank processes its own units (weak scaling) in
    the slowest rank's time."""
    return world * units_per_rank / seconds_per_step


def gpu_arm(args):
    from vision_transformer_attention_gb300 import workloads
    import __graft_entry__
    __graft_entry__.build()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    barrier, max_over_ranks = rank_helpers(dist, dev)

    peaks, peak_src = load_peaks()
    cfg = workloads.CONFIGS[args.workload]
    flops, nbytes, tokens = work_of(cfg)
    sets = device_sets(cfg, dev, nbytes)
    step = make_step(cfg, sets)
    graphs = time_graphs(step, args.steps, args.warmup, args.group)
    with ClockSampler(local) as clk:
        # each repeat times exactly K steps; the line reports the median repeat
        reps = [replay_timed(graphs, barrier) for _ in range(args.repeats)]
        # keep the GPU loaded for the clock samples if the timed region was short
        while sum(reps) < 1500 and len(reps) < args.repeats + 400:
            reps.append(replay_timed(graphs, barrier))
    ms = max_over_ranks(statistics.median(reps))
    clocks = clk.summary()
    per_step_s = ms / 1e3 / args.steps
    value = job_throughput(world, tokens, per_step_s)
    achieved_tflops = flops / per_step_s / 1e12
    del graphs

    # The same step with one input set reused every step, so q, k and v stay in
    # L2 between steps: labelled apart, never the line's value (which reads its
    # inputs from HBM). Only where the step's bytes fit well within L2.
    warm = None
    if nbytes <= L2_BYTES / 2:
        kw = min(args.steps, 500)
        gw = time_graphs(make_step(cfg, sets[:1]), kw, args.warmup, min(args.group, kw))
        tw = max_over_ranks(statistics.median(replay_timed(gw, barrier) for _ in range(5))) / 1e3 / kw
        del gw
        warm = {"ms_per_step": tw * 1e3, "tokens_per_s": job_throughput(world, tokens, tw),
                "tflops": flops / tw / 1e12, "tc_frac": flops / tw / 1e12 / peaks["bf16_tflops"],
                "note": f"one input set ({nbytes / 2**20:.1f} MiB) reused every step, L2-resident; "
                        f"median of 5 timed repeats of {kw} steps; not the line's value"}

    e2e_ms, h2d, d2h = e2e_run(cfg, dev, args.e2e_steps, barrier)
    e2e_ms = max_over_ranks(e2e_ms)
    e2e_value = job_throughput(world, tokens, e2e_ms / 1e3 / args.e2e_steps)

    extra_cfgs = {}
    if not args.headline_only:
        for name in ("swin_t_stage1", "swin_t_stage1_fmap", "irpe_qkv_deit_s", "irpe_k_56x56",
                     "irpe_k_r2_deit_s", "irpe_k_deit_s_cls"):
            if name == args.workload:
                continue
            c = workloads.CONFIGS[name]
            f, b, tk = work_of(c)
            st = make_step(c, device_sets(c, dev, b))
            k = max(20, int(args.steps * 0.2) if name != "irpe_k_56x56" else 200)
            gr = time_graphs(st, k, 5, min(args.group, k))
            t = max_over_ranks(statistics.median(replay_timed(gr, barrier) for _ in range(5))) / 1e3 / k
            del gr
            bound_tc = name == "irpe_k_56x56"
            extra_cfgs[name] = {
                "tokens_per_s": job_throughput(world, tk, t), "ms_per_step": t * 1e3,
                "tflops": f / t / 1e12, "gbs": b / t / 1e9,
                "tc_frac": f / t / 1e12 / peaks["bf16_tflops"],
                "hbm_frac": b / t / 1e9 / peaks["hbm_gbs"],
                "bound": "tensor" if bound_tc else "hbm"}
            torch.cuda.empty_cache()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, N(0,0.02) R^K; no dataset)",
        "config": {**workload_config(cfg),
                   "global_batch": getattr(cfg, "B", getattr(cfg, "num_windows", 0)) * world,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs rotate over {len(sets)} copies ({len(sets) * nbytes / 2**20:.0f} MiB"
                         f" > 3x L2), no flush",
                   "timing": f"CUDA graphs of {args.group} launches; median of {len(reps)} timed "
                             f"repeats of the {args.steps} steps"},
        "repeats": {"n": len(reps), "median_ms": statistics.median(reps), "min_ms": min(reps),
                    "max_ms": max(reps)},
        "tflops": achieved_tflops,
        "warm_l2": warm,
        "tc_frac_of_peak": achieved_tflops / peaks["bf16_tflops"],
        "attainable_frac": achieved_tflops / min(peaks["bf16_tflops"],
                                                 flops / nbytes * peaks["hbm_gbs"] / 1e3),
        "roofline": roofline_of(cfg, flops, nbytes, per_step_s, peaks, peak_src),
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "pipeline": "uploads, compute and downloads on three streams, two device buffer sets"},
        "gpu_launches": args.steps,
        "configs_extra": extra_cfgs,
    }
    if not args.no_cpu_baseline and args.workload == HEADLINE:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm (the oracle)

def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from vision_transformer_attention_gb300 import workloads
    cfg = workloads.CONFIGS[HEADLINE]
    run, S, per_slice_tokens, _ = oracle_runner(cfg)
    # One step = a bounded sample of the workload: two (batch, head) slices per
    # host core, cycling through the batch, so any --steps K finishes in
    # minutes. The per-slice work is exactly cpu_baseline's.
    cores = os.cpu_count() or 1
    per_step = min(S, 2 * cores)

    def step(i):
        sl = (np.arange(per_step) + i * per_step) % S
        return oracle.parallel_slices(run, sl, cores)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    used = 1
    for i in range(args.steps):
        used = step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * per_step * per_slice_tokens / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (the same seeded inputs as the GPU arm)",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"{per_step} of {S} (batch, head) slices per step, fp64 C, "
                                   f"id map built once before timing, split over {used} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--group", type=int, default=100, help="launches per CUDA graph")
    ap.add_argument("--repeats", type=int, default=10,
                    help="timed repeats of the K steps (the median is reported)")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--workload", default=HEADLINE,
                    help="workload timed for the main line (the headline unless profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = args.steps if args.steps is not None else 200
        args.warmup = max(args.warmup if args.warmup is not None else 1, 1)
        reference_arm(args)
        return
    args.steps = args.steps if args.steps is not None else 2000
    args.warmup = max(args.warmup if args.warmup is not None else 20, 3)
    args.group = max(1, min(args.group, args.steps))
    gpu_arm(args)


if __name__ == "__main__":
    main()
