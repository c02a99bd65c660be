#!/usr/bin/env python
"""Benchmark of the MoE routing-and-expert step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

Metric: routed tokens/s per MoE layer (T / layer time) on the 12-layer
MoE-GPT-like routing stream (T=16384 tokens per iteration, E=16 experts,
top-2, H=1024, F=2048 GeLU experts, bf16 weights/activations, fp32
accumulate, window s=10).  One step = one iteration of the whole hot path
over all 12 layers: route, window-statistics update, next-layer prediction,
replica counts, dispatch, grouped expert FFN, combine (every stage a libmoe
kernel, launched through the C ABI on one stream).  value = T * L * steps *
n_gpus / (max over ranks of the timed region).

Inputs are synthetic (seeded Zipf-biased logits with inter-layer correlation,
N(0,1) activations, N(0,0.02) weights; no dataset or checkpoint exists here)
and already resident in HBM; every step touches ~1.5 GB of expert weights
plus ~0.9 GB of activations, far above the 126 MB L2, so no L2 flush is
needed.  `e2e` repeats the measurement through the same public calls with the
per-step inputs (X, logits) copied from pinned host memory and the layer
outputs copied back inside the timed region.

--impl reference times the CPU oracle (NumPy float64, the repository's
correctness reference) on a bounded sample of the same workload; under
torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed tokens/sec per MoE layer (1xB300) and % of HBM / bf16 tensor roofline"
UNIT = "tokens/s"
STAGES = ["route", "stats", "predict", "replicate", "dispatch", "ffn", "combine"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="moe_gpt_stream")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch every call from Python instead of graph replay")
    ap.add_argument("--gather", action="store_true",
                    help="gather the rows in the FFN's loads (moe_expert_ffn_gather) instead of copying them")
    ap.add_argument("--unfused", action="store_true",
                    help="make the five separate front calls instead of moe_layer_front")
    ap.add_argument("--chunks", type=int, default=1,
                    help="EPS-MoE pipeline: dispatch/FFN/combine over this many token chunks on two streams")
    ap.add_argument("--physical-replicas", action="store_true",
                    help="copy each replica's weights into its own slot (moe_replicate_weights) before the FFN")
    ap.add_argument("--replicate-from", choices=["histogram", "prediction"], default="histogram",
                    help="replica table from the layer's own histogram or from the previous layer's prediction")
    ap.add_argument("--ffn-kernel", choices=["auto", "single", "pair", "fused"], default="auto",
                    help="grouped-GEMM kernel of the expert FFN (default: the library's choice)")
    ap.add_argument("--no-pdl", action="store_true", help="ordinary launches instead of programmatic dependent launch")
    ap.add_argument("--fuse-combine", action="store_true",
                    help="the combine in the FFN's second GEMM epilogue (moe_expert_ffn_combine)")
    ap.add_argument("--small-sms", type=int, default=0,
                    help="SMs of the FFN's small-batch kernels (MOE_OPT_FFN_SMALL_SMS; 0, the library's default: no "
                         "small-batch path; -1: the split model chooses)")
    ap.add_argument("--small-threshold", type=int, default=64,
                    help="experts with fewer rows take the small-batch FFN kernel (0: none, no side-stream launches)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="oracle sample size (tokens of one layer)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (small profiling captures; not a bench line)")
    ap.add_argument("--T", type=int, default=0, help="override tokens (small profiling captures; not a bench line)")
    ap.add_argument("--E", type=int, default=0, help="override experts (small profiling captures; not a bench line)")
    ap.add_argument("--sweep", action="store_true",
                    help="time each stage alone over T = 2^14 .. 2^20 (one JSON line per T; not the bench line)")
    ap.add_argument("--quality", action="store_true",
                    help="prediction quality and prediction-driven replication over the workload's iterations "
                         "(one JSON line; not the bench line)")
    ap.add_argument("--quality-iters", type=int, default=200)
    ap.add_argument("--wgrad-bf16", action="store_true", help="--backward: weight gradients written in bf16")
    ap.add_argument("--backward", action="store_true",
                    help="time the layer's backward (moe_ffn_backward + moe_route_backward) instead; one JSON line")
    ap.add_argument("--crossover", action="store_true",
                    help="time the EPS-MoE GEMM crossover shapes on the grouped and small-batch FFN kernels "
                         "(one JSON line per shape; not the bench line)")
    ap.add_argument("--sweep-min-log2", type=int, default=14)
    ap.add_argument("--sweep-max-log2", type=int, default=20)
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# process group (one rank per GPU; replicas only: ranks share no data)
# ----------------------------------------------------------------------------
def dist_init():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    """Max of a host float over ranks (the timing aggregate; no data exchange)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, elapsed_max_s: float) -> float:
    return units_per_rank * world / elapsed_max_s


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        out_dir = os.environ.get("MOE_BENCH_OUT_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"moe_bench_clocks_rank{device_index}.csv")
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            gid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            gid = str(device_index)
        self.gid = gid

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gid}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 8:
                continue
            try:
                rows.append((float(p[0]), float(p[1]), float(p[2]) if p[2] not in ("[N/A]", "N/A") else 0.0,
                             p[3], p[4], p[5], p[6], p[7]))
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for nm, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r[2] for r in rows)}


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------
def algorithmic_work(c, used_experts=None, gather=False):
    """Per-layer algorithmic bytes (HBM stages) and flops (FFN), as the method
    must move them (not what the kernels happen to move).  The FFN must read
    the weights of every expert that received a token (used_experts, counted
    from a layer's histogram; all E when unknown) once, its input rows once and write its output
    rows once (plus the bf16 intermediate written and read back).  With the
    gathered FFN input (gather=True) dispatch moves no rows and the FFN reads
    the T token rows instead of the A dispatched ones."""
    T, E, k, H, F, A = c.T, c.E, c.k, c.H, c.F, c.A
    ngemm = 3 if c.act == "swiglu" else 2
    Eu = E if used_experts is None else used_experts
    work = {
        "route": {"bytes": T * E * 4 + A * 8},
        "stats": {"bytes": 2 * A * 4 + (E + E * E) * 4 * 2 + (E + E * E) * 8 * 2},
        "predict": {"bytes": E * E * 8 + E * 8 + E * E * 4 + E * 8},
        "replicate": {"bytes": E * 16},
        "dispatch": {"bytes": A * 4 + 2 * A * 4 + (0 if gather else T * H * 2 + A * H * 2)},
        "ffn": {"flops": 2 * ngemm * A * H * F,
                "bytes": int(ngemm * Eu * H * F * 2 + (T if gather else A) * H * 2 + A * H * 2
                             + (ngemm - 1) * A * F * 2 * 2)},
        "combine": {"bytes": A * H * 2 + A * 8 + T * H * 2},
    }
    # the fused front does the work of the five calls it replaces
    work["front"] = {"bytes": sum(work[s]["bytes"] for s in ("route", "stats", "predict", "replicate", "dispatch"))}
    return work


def stationary_base(c):
    """First iteration of the workload's stationary phase that is a multiple
    of the window: the skew ramps over the first `alpha_ramp` iterations, then
    stays fixed (moe_gpt_stream: 50)."""
    return -(-c.alpha_ramp // c.window) * c.window


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# the FFN kernels and the host code that sets their launch parameters (the
# fused kernel's lag between a block's GEMM1 and GEMM2 tiles changes its traffic)
FFN_SOURCES = ("ffn.cuh", "ffn_pair.cuh", "ffn_fused.cuh", "ffn_small.cuh", "sm100_ptx.cuh", "moe_api.cu")


def ffn_source_hash():
    """First 16 hex digits of the SHA-256 of the FFN kernel sources."""
    h = hashlib.sha256()
    for name in FFN_SOURCES:
        h.update(open(os.path.join(ROOT, "moe_expert_routing_02_b300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def ffn_traffic_per_launch():
    """DRAM bytes per FFN call from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ffn_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            a, b = line.split(":", 1)
            kv[a.strip()] = b.strip()
    h = ffn_source_hash()
    if kv.get("ffn_source_sha256_16") != h:
        return None
    try:
        return float(kv["dram_bytes_per_ffn_call_full_size"])
    except (KeyError, ValueError):
        return None


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from moe_expert_routing_02_b300 import _build
    _build.build()
    import moe_expert_routing_02_b300 as M
    from moe_expert_routing_02_b300 import workloads as W
    from moe_expert_routing_02_b300.layer import MoELayerStep, capture_slot_graphs

    torch.cuda.set_device(local)
    c = W.config_by_name(args.config)
    if args.layers or args.T or args.E:
        import dataclasses
        c = dataclasses.replace(c, L=min(args.layers, c.L) if args.layers else c.L, T=args.T or c.T,
                                E=args.E or c.E)
    dev = torch.device("cuda", local)
    # The timed steps replay the stream's stationary phase: one distinct
    # iteration per window slot, starting at the first multiple of the window
    # at or after the end of the skew ramp (moe_gpt_stream: iterations 50..59
    # at alpha = 1.2, where hot experts are split into replica groups).
    base_it = stationary_base(c)
    POOL = c.window
    logits = [[torch.from_numpy(l).to(dev) for l in W.make_layer_logits(c, base_it + q)] for q in range(POOL)]
    xs = [W.make_x(c, 0, j, device=dev) for j in range(c.L)]
    weights = [W.make_weights(c, j, device=dev) for j in range(c.L)]
    outs = [torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev) for _ in range(c.L)]
    stats = M.MoEStats(c.L, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats=stats, replicate=True, fused=not args.unfused,
                        gather=args.gather, replicate_from=args.replicate_from,
                        physical_replicas=args.physical_replicas, small_group_threshold=args.small_threshold,
                        fuse_combine=args.fuse_combine, device=dev)
    if args.physical_replicas:
        weights = [MoELayerStep.replica_buffers(w) for w in weights]
    if args.chunks > 1:
        from moe_expert_routing_02_b300.layer import ChunkedLayerStep
        step = ChunkedLayerStep(c.T, c.E, c.k, c.H, c.F, c.act, stats, chunks=args.chunks, device=dev)
        step.fused, step.gather = True, False
        stage_names = ["ffn"]
    stage_names = ["front", "ffn", "combine"] if step.fused else STAGES
    M.moe_set_option(M.MOE_OPT_FFN_KERNEL, {"auto": M.MOE_FFN_KERNEL_AUTO, "single": M.MOE_FFN_KERNEL_SINGLE,
                                            "pair": M.MOE_FFN_KERNEL_PAIR,
                                            "fused": M.MOE_FFN_KERNEL_FUSED}[args.ffn_kernel])
    M.moe_set_option(M.MOE_OPT_PDL, 0 if args.no_pdl else 1)
    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, args.small_sms)

    def run_step(it, ev=None):
        for j in range(c.L):
            step.run(base_it + it, j, logits[it % POOL][j], xs[j], weights[j], outs[j],
                     events=None if ev is None else ev[j])

    def new_events(names=None):
        names = stage_names if names is None else names
        # external=True: inside a captured graph the records become event nodes
        # whose timestamps are readable after a replay
        return [{s: (torch.cuda.Event(enable_timing=True, external=True),
                     torch.cuda.Event(enable_timing=True, external=True))
                 for s in names} for _ in range(c.L)]

    # one eager step first (sets kernel attributes, checks for errors)
    run_step(0)
    torch.cuda.synchronize()
    M.moe_check()

    # The stats update only uses the iteration modulo the window, so one
    # captured graph per ring slot replays every iteration exactly.  The timed
    # graphs record events around the expert FFN only (the roofline kernel);
    # a second set with events around every stage gives the breakdown.
    n_graphs = 0 if args.eager else c.window

    def capture(names):
        return capture_slot_graphs(run_step, n_graphs, lambda: new_events(names))

    graphs, graph_ev = capture(["ffn"]) if n_graphs else ([], [])

    def replay(it, ev=None):
        if n_graphs:
            graphs[it % n_graphs].replay()
        else:
            run_step(it, ev)

    for it in range(args.warmup):
        replay(it)
    torch.cuda.synchronize()
    M.moe_check()

    K = args.steps
    stage_ev = [new_events() for _ in range(K)] if not n_graphs else None
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record()
    for s in range(K):
        replay(args.warmup + s, None if stage_ev is None else stage_ev[s])
    t1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    M.moe_check()
    elapsed = t0.elapsed_time(t1) / 1e3
    elapsed_max = max_over_ranks(elapsed)
    units = c.T * c.L * K
    value = whole_job_value(units, world, elapsed_max)

    def stage_means(sets, names=None):
        names = stage_names if names is None else names
        out = {}
        for sname in names:
            ts = [ev[j][sname][0].elapsed_time(ev[j][sname][1]) for ev in sets for j in range(c.L)
                  if sname in ev[j] and not (sname == "predict" and j == c.L - 1)]
            if ts:
                out[sname] = sum(ts) / len(ts)
        return out

    if n_graphs:
        # FFN time from the timed region (last replay of each slot graph)
        replayed = sorted({(args.warmup + s_i) % n_graphs for s_i in range(K)})
        ffn_ms = stage_means([graph_ev[q] for q in replayed], ["ffn"])["ffn"]
        if args.chunks > 1:
            stage_ms = {"ffn": ffn_ms}   # the chunked step times its whole chunked part as one stage
        else:
            # stage breakdown: instrumented graphs replayed once per slot afterwards
            graphs_all, ev_all = capture(stage_names)
            for q in range(n_graphs):
                graphs_all[q].replay()
            torch.cuda.synchronize()
            stage_ms = stage_means(ev_all)
            del graphs_all
    else:
        stage_ms = stage_means(stage_ev)
        ffn_ms = stage_ms["ffn"]
    stage_note = None
    # experts that received tokens, from the last layer call's histogram (libmoe's own count)
    used = float((step.hist > 0).sum().item())
    work = algorithmic_work(c, used_experts=used, gather=step.gather)
    peaks = load_peaks()
    stages = {}
    for sname in stage_names:
        if sname not in stage_ms:
            continue
        t = stage_ms[sname] / 1e3
        d = {"us_per_layer": round(stage_ms[sname] * 1e3, 2)}
        if "flops" in work[sname]:
            d["tflops"] = round(work[sname]["flops"] / t / 1e12, 1)
            d["frac_bf16"] = round(work[sname]["flops"] / t / 1e12 / peaks["bf16_tflops"], 3)
        d["gbs"] = round(work[sname]["bytes"] / t / 1e9, 1)
        d["frac_hbm"] = round(work[sname]["bytes"] / t / 1e9 / peaks["hbm_gbs"], 3)
        stages[sname] = d
    ffn_t = ffn_ms / 1e3
    fl, by = work["ffn"]["flops"], work["ffn"]["bytes"]
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)   # flop/B
    if fl / by >= ridge:
        achieved = fl / ffn_t / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "peak_source": f"bf16_tflops (burst) of {peaks['source']} peaks: the timed region lasts "
                                   f"{elapsed:.2f} s",
                    "frac_of_sustained_peak": round(achieved / peaks["bf16_tflops_sustained"], 4)}
        if clk and clk.get("sm_mhz") and clk.get("sm_max_mhz"):
            # the burst peak was measured at the maximum SM clock; the rate the
            # tensor pipe can reach scales with the clock the run actually saw
            scale = min(1.0, clk["sm_mhz"] / clk["sm_max_mhz"])
            roofline["frac_at_sampled_clock"] = round(achieved / (peaks["bf16_tflops"] * scale), 4)
            roofline["sampled_sm_mhz_over_max"] = round(scale, 3)
    else:
        achieved = by / ffn_t / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"hbm_gbs of {peaks['source']} peaks",
                    "tflops": round(fl / ffn_t / 1e12, 1)}
    n_ffn = M.moe_ffn_launches(c.A, c.E, c.H, c.F, c.act, args.small_threshold, step.gather)
    ffn_desc = ("moe_expert_ffn: fused GEMM1+GEMM2 launch" if n_ffn in (1, 3) else
                "moe_expert_ffn: GEMM1 and GEMM2 launches") + (" (+2 small-batch launches on the side stream)"
                                                               if n_ffn >= 3 else "")
    roofline.update({"kernel": ffn_desc, "traffic": ffn_traffic_per_launch(),
                     "algorithmic_flops_per_call": fl, "algorithmic_bytes_per_call": by,
                     "arithmetic_intensity": round(fl / by, 1), "ridge_flop_per_byte": round(ridge, 1),
                     "experts_with_tokens": used})
    launches = K * sum(step.launches(j, c.L) for j in range(c.L))
    if stage_note:
        roofline["note"] = stage_note
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_max / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": c.name, "T": c.T, "L": c.L, "E": c.E, "k": c.k, "H": c.H, "F": c.F, "act": c.act,
                   "window": c.window, "replication": "on",
                   "iterations": (f"{base_it}..{base_it + POOL - 1} of the stream (one per window slot, cycled; "
                                  f"alpha = {W.alpha_at(c, base_it):g}, the stationary skewed phase)"),
                   "parallelism": f"replicas x{world} (no data exchange)",
                   "l2": "no flush: each step streams ~1.5 GB of weights + activations, >> 126 MB L2",
                   "launch": "eager" if args.eager else f"CUDA graph per step ({c.window} graphs, one per window slot)",
                   "front": "separate calls" if args.unfused else "moe_layer_front (2 launches)",
                   "ffn_kernel": args.ffn_kernel,
                   "pdl": not args.no_pdl,
                   "small_group_threshold": args.small_threshold,
                   "small_path_sms": "split model" if args.small_sms < 0 else (
                       "none (the grouped kernel takes every expert)" if args.small_sms == 0 else args.small_sms),
                   "combine": "in the FFN's second GEMM epilogue" if args.fuse_combine else "separate kernel",
                   "chunks": args.chunks,
                   "replicas": ("physical copies (moe_replicate_weights)" if args.physical_replicas
                                else "aliasing their expert's weights") + f", table from {args.replicate_from}",
                   "ffn_input": "gathered from x in GEMM1's loads (tile::gather4)" if step.gather
                                else "rows copied into dispatch order",
                   "stage_timing": "CUDA events around each stage, every layer of every timed step" if args.eager
                   else "FFN: events captured around it in the timed graphs (last replay of each); other stages: "
                        "a second set of graphs with events around every stage, replayed once per slot after the "
                        "timed region (each event node adds ~1-2 us)"},
        "roofline": roofline, "stages": stages, "gpu_launches": launches, "clocks": clk,
        "routing": routing_summary(step, c, args.small_threshold),
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, c, step, logits, weights, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline(c, args.cpu_tokens or c.T)
    return result


def routing_summary(step, c, small_threshold):
    """Load balance of the last layer call, from libmoe's own histogram and
    dispatch layout (read back after the timed region): per-expert load max
    and standard deviation over the mean, the replica groups, the largest
    group over the per-expert target A/E, and the experts the small-batch
    path serves (fewer than `small_threshold` rows, chosen per expert)."""
    import numpy as np
    try:
        hist = step.hist.cpu().numpy().astype(np.float64)
        go = step.go_full if hasattr(step, "go_full") else step.go
        go = go.cpu().numpy().astype(np.int64)
        n_groups = int(step.rep_base[-1].item()) if step.replicate else c.E
        rows = np.diff(go[:n_groups + 1])
        mean = hist.mean()
        return {"of": "the last layer call made (after the timed region)",
                "load_max_over_mean": round(float(hist.max() / mean), 3),
                "load_stddev_over_mean": round(float(hist.std() / mean), 3),
                "replica_groups": n_groups, "extra_replicas": n_groups - c.E,
                "largest_group_over_target": round(float(rows.max() / (c.T * c.k / c.E)), 3),
                "experts_without_tokens": int((hist == 0).sum()),
                "small_path_experts": int(((hist > 0) & (hist < small_threshold)).sum())}
    except Exception as e:  # a summary must never cost the measurement line
        return {"error": f"{type(e).__name__}: {e}"}


def run_e2e(args, c, step, logits, weights, dev, world):
    """Same metric through the same calls, with the per-step inputs (logits,
    X) in pinned host memory and every layer's output copied back to pinned
    host memory, inside the timed region.  HostPipeline overlaps the copies in,
    the layer calls and the copies out on three streams (double-buffered)."""
    import torch
    from moe_expert_routing_02_b300.layer import HostPipeline
    h_logits = [[l.cpu().pin_memory() for l in it] for it in logits]
    h_x = [torch.empty((c.T, c.H), dtype=torch.bfloat16).pin_memory() for _ in range(c.L)]
    for j in range(c.L):
        h_x[j].copy_(torch.randn((c.T, c.H), dtype=torch.float32).to(torch.bfloat16))
    h_out = [torch.empty((c.T, c.H), dtype=torch.bfloat16).pin_memory() for _ in range(c.L)]
    pipe = HostPipeline(step, device=dev)

    def run_step(it):
        pipe.run(it, h_logits[it % len(h_logits)], h_x, weights, h_out)

    base = 10_000
    for it in range(args.warmup):
        run_step(base + it)
    torch.cuda.synchronize()
    barrier()
    steps = max(1, min(args.steps, 50))
    t0 = time.perf_counter()
    for s in range(steps):
        run_step(base + args.warmup + s)
    torch.cuda.synchronize()
    el = max_over_ranks(time.perf_counter() - t0)
    h2d = c.L * (c.T * c.E * 4 + c.T * c.H * 2)
    d2h = c.L * c.T * c.H * 2
    return {"value": round(whole_job_value(c.T * c.L * steps, world, el), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(el / steps * 1e3, 3),
            "how": "HostPipeline: H2D of layer j+1, layer j, D2H of layer j-1 on three streams; pinned host buffers"}


# ----------------------------------------------------------------------------
# CPU oracle (the baseline leg and the reference arm)
# ----------------------------------------------------------------------------
def oracle_layer_sample(c, T_s, it=0, seed_layer=0, cache={}):
    """One layer of the workload for the first T_s tokens, every stage in the
    oracle: top-k, histogram + window update + prediction, replica counts,
    dispatch, expert FFN of every assignment, combine.  Returns seconds."""
    import numpy as np
    from moe_expert_routing_02_b300 import workloads as W
    from oracle import moe_oracle as O
    key = (c.name, T_s)
    if key not in cache:
        lg = W.make_layer_logits(c, it, T=T_s, layers=min(2, c.L))
        x = W.bf16_bits(W.make_x(c, it, seed_layer, T=T_s))
        w1, w3, w2 = (None if t is None else W.bf16_bits(t) for t in W.make_weights(c, seed_layer))
        cache.clear()
        cache[key] = (lg, x, w1, w3, w2)
    lg, x, w1, w3, w2 = cache[key]
    t0 = time.perf_counter()
    st = O.WindowStats(len(lg), c.E, c.window)
    prev = None
    for j, l in enumerate(lg):  # layer j-1's routing feeds layer j's co-selection counts
        idx, w = O.topk_gate(l, c.k)
        st.update(it, j, idx, prev)
        prev = idx
    h = O.histogram(idx, c.E)
    st.predict(0)
    rep = O.replicate(h, idx.size)
    go, perm, inv = O.dispatch(idx, c.E, rep[1])
    xp = O.gather_rows(x, perm, c.k)
    y = O.expert_ffn(xp, go, rep[2], w1, w3, w2, c.act)
    O.combine(y, inv, w)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_cpu_baseline(c, T_s, min_reps=3, min_seconds=10.0, max_reps=20):
    # warm once (input generation, imports), then time layer samples until at
    # least `min_reps` of them and `min_seconds` of CPU work are done; then one
    # sample of a quarter of the tokens with the BLAS pool held to one thread
    # (the single-core rate)
    oracle_layer_sample(c, T_s)
    t, reps = 0.0, 0
    while reps < max_reps and (reps < min_reps or t < min_seconds):
        t += oracle_layer_sample(c, T_s)
        reps += 1
    res = {"value": round(reps * T_s / t, 1), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
           "sample": f"{reps} x one layer of {c.name} with {T_s} of {c.T} tokens (all k={c.k} assignments "
                     f"through route, stats+predict over 2 layers' routing, replicate, dispatch, fp64 FFN, "
                     f"combine), {t:.2f} s total; NumPy BLAS threads on {cpu_cores()} host cores"}
    # a child process whose BLAS / OpenMP pools are held to one thread
    T_1 = max(T_s // 4, 1)
    code = ("import sys, bench; from moe_expert_routing_02_b300 import workloads as W; "
            f"c = W.config_by_name({c.name!r}); bench.oracle_layer_sample(c, {T_1}); "
            f"print(bench.oracle_layer_sample(c, {T_1}))")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=600)
        t1 = float(r.stdout.strip().splitlines()[-1])
        res["single_core_value"] = round(T_1 / t1, 1)
        res["single_core_sample"] = (f"one layer of {c.name} with {T_1} tokens in a child process with one "
                                     f"BLAS / OpenMP thread, {t1:.2f} s")
    except Exception as ex:  # reported, not fatal: the all-cores figure above stands
        res["single_core_value"] = None
        res["single_core_sample"] = f"not measured: {type(ex).__name__}"
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from moe_expert_routing_02_b300 import workloads as W
    c = W.config_by_name(args.config)
    T_s = args.cpu_tokens or 4096
    for _ in range(max(args.warmup, 1)):
        oracle_layer_sample(c, T_s)
    ts = [oracle_layer_sample(c, T_s) for _ in range(args.steps)]
    total = sum(ts)
    value = T_s * args.steps / total
    return {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": c.name, "T": c.T, "L": c.L, "E": c.E, "k": c.k, "H": c.H, "F": c.F,
                       "act": c.act, "sample_tokens_per_step": T_s},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"each step: one layer of {c.name} for {T_s} tokens, every stage in the "
                                       f"float64 NumPy oracle"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


class L2Flush:
    """Empties L2 between timed calls: writes a buffer of twice the L2 size
    (evicting everything the previous call left, including its dirty lines),
    then reads a second one of the same size, so that the flush's own dirty
    lines are written back here and not during the next timed call (which
    would otherwise pay up to an L2's worth of write-backs it did not cause)."""

    def __init__(self, dev, l2_bytes=126 * 2 ** 20):
        import torch
        self.w = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(2 * l2_bytes // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def run_sweep(args):
    """Every stage of the path timed alone over T = 2^14 .. 2^20 tokens with the
    moe_gpt_stream workload's distributions (E=16, top-2, H=1024, Zipf bias,
    correlated second layer).  Each stage: 5 warm-up calls, then 20 calls,
    each preceded by an L2 flush (L2Flush: a write, then a read, of 2x the L2
    size, so the timed call pays no write-back of the flush's dirty lines) and
    timed alone with CUDA events; median, p10 and p90.  Fraction of HBM = algorithmic bytes /
    median time / the measured copy bandwidth."""
    import dataclasses
    import torch
    import moe_expert_routing_02_b300 as M
    from moe_expert_routing_02_b300 import workloads as W
    M.lib()
    base = W.config_by_name(args.config)
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    for lg2 in range(args.sweep_min_log2, args.sweep_max_log2 + 1):
        T = 2 ** lg2
        c = dataclasses.replace(base, T=T, L=2)
        E, k, H, A = c.E, c.k, c.H, T * c.k
        lgs = [torch.from_numpy(l).to(dev) for l in W.make_layer_logits(c, 0, layers=2)]
        x = W.make_x(c, 0, 1, device=dev)
        st = M.MoEStats(2, E, c.window)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        idx0, w0 = M.moe_route(lgs[0], k)
        idx1 = torch.empty((T, k), dtype=i32, device=dev)
        w1 = torch.empty((T, k), dtype=f32, device=dev)
        hist = torch.empty(E, dtype=i32, device=dev)
        pred = (torch.empty(E, dtype=f32, device=dev), torch.empty((E, E), dtype=f32, device=dev),
                torch.empty(E, dtype=f32, device=dev))
        rep = (torch.empty(E, dtype=i32, device=dev), torch.empty(E + 1, dtype=i32, device=dev),
               torch.empty(2 * E, dtype=i32, device=dev))
        disp = (torch.empty(2 * E + 1, dtype=i32, device=dev), torch.empty(A, dtype=i32, device=dev),
                torch.empty(A, dtype=i32, device=dev), torch.empty((A, H), dtype=bf, device=dev))
        ws = torch.empty(max(M.workspace_bytes(M.MOE_OP_DISPATCH, T, k, E),
                             M.workspace_bytes(M.MOE_OP_LAYER_FRONT, T, k, E), 16), dtype=torch.uint8, device=dev)
        y = torch.zeros((A, H), dtype=bf, device=dev)
        out = torch.empty((T, H), dtype=bf, device=dev)
        M.moe_route(lgs[1], k, idx=idx1, w=w1)
        M.moe_stats_update(st, 0, 1, idx1, idx0, hist_out=hist)
        M.moe_replicate(hist, A, out=rep)
        front_out = {"idx": idx1, "w": w1, "hist": hist, "p_seq": pred[0], "cond": None, "p_next": None,
                     "copies": rep[0], "rep_base": rep[1], "group_expert": rep[2], "group_offsets": disp[0],
                     "perm": disp[1], "inv_perm": disp[2], "xp": disp[3]}
        stages = {
            "route": (lambda: M.moe_route(lgs[1], k, idx=idx1, w=w1), T * E * 4 + A * 8),
            "stats": (lambda: M.moe_stats_update(st, 0, 1, idx1, idx0, hist_out=hist),
                      2 * A * 4 + (E + E * E) * 4 * 2 + (E + E * E) * 8 * 2),
            "predict": (lambda: M.moe_predict(st, 0, out=pred), E * E * 8 + E * 8 + E * E * 4 + E * 8),
            "replicate": (lambda: M.moe_replicate(hist, A, out=rep), E * 16),
            "dispatch": (lambda: M.moe_dispatch(x, idx1, E, rep[1], out=disp, workspace=ws),
                         A * 4 + T * H * 2 + A * H * 2 + 2 * A * 4),
            "front": (lambda: M.moe_layer_front(lgs[1], x, st, 0, 1, k, idx_prev=idx0, out=front_out, workspace=ws),
                      T * E * 4 + A * 8 + 2 * A * 4 + A * 4 + T * H * 2 + A * H * 2 + 2 * A * 4),
            "combine": (lambda: M.moe_combine(y, disp[2], w1, out=out), A * H * 2 + A * 8 + T * H * 2),
        }
        res = {}
        for name, (fn, nbytes) in stages.items():
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(20):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            M.moe_check()
            ts.sort()
            med = ts[len(ts) // 2]
            gbs = nbytes / (med * 1e-6) / 1e9
            res[name] = {"us_median": round(med, 2), "us_p10": round(ts[2], 2), "us_p90": round(ts[17], 2),
                         "bytes": int(nbytes), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)}
        print(json.dumps({"sweep": f"{c.name} distributions, each stage alone, L2 flushed (written, then read clean) before every call",
                          "T": T, "E": E, "k": k, "H": H, "hbm_peak_gbs": peaks["hbm_gbs"],
                          "peak_source": peaks["source"], "stages": res}), flush=True)
        del lgs, x, st, idx0, w0, idx1, w1, disp, ws, y, out, front_out, stages
        torch.cuda.empty_cache()
    return 0


def backward_flops(c):
    """Algorithmic flops of the expert FFN's backward for one layer: the data
    gradients dA = dY W2^T and dxp = dz W1^T (+ du W3^T), GEMM1 recomputed
    (one GEMM for GeLU, two for SwiGLU) and the weight gradients (2 or 3),
    each 2 A H F: 10 A H F for GeLU, 16 A H F for SwiGLU."""
    return (16 if c.act == "swiglu" else 10) * c.A * c.H * c.F


def run_backward(args):
    """The backward of one routed expert layer at the config's full size:
    moe_ffn_backward (combine, FFN and dispatch backward, all weight
    gradients) plus moe_route_backward, after a forward that produced y.
    W warm-up steps, then K steps timed with CUDA events on the launching
    stream; the operands (xp, dY, intermediates, fp32 gradients) are far
    larger than L2.  The forward FFN (moe_expert_ffn) is timed the same way
    for comparison."""
    import dataclasses
    import torch
    import moe_expert_routing_02_b300 as M
    from moe_expert_routing_02_b300 import workloads as W
    M.lib()
    c = W.config_by_name(args.config)
    if args.T:
        c = dataclasses.replace(c, T=args.T)
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, E, k, H, F = c.T, c.E, c.k, c.H, c.F
    lg = torch.from_numpy(W.make_layer_logits(c, 0, layers=1)[0]).to(dev)
    x = W.make_x(c, 0, 0, device=dev)
    w1, w3, w2 = W.make_weights(c, 0, device=dev)
    idx, w = M.moe_route(lg, k)
    go, perm, inv, xp = M.moe_dispatch(x, idx, E, None)
    ffn_ws = torch.empty(max(M.workspace_bytes(M.MOE_OP_EXPERT_FFN, T, k, E, H, F), 1024), dtype=torch.uint8,
                         device=dev)
    y = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    fwd = lambda: M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, c.act, y=y, workspace=ffn_ws)
    fwd()
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    dout = torch.randn((T, H), generator=g, device=dev).to(torch.bfloat16)
    f32 = dict(dtype=torch.float32, device=dev)
    gdt = torch.bfloat16 if args.wgrad_bf16 else torch.float32
    outs = (torch.empty((T, H), dtype=torch.bfloat16, device=dev), torch.empty((T, k), **f32),
            torch.empty((E, H, F), dtype=gdt, device=dev),
            torch.empty((E, H, F), dtype=gdt, device=dev) if c.act == "swiglu" else None,
            torch.empty((E, F, H), dtype=gdt, device=dev))
    ws = torch.empty(M.moe_ffn_backward_workspace_bytes(T, k, E, H, F), dtype=torch.uint8, device=dev)
    dl = torch.empty((T, E), **f32)

    def bwd():
        M.moe_ffn_backward(x, dout, w, y, perm, inv, go, None, w1, w3, w2, c.act, workspace=ws, out=outs,
                           wgrad_bf16=args.wgrad_bf16)
        M.moe_route_backward(lg, idx, outs[1], out=dl)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        e1.synchronize()
        M.moe_check()
        return e0.elapsed_time(e1) * 1e-3 / steps

    steps, warmup = max(args.steps, 1), max(args.warmup, 3)
    clk = ClockSampler(0)
    clk.start()
    t_bwd = timed(bwd, steps, warmup)
    clocks = clk.stop()
    t_fwd = timed(fwd, steps, warmup)
    fl_b = backward_flops(c)
    fl_f = (6 if c.act == "swiglu" else 4) * c.A * H * F
    # the burst bf16 rate bounds a timed region of well under a second at the
    # maximum clock; the sustained rate (measured under the power cap) is given beside it
    peak = peaks["bf16_tflops"]
    # bytes the backward must move at least: the weights read by the GEMM1
    # recompute, the dA and the dxp GEMMs (W1, W3 twice; W2 once), the fp32
    # weight gradients written, and its inputs and outputs (x, dout, y, dx)
    n1 = 2 if c.act == "swiglu" else 1
    gbytes = 2 if args.wgrad_bf16 else 4
    by_b = (2 * n1 + 1) * E * H * F * 2 + (n1 + 1) * E * H * F * gbytes + 3 * T * H * 2 + c.A * H * 2
    t_tensor = fl_b / (peak * 1e12)
    t_hbm = by_b / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    res = {
        "backward": c.name, "T": T, "E": E, "k": k, "H": H, "F": F, "act": c.act,
        "steps": steps, "warmup": warmup,
        "us_per_backward": round(t_bwd * 1e6, 1),
        "tokens_per_s": round(T / t_bwd, 1),
        "backward_tflops": round(fl_b / t_bwd / 1e12, 1),
        "backward_frac_of_burst_bf16": round(fl_b / t_bwd / 1e12 / peak, 3),
        "backward_frac_of_sustained_bf16": round(fl_b / t_bwd / 1e12 / peaks["bf16_tflops_sustained"], 3),
        "timed_region_s": round(t_bwd * steps, 3),
        "roofline": {"bound": bound, "flops": fl_b, "bytes": by_b,
                     "time_lower_bound_us": round(max(t_tensor, t_hbm) * 1e6, 1),
                     "frac": round(max(t_tensor, t_hbm) / t_bwd, 3),
                     "peaks": "burst bf16 and measured copy rate of MEASURED_PEAKS.json"},
        "us_forward_ffn": round(t_fwd * 1e6, 1),
        "forward_ffn_tflops": round(fl_f / t_fwd / 1e12, 1),
        "backward_over_forward_ffn": round(t_bwd / t_fwd, 2),
        "gpu_launches_per_backward": 8,
        "weight_gradients": "bf16" if args.wgrad_bf16 else "fp32",
        "peak": {"bf16_tflops": peak, "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                 "source": peaks["source"]},
        "clocks": clocks,
        "data": "synthetic: the config's logits, x and weights; dout ~ N(0,1) bf16",
    }
    return res


CROSSOVER_SHAPES = [(5120, 1536), (5120, 14336)]   # (H, F): GEMM2 is M x H x F


def run_crossover(args):
    """GroupGemm vs DenseGemm crossover (EPS-MoE review, analysis of the two
    GEMM forms over the shapes 512x5120x1536, 2048x5120x1536 and
    512x5120x14336, M x N x K): SwiGLU experts with H = 5120 and F = 1536 or
    14336 -- an expert's down projection is exactly the M x 5120 x F GEMM of
    those shapes -- each with M rows, through moe_expert_ffn on the grouped
    tcgen05 kernels (small_group_threshold 0) and on the small-batch
    weight-streaming kernel (threshold above M; rows beyond 64 are taken in
    64-row chunks, each streaming the weights again).  Two layer forms: one
    expert alone (the pages' single GEMMs; few tiles, so neither kernel fills
    the GPU at small M) and 32 experts of M rows each (a fine-grained layer's
    many small groups, the case the threshold decides).  Each timing: 3
    warm-up calls, then 20 calls, each after an L2 flush (weights and rows
    start in HBM), CUDA events around the call alone; median.  One JSON line
    per (H, F, experts) with the times per M and the faster path."""
    import torch
    import moe_expert_routing_02_b300 as M
    M.lib()
    peaks = load_peaks()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = L2Flush(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    forms = [(1, [16, 32, 48, 64, 96, 128, 192, 256, 512, 1024, 2048]), (32, [16, 32, 48, 64, 96, 128, 256, 512])]
    for H, F in CROSSOVER_SHAPES:
        for ne, rows in forms:
            w1 = (torch.randn((ne, H, F), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            w3 = (torch.randn((ne, H, F), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            w2 = (torch.randn((ne, F, H), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            wbytes = 3 * H * F * 2 * ne
            res = []
            for m in rows:
                A = m * ne
                xp = torch.randn((A, H), generator=g, device=dev).to(torch.bfloat16)
                go = torch.arange(0, A + 1, m, dtype=torch.int32, device=dev)
                y = torch.empty((A, H), dtype=torch.bfloat16, device=dev)
                ws = torch.empty(max(M.workspace_bytes(M.MOE_OP_EXPERT_FFN, A, 1, ne, H, F), 1024),
                                 dtype=torch.uint8, device=dev)
                row = {"M": m}
                for name, thr in (("grouped", 0), ("small_batch", 1 << 30)):
                    # the small-batch arm gives the small-batch kernels every SM (the
                    # library's default leaves that path off)
                    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, nsm if name == "small_batch" else 0)
                    fn = lambda: M.moe_expert_ffn(xp, go, None, None, w1, w3, w2, "swiglu", thr, y=y, workspace=ws)
                    for _ in range(3):
                        fn()
                    torch.cuda.synchronize()
                    ts = []
                    for _ in range(20):
                        flush()
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record()
                        fn()
                        e1.record()
                        e1.synchronize()
                        ts.append(e0.elapsed_time(e1) * 1e3)
                    M.moe_check()
                    M.moe_set_option(M.MOE_OPT_FFN_SMALL_SMS, 0)
                    ts.sort()
                    row[name + "_us"] = round(ts[len(ts) // 2], 1)
                flops = 6 * A * H * F
                row["faster"] = "small_batch" if row["small_batch_us"] < row["grouped_us"] else "grouped"
                row["grouped_tflops"] = round(flops / row["grouped_us"] / 1e6, 1)
                row["small_batch_weights_gbs"] = round(wbytes / row["small_batch_us"] / 1e3, 1)
                # lower bound of the call: weights once from HBM, or the flops at the burst bf16 rate
                row["bound_us"] = round(max(wbytes / (peaks["hbm_gbs"] * 1e3), flops / (peaks["bf16_tflops"] * 1e6)),
                                       1)
                res.append(row)
                del xp, y, ws
            cross = [r["M"] for r in res if r["faster"] == "grouped"]
            print(json.dumps({"crossover": f"{ne} expert(s) of M rows each, SwiGLU, H={H}, F={F} "
                                           f"(down projection M x {H} x {F})",
                              "experts": ne, "weights_bytes": wbytes, "rows": res,
                              "smallest_M_where_grouped_is_faster": min(cross) if cross else None,
                              "library_threshold": 64, "peaks": peaks["source"],
                              "timing": "median of 20 calls, L2 flushed (written, then read clean) before each, "
                                        "CUDA events"}), flush=True)
            del w1, w3, w2
            torch.cuda.empty_cache()
    return 0


def _top_overlap(p_pred, load, m=5):
    """Share of the m most loaded experts that are among the m most popular
    predicted ones (ties: lower expert first on both sides)."""
    import numpy as np
    pred = np.lexsort((np.arange(p_pred.size), -p_pred.astype(np.float64)))[:m]
    act = np.lexsort((np.arange(load.size), -load.astype(np.int64)))[:m]
    return len(set(pred.tolist()) & set(act.tolist())) / m


def _max_group_load(load, copies):
    """Largest replica-group row count when each expert's rows are split
    round-robin over its copies + 1 groups."""
    import numpy as np
    n = copies.astype(np.int64) + 1
    return int(np.max((load.astype(np.int64) + n - 1) // n))


def run_quality(args):
    """Next-layer prediction quality and prediction-driven replication on the
    workload's iteration stream (moe_gpt_stream: 200 iterations, Zipf skew
    ramping over the first 50, window s=10).  Per iteration i and layer
    j < L-1, the prediction for layer j+1 made after layer j was recorded is
    scored against layer j+1's routing in the same iteration: top-5 overlap
    (PopFetcher review: ~77% for the naive top-k gate at s = 10) and mean
    absolute error of the load proportions ("Prediction Is All MoE Needs":
    ~1.3%), for the plain window and decay factors 0.9 and 0.7.  Replication:
    the largest replica group of layer j+1 (rows, over the target A/E) with no
    replicas, with the replica table of moe_replicate_predicted on the
    prediction, and with the table of the layer's own histogram (known only
    after routing)."""
    import numpy as np
    import torch
    import moe_expert_routing_02_b300 as M
    from moe_expert_routing_02_b300 import workloads as W
    M.lib()
    c = W.config_by_name(args.config)
    dev = torch.device("cuda", 0)
    L, E, k, T = c.L, c.E, c.k, c.T
    A = T * k
    lams = [1.0, 0.9, 0.7]
    st = M.MoEStats(L, E, c.window)
    acc = {lam: [] for lam in lams}
    err = {lam: [] for lam in lams}
    grp = {"none": [], "predicted": [], "from_own_histogram": []}
    hist = torch.empty(E, dtype=torch.int32, device=dev)
    t0 = time.time()
    for it in range(args.quality_iters):
        lgs = W.make_layer_logits(c, it)
        prev = None
        preds = {}
        for j in range(L):
            idx, _ = M.moe_route(torch.from_numpy(lgs[j]).to(dev), k)
            M.moe_stats_update(st, it, j, idx, prev, hist_out=hist)
            h = hist.cpu().numpy()
            if j > 0:
                for lam in lams:
                    p = preds[lam]
                    acc[lam].append(_top_overlap(p, h))
                    err[lam].append(float(np.mean(np.abs(p.astype(np.float64) - h / h.sum()))))
                target = A / E
                _, cp, _, _ = M.moe_replicate_predicted(preds["p32"], A)
                own, _, _ = M.moe_replicate(hist, A)
                grp["none"].append(_max_group_load(h, np.zeros(E, np.int64)) / target)
                grp["predicted"].append(_max_group_load(h, cp.cpu().numpy()) / target)
                grp["from_own_histogram"].append(_max_group_load(h, own.cpu().numpy()) / target)
            if j < L - 1:
                preds = {}
                for lam in lams:
                    _, _, pn = M.moe_predict_decay(st, j, it, lam)
                    preds[lam] = pn.cpu().numpy()
                    if lam == 1.0:
                        preds["p32"] = pn
            prev = idx
    M.moe_check()
    n_per_it = L - 1
    stable = 50 * n_per_it   # iterations >= 50: the skew no longer drifts

    def summ(v):
        v = np.asarray(v, dtype=np.float64)
        return {"all": round(float(v.mean()), 4), "from_iteration_50": round(float(v[stable:].mean()), 4)}

    return {
        "quality": f"{c.name}: {args.quality_iters} iterations x {L - 1} layer pairs, window s={c.window}, "
                   f"T={T}, E={E}, top-{k}",
        "top5_accuracy": {f"lambda={lam}": summ(acc[lam]) for lam in lams},
        "load_proportion_mae_pct": {f"lambda={lam}": {kk: round(vv * 100, 3) for kk, vv in summ(err[lam]).items()}
                                    for lam in lams},
        "max_group_rows_over_target": {kk: summ(v) for kk, v in grp.items()},
        "pages_for_context": {"top5_accuracy": "about 77% (naive top-k gate, s=10; PopFetcher, 8-32 GPU clusters)",
                              "load_proportion_error": "about 1.3% / 1.8% (GPT3 350M, next 1000 / 2000 steps)"},
        "data": "synthetic (seeded Zipf-biased logits with inter-layer correlation)",
        "seconds": round(time.time() - t0, 1),
    }


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.crossover:
        return run_crossover(args)
    if args.quality:
        print(json.dumps(run_quality(args)), flush=True)
        return 0
    if args.backward:
        print(json.dumps(run_backward(args)), flush=True)
        return 0
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    rank, world, local = dist_init()
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass
    return 0


if __name__ == "__main__":
    sys.exit(main())
