#!/usr/bin/env python3
"""Benchmark: MoE dispatch + combine, microseconds per layer, on one GB300.

One step = one MoE layer's hot path over one batch of synthetic tokens:
(route +) count (k_layout) + scan (k_scan) -> dispatch pack/scatter -> [expert
stand-in, untimed] -> combine, launched with programmatic dependent launch. The
timed value is the device time of the layout + dispatch phase plus the combine
phase (CUDA events on the launching stream around each phase), with
L2 flushed (a 320 MB write, then a 320 MB read so that no dirty line of the
flush is written back inside a timed kernel) before the dispatch phase and
again before the combine phase of every step, so every phase starts cold.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config prefill|decode|...]
  python bench.py --impl reference ...   # the CPU oracle on the same workload

The default workload is the largest one that fits one GPU: prefill, 32 virtual
ranks x 4096 tokens, 256 experts, top-8, H 7168, FP8 dispatch with BF16
combine, per-expert capacity 5120 (1,048,576 assignments). The value is the
median over the timed steps.

Under torchrun (N > 1) every rank runs an independent replica (the path has no
cross-GPU exchange on one GPU per box) and rank 0 prints the max over ranks.
Prints ONE JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine us/layer (effective HBM GB/s vs GB300 peak in roofline)"
KERNEL_SOURCES = {"k_layout+k_scan": "layout.cu", "k_dispatch_bf16": "dispatch.cu",
                  "k_dispatch_fp8": "dispatch.cu", "k_combine": "combine.cu"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="threads of the multi-threaded oracle baseline (0: all host cores)")
    ap.add_argument("--dispatch", default="separate",
                    choices=["separate", "fused", "two_stage", "allgather", "fixed_slots"],
                    help="separate: layout kernels then the dispatch kernel; fused: one "
                         "persistent launch; two_stage: the pack + all-to-all-v comparator; "
                         "allgather: the all-tokens-to-every-rank comparator; fixed_slots: "
                         "fixed per-(source, expert) receive regions (no capacity)")
    ap.add_argument("--pipeline", type=int, default=0,
                    help="also time the token-chunked two-stream pipeline with N chunks")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="override T_r (a smaller case of the same workload, e.g. for ncu)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_init(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def max_over_ranks(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, p in zip(names, parts[3:7]):
                if p.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# measured peaks and committed ncu traffic
# ---------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_sha(kernel: str) -> str:
    """Fingerprint of a kernel's code: its .cu file and the headers it
    includes (transitively, from csrc/ and include/), with comments and
    whitespace removed, so that only a change of that code voids a
    measurement."""
    dirs = [os.path.join(ROOT, "combine_top_histogram_gb300", "csrc"), os.path.join(ROOT, "include")]
    seen, todo, parts = set(), [KERNEL_SOURCES[kernel]], []
    while todo:
        name = todo.pop(0)
        path = next((os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name))),
                    None)
        if name in seen or path is None:
            continue
        seen.add(name)
        with open(path, "rb") as f:
            text = f.read()
        text = re.sub(rb"/\*.*?\*/", b" ", text, flags=re.S)
        text = re.sub(rb"//[^\n]*", b" ", text)
        parts.append((name, re.sub(rb"\s+", b" ", text).strip()))
        todo += [m.decode() for m in re.findall(rb'#include "([^"]+)"', text)]
    h = hashlib.sha256()
    for name, code in sorted(parts):
        h.update(name.encode() + b"\0" + code)
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current source of that kernel for this workload; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    ent = tab.get(workload, {}).get(kernel)
    if not ent or ent.get("source_sha") != source_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_layer_seconds(wl, budget_s: float, max_layers: int = 50, threads: int = 1,
                         elems_target: float = 6.0e7):
    """Times the CPU oracle's route/layout + dispatch + combine (the expert
    stand-in is run untimed) on a bounded sample of the workload: the same
    per-token distribution with fewer tokens per rank when a full layer would
    take too long (about elems_target token-row elements, T*k*H). With
    threads > 1 the route, dispatch and combine run the unchanged oracle
    functions on token ranges, one thread each; the layout (one global stable
    sort) stays on one thread. Returns (seconds per full layer, sample
    description, layers, per-layer times)."""
    import numpy as np

    import oracle
    from combine_top_histogram_gb300 import workloads as W
    elems = wl.T * wl.k * wl.H
    scale = max(1.0, elems / elems_target)
    tr = max(1, int(wl.Tr / scale))
    sw = wl.scaled(wl.name + "_cpu_sample", Tr=tr)
    if wl.cap:
        sw = sw.scaled(sw.name, Tr=tr, cap=max(1, int(round(wl.cap * tr / wl.Tr))))
    inp = W.make_inputs(sw)
    fp8 = sw.dispatch_dtype == W.MOE_FP8_E4M3
    times = []
    t_start = time.perf_counter()
    while len(times) < max_layers and (time.perf_counter() - t_start) < budget_s or len(times) < 1:
        t0 = time.perf_counter()
        if inp.logits is not None:
            ids, w = oracle.route_topk(inp.logits, sw.k, threads=threads)
        else:
            ids, w = inp.ids, inp.w
        lay = oracle.layout(sw.P, sw.Tr, sw.E, sw.k, ids, sw.cap)
        if fp8:
            recv, sc, _ = oracle.dispatch_fp8(sw.P, sw.Tr, sw.E, sw.k, inp.x, w, ids, lay["inv"],
                                              sw.rows_max, threads=threads)
        else:
            recv, _ = oracle.dispatch_bf16(sw.P, sw.Tr, sw.E, sw.k, inp.x, w, ids, lay["inv"],
                                           sw.rows_max, threads=threads)
        t1 = time.perf_counter()
        if fp8:
            y = oracle.expert_dequant_fp8(recv, sc, threads=threads)
        else:
            c = inp.expert_scale if inp.expert_scale is not None else np.ones(sw.E, np.float32)
            y = oracle.expert_scale_bf16(sw.E, lay["expert_offset"], c, recv)
        t2 = time.perf_counter()
        oracle.combine(lay["inv"], w, y, sw.T, sw.k, threads=threads)
        t3 = time.perf_counter()
        times.append((t1 - t0) + (t3 - t2))
    per_layer = statistics.median(times) * (wl.Tr / tr)
    how = ("single-threaded C, -O2" if threads <= 1 else
           f"C, -O2, route/dispatch/combine on {threads} threads over token ranges, "
           "layout on one thread")
    sample = (f"{len(times)} oracle layers of {sw.T} tokens ({tr} per rank, same config), "
              f"median scaled x{wl.Tr / tr:.2f} to {wl.T} tokens; {how}")
    return per_layer, sample, len(times), times


def host_threads(args) -> int:
    return args.cpu_threads if args.cpu_threads > 0 else (os.cpu_count() or 1)


def run_reference(args, wl, rank, world):
    """The reference arm: the CPU oracle as it stands, on all host cores
    (token-range threads), one bounded sample of the workload per step, sized
    so that the whole --steps/--warmup run stays within a few minutes."""
    if rank != 0:
        return 0
    threads = host_threads(args)
    n = args.warmup + args.steps
    target = 6.0e7 * threads * min(1.0, 25.0 / max(1, n))
    per_step = []
    desc = None
    for i in range(n):
        s, desc, _, _ = oracle_layer_seconds(wl, budget_s=0.0, max_layers=1, threads=threads,
                                             elems_target=target)
        if i >= args.warmup:
            per_step.append(s)
    us = statistics.median(per_step) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": "us/layer",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dispatch_dtype == 0 else "fp8_e4m3+bf16",
        "data": "synthetic", "config": {"workload": wl.name},
        "cpu_baseline": {"value": round(us, 3), "unit": "us/layer", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(us, 3), "unit": "us/layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_ours(args, wl, rank, world, local):
    import numpy as np
    import torch

    from combine_top_histogram_gb300 import MoeLayer, accounting
    from combine_top_histogram_gb300 import binding as B
    from combine_top_histogram_gb300 import workloads as W

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    inp = W.make_inputs(wl)
    layer = MoeLayer(wl.P, wl.Tr, wl.E, wl.k, wl.H, wl.dispatch_dtype, wl.cap, str(dev))
    x = torch.from_numpy(inp.x.view(np.int16)).to(dev).view(torch.bfloat16)
    routed = inp.logits is not None
    if routed:
        logits = torch.from_numpy(inp.logits).to(dev)
        w = layer.w
    else:
        ids = torch.from_numpy(inp.ids).to(dev)
        w = torch.from_numpy(inp.w).to(dev)
    c = torch.from_numpy(inp.expert_scale).to(dev) if inp.expert_scale is not None else None
    # L2 flush: write 320 MB (evicts everything), then read another 320 MB so
    # the dirty lines of the write are written back here, outside the timed
    # region, and the next phase starts with a cold, clean L2.
    flush_w = torch.empty(320 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(80 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()

    def layout():
        if routed:
            layer.route_layout(logits, stream)
        else:
            layer.layout(ids, stream)

    def dispatch():
        if args.dispatch == "two_stage":
            layer.dispatch_two_stage(x, w, stream)
        elif args.dispatch == "allgather":
            layer.dispatch_allgather(x, w, stream)
        elif args.dispatch == "fixed_slots":
            layer.dispatch_fixed_slots(x, w, stream)
        elif args.dispatch == "separate":
            layer.dispatch(x, w, stream)

    if args.dispatch == "fused":  # layout and dispatch are one launch
        def layout():
            if routed:
                layer.layout_dispatch_fused(x, logits=logits, stream=stream)
            else:
                layer.layout_dispatch_fused(x, ids=ids, w=w, stream=stream)

    def step(ev, flush=True):
        """One layer; ev[0..3] bracket the layout+dispatch phase and the combine
        phase (no event between the programmatically dependent launches)."""
        if flush:
            flush_l2()
        ev[0].record(stream)
        layout()
        dispatch()
        ev[1].record(stream)
        layer.expert(c, stream)
        if flush:
            flush_l2()
        ev[2].record(stream)
        layer.combine(w, stream)
        ev[3].record(stream)

    def step_diag(ev):
        """The same layer with an event between every kernel (per-kernel times)."""
        flush_l2()
        ev[0].record(stream)
        layout()
        ev[1].record(stream)
        dispatch()
        ev[2].record(stream)
        layer.expert(c, stream)
        ev[5].record(stream)
        flush_l2()
        ev[3].record(stream)
        layer.combine(w, stream)
        ev[4].record(stream)

    def new_events(n):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]

    for ev in new_events(args.warmup):
        step(ev)
    torch.cuda.synchronize(dev)

    # cold: L2 flushed before each phase
    evs = new_events(args.steps)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for ev in evs:
            step(ev)
        torch.cuda.synchronize(dev)
    barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in evs]
    med_ms = statistics.median(step_ms)
    med_ms_all = max_over_ranks(med_ms, world)
    mean_ms_all = max_over_ranks(statistics.fmean(step_ms), world)

    # per-kernel breakdown (events between kernels; diagnostic, same workload)
    devs = new_events(min(args.steps, 50))
    for ev in devs:
        step_diag(ev)
    torch.cuda.synchronize(dev)
    lay_ms = [e[0].elapsed_time(e[1]) for e in devs]
    dis_ms = [e[1].elapsed_time(e[2]) for e in devs]
    com_ms = [e[3].elapsed_time(e[4]) for e in devs]
    exp_ms = [e[2].elapsed_time(e[5]) for e in devs]

    pipeline = None
    if args.pipeline > 0 and args.dispatch == "separate":
        # token-chunked two-stream pipeline, the whole layer incl. the expert
        # stand-in, against the sum of the same stages run one after another
        pevs = new_events(min(args.steps, 50) + 3)
        for i, ev in enumerate(pevs):
            flush_l2()
            ev[0].record(stream)
            if routed:
                layer.forward_pipelined(x, logits=logits, expert_scale=c, chunks=args.pipeline,
                                        stream=stream)
            else:
                layer.forward_pipelined(x, ids=ids, w=w, expert_scale=c, chunks=args.pipeline,
                                        stream=stream)
            ev[1].record(stream)
        torch.cuda.synchronize(dev)
        wall = statistics.fmean([e[0].elapsed_time(e[1]) for e in pevs[3:]])
        stages = statistics.fmean([a + b + x_ + d for a, b, x_, d in
                                   zip(lay_ms, dis_ms, exp_ms, com_ms)])
        pipeline = {"chunks": args.pipeline, "wall_us": round(wall * 1e3, 3),
                    "sum_stages_us": round(stages * 1e3, 3),
                    "sum_over_wall": round(stages / wall, 4),
                    "note": "whole layer incl. the expert stand-in; stages timed serially "
                            "with L2 flushed only before layout and combine"}

    # warm: no flushes (a layer right after the previous one; L2 keeps what fits)
    wevs = new_events(min(args.steps, 100))
    for ev in wevs:
        step(ev, flush=False)
    torch.cuda.synchronize(dev)
    warm_ms = statistics.median([e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in wevs])

    # end to end through the public API: pinned host inputs -> device, layer,
    # result -> pinned host, copies inside the timed region
    x_h = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    if routed:
        r_h = [torch.from_numpy(inp.logits).pin_memory()]
        r_d = [logits]
    else:
        r_h = [torch.from_numpy(inp.ids).pin_memory(), torch.from_numpy(inp.w).pin_memory()]
        r_d = [ids, w]
    out_h = torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory()
    h2d = x_h.numel() * 2 + sum(t.numel() * t.element_size() for t in r_h)
    d2h = out_h.numel() * 2
    e2e_ms = []
    # the first copies from freshly pinned gigabyte buffers run slowly, so the
    # end-to-end loop warms up for as many steps as the device-timed one
    e2e_warm = max(3, args.warmup)
    eevs = new_events(min(args.steps, 50) + e2e_warm)
    for i, ev in enumerate(eevs):
        flush_l2()
        ev[0].record(stream)
        B.moe_copy_h2d_async(x, x_h, stream)
        for a, b in zip(r_d, r_h):
            B.moe_copy_h2d_async(a, b, stream)
        layout()
        dispatch()
        ev[1].record(stream)
        layer.expert(c, stream)
        flush_l2()
        ev[2].record(stream)
        layer.combine(w, stream)
        B.moe_copy_d2h_async(out_h, layer.out, stream)
        ev[3].record(stream)
    torch.cuda.synchronize(dev)
    for ev in eevs[e2e_warm:]:
        e2e_ms.append(ev[0].elapsed_time(ev[1]) + ev[2].elapsed_time(ev[3]))
    e2e_us = max_over_ranks(statistics.median(e2e_ms) * 1e3, world)

    view = layer.layout_view()
    kept = int(view["totals"][0].item())
    # routing shape ("Expert Parallel: MoE Token ...", "Load skew amplifies
    # both compute and communication tails" and "What to record"): expert
    # imbalance I_e = max n_e / mean n_e, rank imbalance I_r = max L_r / mean,
    # local fraction = kept assignments whose expert lives on their source rank
    n_e = view["expert_count"].double().cpu()
    Cm = view["count_matrix"].double().cpu()
    load_r = Cm.sum(dim=0)
    routing_shape = {
        "I_e": round(float(n_e.max() / n_e.mean()), 4) if float(n_e.mean()) > 0 else None,
        "I_r": round(float(load_r.max() / load_r.mean()), 4) if float(load_r.mean()) > 0 else None,
        "local_fraction": round(float(Cm.diagonal().sum() / Cm.sum()), 4) if float(Cm.sum()) > 0 else None,
        "kept": kept, "dropped": int(view["totals"][1].item()),
        "masked": int(view["totals"][2].item()),
        "C_row_sums": [int(v) for v in Cm.sum(dim=1).tolist()],
        "C_col_sums": [int(v) for v in load_r.tolist()],
    }
    kb = accounting.hbm_bytes(wl.P, wl.Tr, wl.E, wl.k, wl.H, layer.fp8, rows=kept, routed=routed)
    pay = accounting.payload_bytes(wl.P, wl.Tr, wl.k, wl.H, layer.fp8, rows=kept)
    dkey = "k_dispatch_fp8" if layer.fp8 else "k_dispatch_bf16"
    lkey = "k_layout+k_scan"
    if args.dispatch == "two_stage":
        dkey = "two_stage(k_send_pos+" + dkey + "+k_a2av)"
    if args.dispatch == "allgather":
        dkey = "allgather(k_allgather+k_allgather_filter)"
    if args.dispatch == "fixed_slots":
        dkey = "fixed_slots(" + dkey + ")"
    if args.dispatch == "fused":
        lkey = "k_fused(route+layout+dispatch)"
        means = {lkey: statistics.fmean([a + b for a, b in zip(lay_ms, dis_ms)]),
                 "k_combine": statistics.fmean(com_ms)}
        bytes_of = {lkey: kb.layout + kb.dispatch, "k_combine": kb.combine}
    else:
        means = {lkey: statistics.fmean(lay_ms), dkey: statistics.fmean(dis_ms),
                 "k_combine": statistics.fmean(com_ms)}
        bytes_of = {lkey: kb.layout, dkey: kb.dispatch, "k_combine": kb.combine}
    dom = max(means, key=means.get)
    peak, peak_kind = hbm_peak()
    achieved = bytes_of[dom] / (means[dom] * 1e-3) / 1e9
    traffic = committed_traffic(dom, wl.name) if dom in KERNEL_SOURCES else None
    per_kernel_gbs = {k: round(bytes_of[k] / (v * 1e-3) / 1e9, 1) for k, v in means.items()}
    cpu = cpu_mt = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline and world == 1:
        s, desc, n, _ = oracle_layer_seconds(wl, args.cpu_seconds)
        cpu = {"value": round(s * 1e6, 1), "unit": "us/layer", "cores": 1, "kind": "oracle",
               "sample": desc}
        nt = host_threads(args)
        s, desc, n, _ = oracle_layer_seconds(wl, args.cpu_seconds, threads=nt)
        cpu_mt = {"value": round(s * 1e6, 1), "unit": "us/layer", "cores": nt, "kind": "oracle",
                  "sample": desc}
    value_us = med_ms_all * 1e3
    line = {
        "metric": METRIC, "value": round(value_us, 3), "unit": "us/layer",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(med_ms_all, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3+bf16" if layer.fp8 else "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "P": wl.P, "tokens_per_rank": wl.Tr, "E": wl.E,
                   "top_k": wl.k, "hidden": wl.H, "capacity": wl.cap,
                   "l2": "flushed (320 MB write, then 320 MB read) before the dispatch and "
                         "the combine phase of every timed step",
                   "replicas": world, "dispatch": args.dispatch},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": bytes_of[dom]},
        "cpu_baseline": cpu,
        "cpu_baseline_mt": cpu_mt,
        "e2e": {"value": round(e2e_us, 3), "unit": "us/layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (2 if args.dispatch == "fused" else 6 if args.dispatch == "two_stage"
                         else 5 if args.dispatch == "allgather" else 4) * args.steps,
        "clocks": clk.summary(),
        "per_kernel_us": {k: round(v * 1e3, 3) for k, v in means.items()},
        "per_kernel_gbs": per_kernel_gbs,
        "mean_us_per_layer": round(mean_ms_all * 1e3, 3),
        "assignments_per_s": round(world * wl.Na / (med_ms_all * 1e-3), 1),
        "effective_gbs": round((kb.layout + kb.dispatch + kb.combine) / (med_ms_all * 1e-3) / 1e9, 1),
        "payload_gbs": round(pay["total"] / (med_ms_all * 1e-3) / 1e9, 1),
        "warm_us_per_layer": round(warm_ms * 1e3, 3),
        "kept_rows": kept,
        "routing": routing_shape,
        "pipeline": pipeline,
        "host_cores": os.cpu_count(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    from combine_top_histogram_gb300 import workloads as W
    if args.config not in W.CONFIGS:
        raise SystemExit(f"unknown --config {args.config}; choose from {list(W.CONFIGS)}")
    wl = W.CONFIGS[args.config]
    if args.tokens_per_rank:
        tr = args.tokens_per_rank
        cap = W.prefill_capacity(wl.P * tr, wl.k, wl.E) if wl.cap else 0
        wl = wl.scaled(f"{wl.name}_tr{tr}", Tr=tr, cap=cap)
    rank, world, local = dist_init(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, wl, rank, world)
        return run_ours(args, wl, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
