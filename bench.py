#!/usr/bin/env python3
"""Throughput of the routed int4 MoE layer on B300: one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 80b-dec]
                    [--impl ours|reference]

One bench step = `--tokens` (default 1000) batch-1 decode tokens, each a full
moe_layer_forward pass of the layer (router GEMV, top-k, fused int4 gate/up SwiGLU, down +
weighted combine + gated shared expert) on its own seeded x, every expert
read by indirection through the shuffled slot table of an all-resident HBM
pool.  The step is captured once as a CUDA graph and replayed.  To keep the
weights from being served by the 126 MB L2, consecutive tokens rotate through
R full copies of the layer (R chosen so the rotating working set is at least
3x L2).

Reported: tokens/s (whole job, all ranks), the layer step's achieved HBM
bandwidth on algorithmic bytes (active expert bytes over the event-timed
duration of sampled layer calls) against the measured copy peak, the oracle's
CPU throughput on a bounded sample, and an end-to-end number through the
public C-ABI calls with pinned host buffers and copies inside the timed
region.  Multi-GPU runs are independent replicas (the layer does not shard
at batch 1); no collective touches the data path.

`--impl reference` times the CPU oracle instead (rank 0 only).
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from int4_routed_expert_06_b300 import synth  # noqa: E402

METRIC = "routed-MoE layer tokens/s (decode, 512e top-10 int4); HBM GB/s vs peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
KERNELS_PER_TOKEN = 3  # single-token path: router, gate/up SwiGLU (+ top-k), down + combine (+ top-k)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload_desc(shape) -> str:
    return (f"{shape.name}: routed MoE layer H={shape.hidden} E={shape.n_experts} top-{shape.top_k} "
            f"I={shape.inter} shared I={shape.shared_inter} sigmoid-gated, int4 affine g{shape.group} "
            f"{shape.qscale} scale/bias, {shape.act} x/y, batch-1 decode")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [c.strip() for c in line.split(",")]
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


# ---------------------------------------------------------------- CPU oracle

def oracle_tokens_per_s(layer_w, shape, xs, budget_s: float, max_tokens: int):
    """Time the CPU oracle on the first tokens of the seeded decode sequence."""
    from oracle import oracle as O
    L = O.Layer(layer_w, shape.group, shape.top_k)
    L.forward(xs[:1])  # compile / load outside the clock
    n, t0 = 0, time.perf_counter()
    while n < max_tokens and (time.perf_counter() - t0) < budget_s:
        L.forward(xs[n:n + 1])
        n += 1
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def run_reference(args, shape, rank):
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_layer(shape, device=dev)
    xs = synth.decode_xs(shape, max(args.steps + args.warmup, 1), device=dev)
    from oracle import oracle as O
    L = O.Layer(w, shape.group, shape.top_k)
    for j in range(args.warmup):
        L.forward(xs[j:j + 1])
    t0 = time.perf_counter()
    for j in range(args.steps):
        L.forward(xs[args.warmup + j:args.warmup + j + 1])
    dt = time.perf_counter() - t0
    v = args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(shape), "tokens_per_step": 1,
                                        "l2": "n/a (host)"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} seeded decode tokens (x seeds {synth.DECODE_X_SEED0 + args.warmup}+)"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="80b-dec", choices=["80b-dec", "35b-dec"])
    ap.add_argument("--tokens", type=int, default=1000, help="decode tokens per bench step")
    ap.add_argument("--replicas", type=int, default=0, help="layer copies to rotate through (0 = >= 3x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    assert args.warmup >= 0 and args.steps >= 1

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape = synth.SHAPES[args.workload]

    if args.impl == "reference":
        run_reference(args, shape, rank)
        return

    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    _build.build()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # ---- workload
    w = synth.make_layer(shape, device="cuda")
    slots = synth.shuffled_slots(shape.n_experts, shape.weight_seed)
    per_token = synth.active_expert_bytes(shape)
    router_bytes = shape.n_experts * shape.hidden * 2 + shape.hidden * 2
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    R = args.replicas if args.replicas > 0 else max(1, math.ceil(3 * l2 / (per_token + router_bytes)))
    dl = B.DeviceLayer(shape, w, slots, replicas=R)
    T = args.tokens
    xs = synth.decode_xs(shape, T, device="cuda")
    ys = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device="cuda")
    cfg = dl.cfg
    nb = B.moe_layer_workspace_bytes(cfg, 1)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

    def one_step():
        for j in range(T):
            B.moe_layer_forward(cfg, dl.struct(j % R), xs[j:j + 1], 1, ys[j:j + 1], None, None, None, ws, nb)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        one_step()  # eager warm-up: sets kernel attributes before capture
    torch.cuda.synchronize()
    assert B.moe_get_device_error(stream) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    # ---- timed region
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            start.record(stream)
            for _ in range(args.steps):
                graph.replay()
            end.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        if dist:
            dist.barrier()
    ms = start.elapsed_time(end)
    if B.moe_get_device_error(stream) != 0:
        raise RuntimeError("a kernel recorded a device error during the bench")
    ms_all = torch.tensor([ms], device="cuda")
    if dist:
        dist.all_reduce(ms_all, op=dist.ReduceOp.MAX)
    ms_max = float(ms_all.item())
    tokens_total = args.steps * T * world
    value = tokens_total / (ms_max / 1e3)

    # ---- end to end through the public calls: pinned host x in, pinned host y out
    e2e_steps = min(args.steps, 3)
    x_host = xs.cpu().pin_memory()
    y_host = torch.empty((T, shape.hidden), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(xs)
    y_dev = torch.empty_like(ys)
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            x_dev.copy_(x_host, non_blocking=True)
            for j in range(T):
                B.moe_layer_forward(cfg, dl.struct(j % R), x_dev[j:j + 1], 1, y_dev[j:j + 1], None, None, None,
                                    ws, nb)
            y_host.copy_(y_dev, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_all = torch.tensor([e2e_ms], device="cuda")
    if dist:
        dist.all_reduce(e2e_all, op=dist.ReduceOp.MAX)
    e2e_value = e2e_steps * T * world / (float(e2e_all.item()) / 1e3)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---- roofline of the layer step.  Its three kernels (router, gate/up
    # SwiGLU, down + combine) overlap under programmatic dependent launch, so
    # the unit timed is one whole layer call: the event-timed replays divided
    # by the calls they contain.
    peak, peak_kind = peaks()
    mean_us = ms * 1e3 / (args.steps * T)
    achieved = per_token / (mean_us * 1e-6) / 1e9
    step_gbs = achieved
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                traffic = json.load(f).get(args.workload)
        except Exception:
            traffic = None

    cpu = None
    if not args.no_cpu_baseline:
        v, n, dt = oracle_tokens_per_s(w, shape, xs, args.cpu_seconds, 400)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} of the {T} seeded decode tokens of one bench step ({dt:.1f} s, "
                         "single-threaded C, fp64)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(shape), "tokens_per_step": T, "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2: tokens rotate through {R} full layer copies "
                         f"({R * dl.stride * dl.n_slots / 1e9:.1f} GB; the weights {R} tokens touch are "
                         f"{R * (per_token + router_bytes) / 1e6:.0f} MB vs the {l2 / 1e6:.0f} MB L2)",
                   "graph": "one CUDA graph per step (route + experts calls per token)"},
        "active_expert_bytes_per_token": per_token,
        "hbm": {"achieved_gbs_step": step_gbs, "frac_measured_step": step_gbs / peak,
                "frac_nominal_8tbs_step": step_gbs / NOMINAL_HBM_GBS},
        "roofline": {"kernel": "decode layer call: router + gate/up SwiGLU + down/combine kernels, PDL-chained "
                               "(timed as one unit)",
                     "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "mean_us": mean_us,
                     "algorithmic_bytes_per_launch": per_token},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": x_host.numel() * 2,
                "d2h_bytes_per_step": y_host.numel() * 2,
                "how": "per step: one pinned H2D of the step's x, moe_layer_forward per token (eager, "
                       "no graph), one pinned D2H of y"},
        "clocks": clk.summary(),
        "gpu_launches": KERNELS_PER_TOKEN * T * args.steps,
        "wall_s": t_wall,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
