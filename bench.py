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

Reported: tokens/s (whole job, all ranks), the layer call's achieved HBM
bandwidth on algorithmic bytes (active expert bytes over the event-timed
mean duration of one layer call) against the measured copy peak, the oracle's
CPU throughput on a bounded sample (single-GPU runs), and an end-to-end number through the
public C-ABI calls with pinned host buffers and copies inside the timed
region.  Multi-GPU runs are independent replicas (the layer does not shard
at batch 1); no collective touches the data path.

`--impl reference` times the CPU oracle instead (rank 0 only).

`--workload 35b-dec`, `80b-dec-int8` and `35b-dec-int8` time the same decode
loop on the 35B-shaped layer and on both layers with affine int8 codes.

Five more workloads print their own line (not the default):

- `--workload 80b-stack-file`: the stack with the expert backing store on a
  file (one pread per missed expert, then one copy into its slot).

- `--workload 80b-pool-sweep`: tokens/s and hit rate of an 8-layer stack
  through the bounded pool (device-side policy) against pool size and
  routing skew, beside the all-resident stack.

- `--workload 80b-batch`: tokens/s of one 80B-shaped layer call of T = 1 ..
  64 tokens on each kernel path (generic kernels, tcgen05 grouped GEMMs, and
  the default choice).

- `--workload 80b-prefill`: one step = one 4096-token layer call (Zipf-skewed
  routing, tcgen05 grouped GEMMs); tokens/s and TFLOP/s on algorithmic flops
  against the measured bf16 peak.
- `--workload 80b-stack`: one step = one decode token through a 48-layer
  stack served from a bounded HBM slot pool (25% of each layer's experts,
  LFU+recency, misses filled from pinned host memory on a side stream);
  tokens/s, hit rate, misses and exposed copy time per token, the measured
  pinned host-to-device copy rate, and bit-identity of every layer output
  with an all-resident run of the same stack.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
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


def metric_of(shape) -> str:
    """The metric a workload's line reports (METRIC for the 80B decode layer)."""
    if shape.name == "80b-prefill":
        return (f"routed-MoE layer prefill tokens/s ({shape.tokens} tokens, {shape.n_experts}e "
                f"top-{shape.top_k} int4, Zipf-skewed routing)")
    if shape.name == "80b-stack":
        return "80B-stack decode tokens/s through a bounded HBM expert pool (25% of experts per layer)"
    return (f"routed-MoE layer tokens/s (decode, {shape.n_experts}e top-{shape.top_k} int{shape.bits}); "
            "HBM GB/s vs peak")


assert metric_of(synth.DEC_80B) == METRIC
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
KERNELS_PER_TOKEN = 3  # single-token path: router (+ x records), gate/up (top-k, SwiGLU), down (+ combine)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources of the kernels one prefill layer call launches (router GEMM and
# shared-gate GEMV, top-k, bucketing, the grouped-GEMM path)
PREFILL_SOURCES = ("router_gemm.cu", "kernels_decode.cu", "bucket.cu", "prefill.cu")


def sources_digest(names) -> str:
    """sha256 over the named kernel sources, concatenated in the given order."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "int4_routed_expert_06_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per layer call from the committed ncu capture, or None when
    the kernel sources have changed since the counters were taken."""
    if workload == "80b-prefill":
        srcs, rec = PREFILL_SOURCES, os.path.join(ROOT, "profiles", "prefill_layer_traffic.txt")
    else:
        srcs, rec = ("kernels_token.cu",), os.path.join(ROOT, "profiles", "decode_layer_traffic.txt")
    try:
        digest = sources_digest(srcs)
        with open(rec) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 5 and not line.startswith("#") and parts[0] == workload:
                    return int(parts[-1]) if parts[1] == digest else None
    except OSError:
        return None
    return None


def workload_desc(shape) -> str:
    if shape.name == "80b-prefill":
        mode = f"{shape.tokens}-token prefill, Zipf(s={shape.zipf_s}) router bias"
    elif shape.name == "80b-stack":
        mode = (f"{shape.layers}-layer stack, {shape.pool_slots} pool slots per layer, "
                f"Zipf(s={shape.zipf_s}) router bias, batch-1 decode")
    else:
        mode = "batch-1 decode"
    return (f"{shape.name}: routed MoE layer H={shape.hidden} E={shape.n_experts} top-{shape.top_k} "
            f"I={shape.inter} shared I={shape.shared_inter} sigmoid-gated, int{shape.bits} affine g{shape.group} "
            f"{shape.qscale} scale/bias, {shape.act} x/y, {mode}")


# ---------------------------------------------------------------- ranks

def max_over_ranks(x: float, dist=None, device: str = "cuda") -> float:
    """The largest x over all ranks of the process group (x itself without
    one): the job's time is its slowest replica's."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max / 1e3)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        # The timed region starts only once nvidia-smi has printed its first
        # sample: its start-up work in the driver otherwise lands inside it.
        self.first = ""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.first = self.proc.stdout.readline()
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                rest, _ = self.proc.communicate(timeout=5)
                self.out = rest  # the first sample was taken before the timed region
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

def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_tokens_per_s(layer_w, shape, xs, budget_s: float, max_tokens: int, threads: int = 1):
    """Time the CPU oracle on the first tokens of xs (one token a call), its
    loops over output rows on `threads` threads."""
    from oracle import oracle as O
    O.set_threads(threads)
    try:
        L = O.Layer(layer_w, shape.group, shape.top_k)
        L.forward(xs[:1])  # compile / load outside the clock
        n, t0 = 0, time.perf_counter()
        while n < max_tokens and (time.perf_counter() - t0) < budget_s:
            L.forward(xs[n:n + 1])
            n += 1
        dt = time.perf_counter() - t0
    finally:
        O.set_threads(1)
    return n / dt, n, dt


def cpu_baseline_of(layer_w, shape, xs, budget_s: float, max_tokens: int, what: str, per_token_factor: float = 1.0):
    """The oracle on all available host cores (OpenMP over output rows) and on
    one core, each on a bounded sample of xs; tokens/s divided by
    per_token_factor (the layers a token passes through)."""
    cores = host_cores()
    v, n, dt = oracle_tokens_per_s(layer_w, shape, xs, budget_s / 2, max_tokens, threads=cores)
    v1, n1, dt1 = oracle_tokens_per_s(layer_w, shape, xs, budget_s / 2, max_tokens, threads=1)
    return {"value": v / per_token_factor, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}: {n} tokens in {dt:.1f} s on {cores} cores (plain C, fp64, OpenMP over output "
                      f"rows)",
            "single_thread": {"value": v1 / per_token_factor, "cores": 1,
                              "sample": f"{n1} tokens in {dt1:.1f} s on one core"}}


def run_reference(args, shape, rank):
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_layer(shape, device=dev)
    n = max(args.steps + args.warmup, 1)
    if shape.name == "80b-prefill":  # tokens of the seeded 4096-token batch, one at a time
        xs = synth.make_x(shape, synth.PREFILL_X_SEED, device=dev)[:n]
    else:
        xs = synth.decode_xs(shape, n, device=dev)
    from oracle import oracle as O
    cores = host_cores()
    O.set_threads(cores)
    L = O.Layer(w, shape.group, shape.top_k)
    for j in range(args.warmup):
        L.forward(xs[j:j + 1])
    t0 = time.perf_counter()
    for j in range(args.steps):
        L.forward(xs[args.warmup + j:args.warmup + j + 1])
    dt = time.perf_counter() - t0
    O.set_threads(1)
    # a stack token is one pass through every layer: the oracle's per-layer
    # rate divided by the layer count (layer 0's weights stand for all)
    v = args.steps / dt / max(shape.layers, 1)
    print(json.dumps({
        "impl": "reference", "metric": metric_of(shape), "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(shape), "tokens_per_step": 1,
                                        "l2": "n/a (host)"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} seeded tokens, one a call, OpenMP over output rows on {cores} "
                                   f"cores" + (" (layer 0's weights stand for each of the stack's layers)"
                                               if shape.layers > 1 else "")},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- prefill

def prefill_flops(shape, T: int) -> int:
    """Algorithmic flops of one T-token layer call: router (E rows + shared
    gate), k routed and one shared SwiGLU expert per token (gate, up, down)."""
    H = shape.hidden
    per_tok = (2 * H * (shape.n_experts + 1) + shape.top_k * 6 * H * shape.inter
               + (6 * H * shape.shared_inter if shape.shared_inter else 0))
    return T * per_tok


def run_prefill(args, shape):
    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    _build.build()
    torch.cuda.set_device(0)
    T = shape.tokens
    w = synth.make_layer(shape, device="cuda")
    dl = B.DeviceLayer(shape, w, synth.shuffled_slots(shape.n_experts, shape.weight_seed))
    x = synth.make_x(shape, synth.PREFILL_X_SEED, device="cuda")
    y = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    cfg = dl.cfg
    nb = B.moe_layer_workspace_bytes(cfg, T)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # inputs were made on the default stream

    def step():
        B.moe_layer_forward(cfg, dl.struct(), x, T, y, None, idx, None, ws, nb, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert B.moe_get_device_error(stream) == 0
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("prefill_steps")  # lets a profiler select the timed launches
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    ms = start.elapsed_time(end) / args.steps
    if B.moe_get_device_error(stream) != 0:
        raise RuntimeError("a kernel recorded a device error during the bench")
    counts = torch.bincount(idx.flatten().long(), minlength=shape.n_experts)
    flops = prefill_flops(shape, T)
    tf = flops / (ms * 1e-3) / 1e12
    pk = peak_bf16()
    # end to end: pinned x in, pinned y out, around the same call
    xh, yh = x.cpu().pin_memory(), torch.empty_like(y, device="cpu").pin_memory()
    xd = torch.empty_like(x)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = min(args.steps, 5)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            xd.copy_(xh, non_blocking=True)
            B.moe_layer_forward(cfg, dl.struct(), xd, T, y, None, idx, None, ws, nb, stream)
            yh.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e = n_e2e * T / (e0.elapsed_time(e1) * 1e-3)
    cpu = None
    if not args.no_cpu_baseline:  # per token, on a bounded sample of the batch (the layer is per-token)
        cpu = cpu_baseline_of(w, shape, x, args.cpu_seconds, 200,
                              f"first tokens of the {T}-token batch, one a call; tokens/s of the batch "
                              "extrapolated per token")
    print(json.dumps({
        "metric": metric_of(shape),
        "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 MMA (f32 accumulate in TMEM)", "data": "synthetic",
        "config": {"workload": f"80b-prefill: T={T}, H={shape.hidden} E={shape.n_experts} top-{shape.top_k} "
                               f"I={shape.inter} shared I={shape.shared_inter}, int4 g{shape.group} f16 "
                               f"scale/bias, Zipf(s={shape.zipf_s}) router bias",
                   "l2": "inputs larger than L2: every step reads all 512 experts' weights (906 MB)",
                   "experts_used": int((counts > 0).sum()), "max_tokens_per_expert": int(counts.max()),
                   "min_tokens_per_used_expert": int(counts[counts > 0].min())},
        "roofline": {"kernel": "prefill layer call (router, top-k, bucketing, gather, tcgen05 grouped GEMMs "
                               "gate/up and down, combine), timed as one unit",
                     "bound": "tensor", "achieved": tf, "peak": pk[0], "peak_kind": pk[1], "unit": "TFLOP/s",
                     "frac": tf / pk[0], "traffic": recorded_traffic("80b-prefill"),
                     "traffic_note": "DRAM bytes of all kernels of one call (ncu, committed record)",
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": xh.numel() * 2,
                "d2h_bytes_per_step": yh.numel() * 2},
        "cpu_baseline": cpu,
        "clocks": clk.summary(),
    }), flush=True)


def peak_bf16():
    """Sustained dense bf16 TFLOP/s (a step timed inside a long loop)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured, sustained"
    except Exception:
        return 1400.0, "fallback, sustained"


# ---------------------------------------------------------------- stack

def layer_input(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    """The input of the next MoE layer in the stack workload: the residual
    stream x [T, H] scaled to unit RMS per token (fp32 arithmetic, result in
    x's dtype).  Workload chaining, not layer arithmetic: without a norm
    between layers the SwiGLU experts, whose output grows with the square of
    their input, drive a residual chain of random layers to overflow within a
    few dozen layers."""
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(dim=-1, keepdim=True) + eps)).to(x.dtype)


def host_bytes_available() -> int:
    avail = 0
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            v = f.read().strip()
        if v != "max":
            with open("/sys/fs/cgroup/memory.current") as f:
                cur = int(f.read().strip())
            avail = min(avail, int(v) - cur)
    except (OSError, ValueError):
        pass
    return avail


def run_stack(args, shape):
    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    from int4_routed_expert_06_b300.stack import PooledStack
    _build.build()
    torch.cuda.set_device(0)
    E, k = shape.n_experts, shape.top_k
    per_layer = E * synth.expert_bytes(shape)
    L = shape.layers
    fit = int(0.6 * host_bytes_available()) // per_layer
    if fit < L:
        L = max(1, fit)
    resident = []
    first = {}

    def weights(l):
        w = synth.make_layer(shape, seed=shape.weight_seed + l, device="cuda")
        resident.append(B.DeviceLayer(shape, w, torch.arange(E, dtype=torch.int32)))
        if l == 0:
            first["w"] = w
        return w

    t_build = time.perf_counter()
    st = PooledStack(shape, L, shape.pool_slots, weights, device_policy=True)
    t_build = time.perf_counter() - t_build
    n = args.warmup + args.steps
    x0 = synth.decode_xs(shape, n, seed0=synth.STACK_X_SEED0, device="cuda")
    Y = torch.empty((n, L, shape.hidden), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    st.workspace(1)

    def token(j):
        h = x0[j:j + 1]
        for l in range(L):
            st.layer_forward(l, layer_input(h), Y[j, l:l + 1], stream=stream)
            h = (h.float() + Y[j, l:l + 1].float()).to(torch.bfloat16)

    with torch.cuda.stream(stream):
        for j in range(args.warmup):  # eager: fills the pool, sets kernel attributes
            token(j)
    torch.cuda.synchronize()
    # the timed tokens, every layer of each, as one CUDA graph: the pool's
    # lookups and fills are kernels, so nothing waits on the host
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for j in range(args.warmup, n):
            token(j)
    torch.cuda.synchronize()
    s0 = st.stats()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            start.record(stream)
            graph.replay()
            end.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    ms = start.elapsed_time(end)
    s1 = st.stats()
    if B.moe_get_device_error() != 0:
        raise RuntimeError("a kernel recorded a device error during the bench")
    del graph
    d = {key: s1[key] - s0[key] for key in ("hits", "misses", "evictions", "bytes_filled", "lookups")}
    # the same tokens through all-resident layers, also one graph: timing, and
    # bit-identity of every layer output
    cfg = st.cfg
    nb = B.moe_layer_workspace_bytes(cfg, 1)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    YR = torch.empty_like(Y)

    def token_resident(j):
        h = x0[j:j + 1]
        for l in range(L):
            B.moe_layer_forward(cfg, resident[l].struct(), layer_input(h), 1, YR[j, l:l + 1], None, None, None,
                                ws, nb, stream)
            h = (h.float() + YR[j, l:l + 1].float()).to(torch.bfloat16)

    with torch.cuda.stream(stream):
        token_resident(0)
    torch.cuda.synchronize()
    graph_r = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_r, stream=stream):
        for j in range(args.warmup, n):
            token_resident(j)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        r0.record(stream)
        graph_r.replay()
        r1.record(stream)
    torch.cuda.synchronize()
    res_ms = r0.elapsed_time(r1)
    del graph_r
    diff = (YR[args.warmup:] != Y[args.warmup:]).reshape(args.steps * L, -1).any(dim=1)
    n_mism = int(diff.sum().item())
    # pinned host -> device copy rate for blob-sized copies (the fills' own size)
    blob = st.blob_bytes
    dst = torch.empty((64, blob), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        for rep in range(2):
            c0.record(side)
            for i in range(64):
                dst[i].copy_(st.backing[0, i, :blob], non_blocking=True)
            c1.record(side)
    torch.cuda.synchronize()
    h2d_gbs = 64 * blob / (c0.elapsed_time(c1) * 1e-3) / 1e9
    K = args.steps
    cpu = None
    if not args.no_cpu_baseline:  # layer 0's oracle per layer-token, over the stack's layers
        xin = torch.cat([layer_input(x0[j:j + 1]) for j in range(min(n, 64))])
        cpu = cpu_baseline_of(first["w"], shape, xin, args.cpu_seconds, 200,
                              f"layer 0 of the stack on its first layer inputs; tokens/s through {L} layers "
                              "= the per-layer rate / the layer count", per_token_factor=L)
    lookups = max(d["hits"] + d["misses"], 1)
    print(json.dumps({
        "metric": metric_of(shape),
        "value": K / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "s32/f32", "data": "synthetic",
        "config": {"workload": f"80b-stack: {L} layers (of {shape.layers}) x E={E} top-{k}, "
                               f"{shape.pool_slots} slots/layer, Zipf(s={shape.zipf_s}) router bias, "
                               "residual stream h_(l+1) = bf16(h_l + y_l), layer input bf16(h_l / rms(h_l)), batch-1 decode",
                   "layers_run": L, "layers_named": shape.layers,
                   "host_memory_note": (None if L == shape.layers else
                                        f"pinned backing store limited to {L} layers by host memory"),
                   "l2": f"pool {L * shape.pool_slots * st.stride / 1e9:.1f} GB and {L} resident layers, "
                         "far beyond L2", "build_s": t_build},
        "pool": {"policy": "LFU + recency, run on the device (lookup and fill kernels); timed tokens are one "
                           "CUDA graph", "hit_rate": d["hits"] / lookups, "misses_per_token": d["misses"] / K,
                 "fill_bytes_per_token": d["bytes_filled"] / K, "evictions": d["evictions"],
                 "added_us_per_token": (ms - res_ms) * 1e3 / K,
                 "fill_gbs_effective": d["bytes_filled"] / max((ms - res_ms) * 1e-3, 1e-9) / 1e9,
                 "pcie_h2d_gbs_blob_copies": h2d_gbs,
                 "copy_bound_us_per_token": d["bytes_filled"] / K / (h2d_gbs * 1e9) * 1e6},
        "resident": {"tokens_per_s": K / (res_ms * 1e-3),
                     "note": "same tokens, all experts resident, one CUDA graph"},
        "bit_identical_to_resident": n_mism == 0, "mismatched_layer_outputs": n_mism,
        "all_outputs_finite": bool(torch.isfinite(Y[args.warmup:].float()).all()),
        "layer_outputs_compared": K * L,
        "roofline": {"bound": "pcie", "achieved": d["bytes_filled"] / (ms * 1e-3) / 1e9,
                     "peak": h2d_gbs, "unit": "GB/s", "frac": d["bytes_filled"] / (ms * 1e-3) / 1e9 / h2d_gbs,
                     "traffic": None, "peak_kind": "measured in this run: 64 pinned blob copies"},
        "cpu_baseline": cpu,
        "clocks": clk.summary(), "wall_s": t_wall,
    }), flush=True)
    st.close()


# ---------------------------------------------------------------- policy study

POLICY_RULES = {"lfu_recency": 0, "lru": 1, "lfu": 2}  # MOE_POOL_* codes of the C ABI


def routing_trace(shape, layer: int, tokens: int):
    """Top-k expert ids [tokens, k] of one stack layer on unit-RMS Gaussian
    layer inputs.  The stack's own router weights and Zipf bias (synth's
    draws for that layer); the inputs stand in for the normalised residual
    stream, which also has unit RMS per token."""
    r = synth.make_router(shape, shape.weight_seed + layer, "cpu")
    g = torch.Generator().manual_seed(9000 + layer)
    x = torch.randn((tokens, shape.hidden), generator=g)
    logits = x @ r["w_router"].float().t()
    if r["router_bias"] is not None:
        logits = logits + r["router_bias"]
    return torch.topk(logits, shape.top_k, dim=1).indices.to(torch.int32)


def fs_type(path: str) -> str:
    """File-system type of the mount holding path (from /proc/mounts)."""
    best, typ = "", "unknown"
    try:
        real = os.path.realpath(path)
        with open("/proc/mounts") as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and real.startswith(parts[1]) and len(parts[1]) > len(best):
                    best, typ = parts[1], parts[2]
    except OSError:
        pass
    return typ


def run_stack_file(args, shape):
    """The stack served from the bounded pool with the backing store on a
    file (the storage tier below host memory): one pread per missed expert
    into pinned staging, then one copy into its slot; host-side policy,
    eager per-layer calls.  Layers limited by the free space of --tier-dir."""
    import shutil
    import tempfile
    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    from int4_routed_expert_06_b300.stack import PooledStack
    _build.build()
    torch.cuda.set_device(0)
    tdir = args.tier_dir or tempfile.gettempdir()
    E = shape.n_experts
    per_layer = E * ((synth.expert_bytes(shape) + 4095) // 4096 * 4096)
    L = max(1, min(8, int(0.5 * shutil.disk_usage(tdir).free) // per_layer))
    path = os.path.join(tdir, f"moe_stack_{os.getpid()}.qpack")
    try:
        t_build = time.perf_counter()
        st = PooledStack(shape, L, shape.pool_slots,
                         lambda l: synth.make_layer(shape, seed=shape.weight_seed + l, device="cuda"),
                         file_path=path, readers=args.readers)
        t_build = time.perf_counter() - t_build
        n = args.warmup + args.steps
        x0 = synth.decode_xs(shape, n, seed0=synth.STACK_X_SEED0, device="cuda")
        y = torch.empty((1, shape.hidden), dtype=torch.bfloat16, device="cuda")

        def token(j):
            h = x0[j:j + 1]
            for l in range(L):
                st.layer_forward(l, layer_input(h), y)
                h = (h.float() + y.float()).to(torch.bfloat16)

        for j in range(args.warmup):
            token(j)
        torch.cuda.synchronize()
        s0, f0 = st.stats(), B.slot_pool_file_stats(st.handle)
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for j in range(args.warmup, n):
            token(j)
        e1.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        ms = e0.elapsed_time(e1)
        s1, f1 = st.stats(), B.slot_pool_file_stats(st.handle)
        if B.moe_get_device_error() != 0:
            raise RuntimeError("a kernel recorded a device error during the bench")
        K = args.steps
        hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
        rb, rns = f1["bytes_read"] - f0["bytes_read"], f1["read_ns"] - f0["read_ns"]
        print(json.dumps({
            "metric": f"{L}-layer 80B-stack decode tokens/s with the expert backing store on a file",
            "value": K / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "s32/f32", "data": "synthetic",
            "config": {"workload": f"{L} layers x E={E} top-{shape.top_k} int4, {shape.pool_slots} slots/layer, "
                                   f"Zipf(s={shape.zipf_s}) router bias, batch-1 decode, backing store on a file",
                       "file_system": fs_type(tdir), "direct_io": f1["direct"], "readers": args.readers,
                       "file_gb": L * per_layer / 1e9, "build_s": t_build},
            "tier": {"hit_rate": hits / max(hits + misses, 1), "misses_per_token": misses / K,
                     "read_gbs": rb / max(rns * 1e-9, 1e-9) / 1e9, "read_ms_per_token": rns / 1e6 / K,
                     "bytes_read_per_token": rb / K},
            "wall_s": wall,
        }), flush=True)
        st.close()
    finally:
        if os.path.exists(path):
            os.remove(path)


def run_pool_sweep(args, shape):
    """Tokens/s of a stack of 80B-shaped layers served from the bounded pool
    (device-side LFU + recency, timed tokens as one CUDA graph) against the
    pool size (1/8, 1/4, 1/2 of each layer's experts) and the skew of the
    routing (router bias Zipf s = 0.6, 1.1, 1.6), with the all-resident stack
    on the same tokens beside each point."""
    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    from int4_routed_expert_06_b300.stack import PooledStack
    _build.build()
    torch.cuda.set_device(0)
    E = shape.n_experts
    L = min(8, max(1, int(0.4 * host_bytes_available()) // (E * synth.expert_bytes(shape))))
    base = [synth.make_layer(shape, seed=shape.weight_seed + l, device="cuda") for l in range(L)]
    zipfs, fracs = (0.6, 1.1, 1.6), (8, 4, 2)
    W, K = max(16, args.warmup), max(8, args.steps)
    x0 = synth.decode_xs(shape, W + K, seed0=synth.STACK_X_SEED0, device="cuda")
    stream = torch.cuda.Stream()

    def run_graph(fwd):
        with torch.cuda.stream(stream):
            for j in range(W):
                fwd(j)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(W, W + K):
                fwd(j)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return K / (e0.elapsed_time(e1) * 1e-3)

    y = torch.empty((1, shape.hidden), dtype=torch.bfloat16, device="cuda")
    table = []
    with ClockSampler(0) as clk:
        for zs in zipfs:
            sz = dataclasses.replace(shape, zipf_s=zs)
            ws_ = []
            for l in range(L):
                w = dict(base[l])
                w["router_bias"] = synth.zipf_router_bias(sz, shape.weight_seed + l, device="cuda")
                ws_.append(w)
            resident = [B.DeviceLayer(sz, ws_[l], torch.arange(E, dtype=torch.int32)) for l in range(L)]
            cfg = resident[0].cfg
            nb = B.moe_layer_workspace_bytes(cfg, 1)
            wsb = torch.empty(nb, dtype=torch.uint8, device="cuda")

            def fwd_res(j):
                h = x0[j:j + 1]
                for l in range(L):
                    B.moe_layer_forward(cfg, resident[l].struct(), layer_input(h), 1, y, None, None, None, wsb, nb,
                                        stream)
                    h = (h.float() + y.float()).to(torch.bfloat16)

            res_tps = run_graph(fwd_res)
            del resident
            for fr in fracs:
                st = PooledStack(sz, L, E // fr, lambda l: ws_[l], device_policy=True)
                st.workspace(1)

                def fwd_pool(j):
                    h = x0[j:j + 1]
                    for l in range(L):
                        st.layer_forward(l, layer_input(h), y, stream=stream)
                        h = (h.float() + y.float()).to(torch.bfloat16)

                s_0 = None
                with torch.cuda.stream(stream):
                    for j in range(W):
                        fwd_pool(j)
                torch.cuda.synchronize()
                s_0 = st.stats()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for j in range(W, W + K):
                        fwd_pool(j)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                tps = K / (e0.elapsed_time(e1) * 1e-3)
                s_1 = st.stats()
                if B.moe_get_device_error() != 0:
                    raise RuntimeError("a kernel recorded a device error during the pool sweep")
                hits, misses = s_1["hits"] - s_0["hits"], s_1["misses"] - s_0["misses"]
                table.append({"zipf_s": zs, "pool_fraction": 1.0 / fr, "slots_per_layer": E // fr,
                              "tokens_per_s": round(tps, 1), "hit_rate": round(hits / max(hits + misses, 1), 4),
                              "misses_per_token": round(misses / K, 2),
                              "resident_tokens_per_s": round(res_tps, 1)})
                del g
                st.close()
    head = next(r for r in table if r["zipf_s"] == 1.1 and r["pool_fraction"] == 0.25)
    print(json.dumps({
        "metric": f"{L}-layer 80B-stack decode tokens/s through the bounded pool against pool size and routing skew",
        "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": W,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s32/f32", "data": "synthetic",
        "config": {"workload": f"{L} layers x E={E} top-{shape.top_k} int4, batch-1 decode, pool 1/8, 1/4, 1/2 of "
                               "each layer's experts, router bias Zipf s = 0.6, 1.1, 1.6, LFU + recency on the device",
                   "value_at": "pool 1/4, Zipf s = 1.1",
                   "timing": "warm-up tokens eager, then the timed tokens (every layer) as one CUDA graph"},
        "sweep": table, "clocks": clk.summary(), "gpu_launches": None,
    }), flush=True)


def run_batch_sweep(args, shape):
    """Small decode batches: tokens/s of one 80B-shaped layer call at T = 1 ...
    64 on each kernel path (1: generic kernels, 2: tcgen05 grouped GEMMs from
    T = 2, 0: the default choice).  Each point is a CUDA graph of calls whose
    seeded x rotate through layer copies larger than L2 together."""
    from int4_routed_expert_06_b300 import binding as B
    from int4_routed_expert_06_b300 import build as _build
    _build.build()
    torch.cuda.set_device(0)
    w = synth.make_layer(shape, device="cuda")
    slots = synth.shuffled_slots(shape.n_experts, shape.weight_seed)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    layer_bytes = shape.n_experts * synth.expert_bytes(shape)
    R = args.replicas if args.replicas > 0 else max(2, math.ceil(3 * l2 / layer_bytes) + 1)
    dl = B.DeviceLayer(shape, w, slots, replicas=R)
    cfg = dl.cfg
    Ts = [1, 2, 4, 8, 16, 32, 64]
    calls = 8 * R
    stream = torch.cuda.Stream()
    table = []
    with ClockSampler(0) as clk:
        for T in Ts:
            xs = synth.make_x(shape, 4000 + T, T * calls, device="cuda")
            ys = torch.empty((T * calls, shape.hidden), dtype=torch.bfloat16, device="cuda")
            row = {"T": T}
            for path in (1, 2, 0):
                if T == 1 and path == 2:
                    continue
                B.moe_set_kernel_path(path)
                try:
                    nb = B.moe_layer_workspace_bytes(cfg, T)
                    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

                    def run():
                        for j in range(calls):
                            B.moe_layer_forward(cfg, dl.struct(j % R), xs[j * T:(j + 1) * T], T,
                                                ys[j * T:(j + 1) * T], None, None, None, ws, nb)

                    with torch.cuda.stream(stream):
                        run()
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        run()
                finally:
                    B.moe_set_kernel_path(0)
                with torch.cuda.stream(stream):
                    for _ in range(max(3, args.warmup)):
                        g.replay()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(args.steps):
                        g.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / (args.steps * calls)
                row[{1: "generic", 2: "grouped_gemm", 0: "default"}[path]] = {
                    "us_per_call": round(us, 2), "tokens_per_s": round(T / (us * 1e-6), 1)}
                del g
            table.append(row)
    if B.moe_get_device_error(stream) != 0:
        raise RuntimeError("a kernel recorded a device error during the sweep")
    best = max(r["default"]["tokens_per_s"] for r in table)
    line = {
        "metric": "routed-MoE layer tokens/s at small decode batches (80B layer, one call of T tokens)",
        "value": table[-1]["default"]["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 tensor-core GEMMs (grouped) / s32 dp4a and f32 (single-token, generic)", "data": "synthetic",
        "config": {"workload": workload_desc(shape).replace("batch-1 decode", "decode batches T = 1..64"),
                   "value_at": "T = 64, default path", "calls_per_graph": calls,
                   "l2": f"calls rotate through {R} layer copies ({R * layer_bytes / 1e9:.1f} GB)"},
        "sweep": table, "best_default_tokens_per_s": best,
        "clocks": clk.summary(), "gpu_launches": None,
    }
    print(json.dumps(line), flush=True)


def run_policy_study(args):
    """Hit rate of the slot pool's host policy (the library's own
    slot_pool_lookup) against pool fraction, Zipf skew and eviction rule, on
    routing traces of the 80B stack's layers.  Only lookups run: placeholder
    addresses stand in for the pool and backing store, which a lookup never
    touches."""
    import dataclasses
    from int4_routed_expert_06_b300 import binding as B

    base = synth.STACK_80B
    E = base.n_experts
    layers, warm, tokens = 4, 32, max(args.steps, 64)
    placeholder = 1 << 40  # 256-byte aligned, never dereferenced by a lookup
    cfg = B.config_for(base)
    stride = B.moe_blob_layout_get(cfg, base.inter).bytes
    rows = []
    t0 = time.perf_counter()
    for s in (0.0, 0.8, 1.1, 1.4):
        shape = dataclasses.replace(base, zipf_s=s)
        traces = [routing_trace(shape, l, warm + tokens).tolist() for l in range(layers)]
        for frac in (0.10, 0.25, 0.50):
            slots = int(round(frac * E))
            for rule, code in POLICY_RULES.items():
                p = B.slot_pool_create(cfg, layers, slots, placeholder, layers * slots * stride, placeholder,
                                       stride, side_stream=0)
                try:
                    B.slot_pool_set_policy(p, code)
                    for j in range(warm + tokens):
                        if j == warm:
                            s0 = B.slot_pool_stats(p)
                        for l in range(layers):
                            B.slot_pool_lookup(p, l, traces[l][j])
                    s1 = B.slot_pool_stats(p)
                finally:
                    B.slot_pool_destroy(p)
                hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
                rows.append({"zipf_s": s, "pool_fraction": frac, "slots": slots, "rule": rule,
                             "hit_rate": hits / max(hits + misses, 1), "misses_per_token_layer": misses / (tokens * layers)})
    dt = time.perf_counter() - t0
    head = next(r for r in rows if r["zipf_s"] == base.zipf_s and r["pool_fraction"] == 0.25
                and r["rule"] == "lfu_recency")
    print(json.dumps({
        "metric": "slot-pool hit rate against pool fraction, Zipf skew and eviction rule (host policy)",
        "value": head["hit_rate"], "unit": "hit rate", "higher_is_better": True,
        "steps": tokens, "warmup": warm, "data": "synthetic",
        "config": {"workload": f"80b-stack routers: E={E} top-{base.top_k}, {layers} layers, {tokens} tokens "
                               f"after {warm} warm-up tokens, unit-RMS Gaussian layer inputs",
                   "headline": "pool 25%, Zipf s=1.1, LFU+recency (the stack workload's setting)"},
        "table": rows, "host_s": dt,
    }), flush=True)


# ---------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="80b-dec",
                    choices=["80b-dec", "35b-dec", "80b-dec-int8", "35b-dec-int8", "80b-prefill", "80b-stack",
                             "80b-batch", "80b-pool-sweep", "80b-stack-file", "policy-study"])
    ap.add_argument("--tier-dir", default="", help="directory of the stack-file workload's backing file")
    ap.add_argument("--readers", type=int, default=4, help="read threads of the file tier")
    ap.add_argument("--tokens", type=int, default=1000, help="decode tokens per bench step")
    ap.add_argument("--replicas", type=int, default=0, help="layer copies to rotate through (0 = >= 3x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    assert args.warmup >= 0 and args.steps >= 1

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload == "policy-study":
        if rank == 0:  # host-only: the pool's eviction rules on routing traces
            run_policy_study(args)
        return
    if args.workload == "80b-batch":
        if rank == 0:
            run_batch_sweep(args, synth.DEC_80B)
        return
    if args.workload == "80b-pool-sweep":
        if rank == 0:
            run_pool_sweep(args, synth.STACK_80B)
        return
    if args.workload == "80b-stack-file":
        if rank == 0:
            run_stack_file(args, synth.STACK_80B)
        return
    shape = synth.SHAPES[args.workload]

    if args.impl == "reference":
        run_reference(args, shape, rank)
        return
    if shape.name in ("80b-prefill", "80b-stack"):
        if rank == 0:  # single-GPU workloads: other ranks have nothing to do
            (run_prefill if shape.name == "80b-prefill" else run_stack)(args, shape)
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
    ms_max = max_over_ranks(ms, dist, "cuda")
    value = job_tokens_per_s(args.steps * T, world, ms_max)

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
    e2e_value = job_tokens_per_s(e2e_steps * T, world, max_over_ranks(e0.elapsed_time(e1), dist, "cuda"))

    # ---- the same tokens through one copy of the layer (no rotation): the
    # router, the shared expert and repeatedly chosen experts can stay in L2
    graph1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph1, stream=stream):
        for j in range(T):
            B.moe_layer_forward(cfg, dl.struct(0), xs[j:j + 1], 1, ys[j:j + 1], None, None, None, ws, nb)
    steps1 = max(1, min(args.steps, 20))
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph1.replay()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        for _ in range(steps1):
            graph1.replay()
        n1.record(stream)
    torch.cuda.synchronize()
    nr_us = n0.elapsed_time(n1) * 1e3 / (steps1 * T)
    del graph1

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---- roofline of the layer step.  Its two kernels (router; experts:
    # top-k, gate/up SwiGLU, down + combine) overlap under programmatic
    # dependent launch, so the unit timed is one whole layer call: the
    # event-timed replays divided by the calls they contain.
    peak, peak_kind = peaks()
    mean_us = ms * 1e3 / (args.steps * T)
    achieved = per_token / (mean_us * 1e-6) / 1e9
    step_gbs = achieved
    traffic = recorded_traffic(args.workload)

    cpu = None
    if not args.no_cpu_baseline and world == 1:  # the oracle's baseline is an N = 1 figure
        cpu = cpu_baseline_of(w, shape, xs, args.cpu_seconds, 400,
                              f"first tokens of the {T} seeded decode tokens of one bench step")

    line = {
        "metric": metric_of(shape), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s32/f32", "data": "synthetic",
        "dtype_note": f"int{shape.bits} codes x 16-bit fixed-point activations in dp4a (s32), group scales and "
                      "sums in f32; bf16 x in, bf16 y out",
        "config": {"workload": workload_desc(shape), "tokens_per_step": T, "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2: tokens rotate through {R} full layer copies "
                         f"({R * dl.stride * dl.n_slots / 1e9:.1f} GB; the weights {R} tokens touch are "
                         f"{R * (per_token + router_bytes) / 1e6:.0f} MB vs the {l2 / 1e6:.0f} MB L2)",
                   "graph": "one CUDA graph per step (one moe_layer_forward per token)"},
        "active_expert_bytes_per_token": per_token,
        "hbm": {"achieved_gbs_step": step_gbs, "frac_measured_step": step_gbs / peak,
                "frac_nominal_8tbs_step": step_gbs / NOMINAL_HBM_GBS},
        "roofline": {"kernel": "decode layer call: router_tok_kernel + gateup_tok_kernel (top-k, gate/up "
                               "SwiGLU) + down_tok_kernel (down + combine), PDL-chained, timed as one unit",
                     "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "mean_us": mean_us,
                     "algorithmic_bytes_per_launch": per_token},
        "cpu_baseline": cpu,
        "non_rotated": {"tokens_per_s": job_tokens_per_s(T, world, nr_us * T / 1e3), "us_per_call": nr_us,
                        "achieved_gbs": per_token / (nr_us * 1e-6) / 1e9,
                        "note": "one layer copy for every token: weights that repeat across tokens (router, "
                                "shared expert, experts chosen again) may come from L2; not a roofline figure"},
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
