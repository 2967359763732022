#!/usr/bin/env python
"""Benchmark of the routed MoE layer forward on GB300.

Metric: microseconds per routed-MoE layer-step (lower is better) and the
weight bandwidth it implies against the measured HBM peak.  One step is one
pass of every layer of the workload (router, top-k, union, expert sweep,
blend) over one batch of `rows` token rows, replayed from one CUDA graph;
every layer streams its own distinct weights, so each step touches far more
bytes than the 129 MB L2 and no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--rows R] [--layers L] [--impl ours|reference]

N > 1 runs as one process per GPU under torch.distributed.run; every rank
runs an independent replica of the workload (the layer has no exchange step
on one GPU), the timed region is bracketed by barriers and the slowest rank's
time is reported.  --impl reference times the CPU oracle on the same
workload (rank 0 only).

The default line is the single-row decode workload (48 layers) with its down
projections in the t layout (the fused one-row form; --down-layout picks the
layout, "auto" = t for one-row workloads).  Beside it, under "rows_1_to_8",
the same measurement (µs per layer-step, mean union, roofline fraction of
the kernel alone and of the graph step) for the decode workload with
output-major down projections and with FP8 and BF16 expert matrices, for
the full sweep at every row count 1..8, for the speculative-verify rows 2, 3
and 4, and for the eight-row prefill sub-chunk with independent and with
correlated rows; under "variants", for the layer's variants: prefill calls
of 16 and 32 rows, an ungated and an absent shared expert, unnormalised
top-k weights, and the one-row GEMV lever.  The CPU-baseline leg times the
oracle on all host cores and on one, and compares its outputs for the first
and last timed layers of each workload with the GPU's (the "parity"
verdicts).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per routed-MoE layer-step & weight GB/s vs GB300 HBM peak, rows=1..8"
UNIT = "us/layer-step"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas: barrier and max over ranks only)
# ---------------------------------------------------------------------------

def dist_init(device_type: str = "cuda"):
    """(rank, world, local_rank); initialises the process group when the
    launcher set WORLD_SIZE > 1."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    if device_type == "cuda":
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist.init_process_group("gloo")
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(v: float, device_type: str = "cuda") -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return v
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if device_type == "cuda" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_us_per_unit(max_elapsed_ms: float, units_per_rank: int, world: int) -> float:
    """Whole-job microseconds per unit: every rank processed units_per_rank
    units within the slowest rank's time."""
    return max_elapsed_ms * 1000.0 / (units_per_rank * world)


# ---------------------------------------------------------------------------
# Bytes
# ---------------------------------------------------------------------------

def nvfp4_bytes(n: int, k: int) -> int:
    return n * k // 2 + n * k // 16


def layer_bytes(shape, rows: int, U: int) -> int:
    """Algorithmic bytes of one layer-step: every union expert's gate, up and
    down weights and scales once (+3 fp32 scale2), the shared expert, the
    router, the correction bias, the shared-expert gate vector, x and out."""
    H, E, I, Is = shape.hidden, shape.num_experts, shape.moe_inter, shape.shared_inter
    fmt = getattr(shape, "expert_fmt", "nvfp4")

    def mat(n, k):   # one expert matrix in the expert format
        return nvfp4_bytes(n, k) if fmt == "nvfp4" else n * k * (1 if fmt == "fp8" else 2)

    b = U * (3 * mat(I, H) + 12)
    if shape.has_shared:
        b += 3 * mat(Is, H) + 12
        if shape.shared_gated:
            b += H * 2
    b += E * H * 2 if shape.router_fmt == "bf16" else nvfp4_bytes(E, H) + 4
    if shape.scoring == "sigmoid":
        b += E * 4
    b += 2 * rows * H * 2
    return b


# ---------------------------------------------------------------------------
# Peaks, clocks, committed ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    d = os.path.join(ROOT, "routed_moe_decode_router_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str, rows: int, t_layout: bool = False,
                      fmt: str = "nvfp4", variant: str | None = None):
    """DRAM bytes per launch of `kernel` from a committed ncu summary under
    profiles/, if it was taken on the current kernel sources (else None).
    Lines of the t layout carry "layout=t" after the row count, lines of FP8
    or BF16 experts "fmt=fp8" / "fmt=bf16" after that, and lines of a layer
    variant (another shared expert, the GEMV lever, ...) "variant=<name>"
    after that."""
    src = kernel_source_hash()
    pat = re.compile(r"bench-traffic:\s*kernel=(\S+)\s+workload=(\S+)\s+rows=(\d+)\s+"
                     r"(?:layout=(\w+)\s+)?(?:fmt=(\w+)\s+)?(?:variant=(\S+)\s+)?"
                     r"bytes_per_launch=(\d+)\s+src=(\w+)")
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                m = pat.search(line)
                if (m and m.group(1) == kernel and m.group(2) == workload
                        and int(m.group(3)) == rows and (m.group(4) == "t") == t_layout
                        and (m.group(5) or "nvfp4") == fmt and m.group(6) == variant
                        and m.group(8) == src):
                    return int(m.group(7))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Workload
# ---------------------------------------------------------------------------

def build_workload(name, rows, n_layers, device, t_layout=False, fmt="nvfp4"):
    import dataclasses

    import torch
    from routed_moe_decode_router_gb300 import layer as L
    from routed_moe_decode_router_gb300 import synth
    wl = synth.WORKLOADS[name]
    shape = dataclasses.replace(wl.shape, expert_fmt=fmt)
    layers = [L.DeviceLayer(synth.make_layer(shape, wl.seed_base + l, device=device),
                            device=device, t_layout=t_layout) for l in range(n_layers)]
    xbuf = torch.empty((n_layers, rows, shape.hidden), dtype=torch.bfloat16, device=device)
    for l in range(n_layers):
        xbuf[l] = synth.make_rows(shape, rows, seed=wl.seed_base + 500 + l, device=device,
                                  corr=wl.corr)
    outbuf = torch.empty_like(xbuf)
    return wl, shape, layers, xbuf, outbuf


def workload_config(wl, shape, rows, n_layers, extra=None):
    c = {"workload": wl.name, "rows": rows, "layers": n_layers, "hidden": shape.hidden,
         "num_experts": shape.num_experts, "top_k": shape.top_k,
         "moe_inter": shape.moe_inter, "shared_inter": shape.shared_inter,
         "scoring": shape.scoring, "router": shape.router_fmt,
         "activations": "independent N(0,1)" if wl.corr is None
         else "correlated rows, a=%.3f" % wl.corr}
    if extra:
        c.update(extra)
    return c


def oracle_forward(dl, x, nthreads):
    """The oracle's forward of one layer on host rows x (copies only the
    experts it selects to the host); returns (result, seconds)."""
    from oracle import oracle
    _, ids, _ = oracle.OracleLayer(dl.layer, experts=()).route(x)
    ol = oracle.OracleLayer(dl.layer, experts=set(int(v) for v in ids.ravel()))
    t0 = time.perf_counter()
    res = ol.forward(x, nthreads=nthreads)
    return res, time.perf_counter() - t0


def parity_verdict(pairs):
    """GPU outputs against the oracle's on the same layers: bf16 out vs fp64
    out (rel-L2 <= 5e-3, max-abs <= 3e-2, the parity tests' bar) and the
    selected experts (ids of the workspace's last layer are not kept, so the
    comparison is on the outputs)."""
    import numpy as np
    rel, mab = [], []
    for got, want in pairs:
        g = got.float().cpu().numpy().astype(np.float64)
        rel.append(float(np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)))
        mab.append(float(np.abs(g - want).max()))
    return {"layers_checked": len(pairs), "max_rel_l2": max(rel), "max_abs": max(mab),
            "ok": bool(max(rel) <= 5e-3 and max(mab) <= 3e-2)}


def cpu_baseline(layers, xbuf, outbuf, rows, sample_s, nthreads, sample_1core_s):
    """The oracle as it stands on the host cores: whole layer forwards of
    the same workload, layer after layer, until `sample_s` seconds of oracle
    time have been spent (setup copies of the selected experts untimed), then
    the same on one core for `sample_1core_s`.  The first and last layers'
    oracle outputs are also compared with the GPU's outputs of the timed
    region (outbuf), as the parity verdict of the line."""
    from oracle import oracle
    oracle.build()
    spent, n, used = 0.0, 0, 1
    outs = {}
    for l, dl in enumerate(layers):
        x = xbuf[l].cpu()
        res, dt = oracle_forward(dl, x, nthreads)
        outs[l] = res["out"]
        spent += dt
        n += 1
        tasks = rows * (dl.shape.top_k + (1 if dl.shape.has_shared else 0))
        used = max(used, min(nthreads, tasks))
        if spent >= sample_s:
            break
    last = len(layers) - 1
    if last not in outs:
        outs[last], _ = oracle_forward(layers[last], xbuf[last].cpu(), nthreads)
        outs[last] = outs[last]["out"]
    spent1, n1 = 0.0, 0
    for l, dl in enumerate(layers):
        _, dt = oracle_forward(dl, xbuf[l].cpu(), 1)
        spent1 += dt
        n1 += 1
        if spent1 >= sample_1core_s:
            break
    return {"value": spent / n * 1e6, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "%d of the workload's layers, %d row(s) each, whole-layer oracle "
                      "forwards on %d host threads" % (n, rows, used),
            "value_1core": spent1 / n1 * 1e6,
            "sample_1core": "%d layers on one host thread" % n1,
            "parity": parity_verdict([(outbuf[0], outs[0]), (outbuf[last], outs[last])])}


def time_graph(layers, xbuf, outbuf, ws, rows, steps, warmup, stream, gemv=False):
    """One CUDA graph over every layer of the workload; µs per layer-step of
    `steps` replays after `warmup` (events on the launching stream).  Returns
    (graph, elapsed ms, per-layer union sizes)."""
    import torch
    from routed_moe_decode_router_gb300 import layer as L
    U = []
    with torch.cuda.stream(stream):
        for l, dl in enumerate(layers):
            L.forward(dl, xbuf[l], ws, out=outbuf[l], gemv=gemv)
            _, _, uni = L.read_routing(dl, ws, rows)
            U.append(uni["U"])
    stream.synchronize()
    if ws.status() != 0:
        raise RuntimeError("device status set during setup")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l, dl in enumerate(layers):
            L.forward(dl, xbuf[l], ws, out=outbuf[l], gemv=gemv)
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(steps):
        g.replay()
    ev1.record()
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    return g, ev0.elapsed_time(ev1), U


def time_kernels(layers, xbuf, outbuf, ws, rows, steps, stream, gemv=False):
    """Mean duration of the layer kernel alone: events recorded around each
    launch on the launching stream (layers back to back, no overlap)."""
    import torch
    from routed_moe_decode_router_gb300 import native as N
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in layers]
    for row in evs:                  # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    stream.synchronize()
    kern_ms = 0.0
    with torch.cuda.stream(stream):
        for _ in range(steps):
            for l, dl in enumerate(layers):
                N.moe_forward_timed(dl.config(gemv=gemv), dl.weights, xbuf[l].data_ptr(),
                                    outbuf[l].data_ptr(), rows, ws.ptr, ws.nbytes,
                                    stream.cuda_stream, [e.cuda_event for e in evs[l]])
            stream.synchronize()
            for l in range(len(layers)):
                kern_ms += evs[l][0].elapsed_time(evs[l][1])
    return kern_ms / (steps * len(layers))


@dataclasses.dataclass(frozen=True)
class Extra:
    """One further measured workload: a named workload at `rows` rows over
    `layers` layers, optionally with the activations of another workload,
    the t layout, another expert format, the GEMV lever, or MoeShape fields
    overridden ((name, value) pairs; `variant` names the change)."""
    workload: str
    rows: int
    layers: int
    corr_from: str | None = None
    t_layout: bool = False
    fmt: str = "nvfp4"
    gemv: bool = False
    shape: tuple = ()
    variant: str | None = None


# Further workloads measured beside the headline line (the metric is quoted
# for rows = 1..8): the decode workload with output-major down projections
# and with FP8 and BF16 experts, the full sweep at every row count 1..8, the
# speculative-verify rows 2, 3 and 4, and the eight-row prefill sub-chunk
# with independent and with correlated rows.  Fewer layers than the full
# stacks, each still far more distinct weight bytes per step than the
# 129 MB L2.  Consecutive lines of the same layer stack share one build.
EXTRA_CONFIGS = (
    [Extra("decode_h2048_e128", 1, 48),
     Extra("decode_h2048_e128", 1, 48, fmt="fp8"),
     Extra("decode_h2048_e128", 1, 48, fmt="bf16"),
     Extra("sweep_h4096_e160", 1, 16, t_layout=True)]
    + [Extra("sweep_h4096_e160", r, 16) for r in range(2, 9)]
    + [Extra("verify_h4096_e256", r, 16) for r in (2, 3, 4)]
    + [Extra("prefill8_h2048_e512", 8, 16),
       Extra("prefill8_h2048_e512", 8, 16, corr_from="verify_h4096_e256")])

# The layer's variants, each measured once: an ungated and an absent shared
# expert and unnormalised top-k weights (decode, t layout), the one-row GEMV
# lever (decode, both layouts), and calls of 16 and 32 rows (prefill: two
# and four 8-row sub-chunks plus the call's union; their algorithmic bytes
# count the call's union once, while each sub-chunk sweeps its own union).
VARIANT_CONFIGS = [
    Extra("prefill8_h2048_e512", 16, 16, variant="rows16"),
    Extra("prefill8_h2048_e512", 32, 8, variant="rows32"),
    Extra("decode_h2048_e128", 1, 48, t_layout=True, shape=(("shared_gated", False),),
          variant="ungated_shared"),
    Extra("decode_h2048_e128", 1, 48, t_layout=True, shape=(("has_shared", False),),
          variant="no_shared"),
    Extra("decode_h2048_e128", 1, 48, t_layout=True, shape=(("norm_topk_prob", False),),
          variant="no_norm"),
    Extra("decode_h2048_e128", 1, 48, gemv=True, variant="gemv_lever"),
    Extra("decode_h2048_e128", 1, 48, t_layout=True, gemv=True, variant="gemv_lever_t"),
]


def launches_per_layer(shape, rows: int, t_layout: bool) -> int:
    """Kernel launches of one moe_forward: one per sub-chunk (min(8, 64/k)
    rows; one row with the t layout), plus the union kernel when a call has
    more than one sub-chunk."""
    cr = 1 if t_layout else min(8, 64 // shape.top_k)
    n = (rows + cr - 1) // cr
    return n + (1 if n > 1 else 0)


def use_t_layout(choice: str, rows: int) -> bool:
    return choice == "t" or (choice == "auto" and rows == 1)


def measure_extra(ex: Extra, steps, warmup, dev, stream, peak, nthreads, with_parity,
                  cache=None):
    """µs per layer-step, mean union, roofline fractions (kernel alone and
    graph step) and, on rank 0, the parity verdict of one extra workload.
    `cache` (a dict) keeps the last layer stack for the next line of the
    same stack."""
    import torch
    from routed_moe_decode_router_gb300 import layer as L
    from routed_moe_decode_router_gb300 import synth
    name, rows, n_layers, t_layout, fmt, gemv = (ex.workload, ex.rows, ex.layers, ex.t_layout,
                                                 ex.fmt, ex.gemv)
    wl = synth.WORKLOADS[name]
    shape = dataclasses.replace(wl.shape, expert_fmt=fmt, **dict(ex.shape))
    corr = wl.corr if ex.corr_from is None else synth.WORKLOADS[ex.corr_from].corr
    cache = {} if cache is None else cache
    key = (name, fmt, t_layout, ex.shape, n_layers)
    if cache.get("key") != key:
        cache.clear()
        torch.cuda.empty_cache()
        cache["layers"] = [L.DeviceLayer(synth.make_layer(shape, wl.seed_base + l, device=dev),
                                         device=dev, t_layout=t_layout) for l in range(n_layers)]
        cache["key"] = key
    layers = cache["layers"]
    xbuf = torch.empty((n_layers, rows, shape.hidden), dtype=torch.bfloat16, device=dev)
    for l in range(n_layers):
        xbuf[l] = synth.make_rows(shape, rows, seed=wl.seed_base + 500 + l, device=dev,
                                  corr=corr)
    outbuf = torch.empty_like(xbuf)
    ws = L.Workspace(shape, device=dev, t_layout=t_layout)
    _, ms, U = time_graph(layers, xbuf, outbuf, ws, rows, steps, warmup, stream, gemv=gemv)
    us = ms * 1000.0 / (steps * n_layers)
    kern_ms = time_kernels(layers, xbuf, outbuf, ws, rows, max(1, min(steps, 10)), stream,
                           gemv=gemv)
    bytes_per_layer = sum(layer_bytes(shape, rows, u) for u in U) / n_layers
    out = {"workload": name, "rows": rows, "layers": n_layers,
           "down_layout": "t (input-major)" if t_layout else "output-major",
           "expert_fmt": fmt,
           "activations": "independent N(0,1)" if corr is None
           else "correlated rows, a=%.3f" % corr,
           "us_per_layer_step": round(us, 3), "union_mean": round(sum(U) / len(U), 3),
           "algorithmic_bytes_per_layer": int(bytes_per_layer),
           "kernel_us": round(kern_ms * 1000.0, 3),
           "roofline_frac_kernel": round(bytes_per_layer / (kern_ms * 1e-3) / 1e9 / peak, 4),
           "roofline_frac_graph": round(bytes_per_layer / (us * 1e-6) / 1e9 / peak, 4),
           "launches_per_layer": launches_per_layer(shape, rows, t_layout),
           "traffic": committed_traffic("moe_layer_kernel", name, rows, t_layout, fmt,
                                        ex.variant)}
    if ex.variant:
        out["variant"] = ex.variant
        out["shape_changes"] = {k: v for k, v in ex.shape}
        out["gemv_lever"] = gemv
    if with_parity:
        from oracle import oracle
        oracle.build()
        pairs = []
        for l in (0, n_layers - 1):
            res, _ = oracle_forward(layers[l], xbuf[l].cpu(), nthreads)
            pairs.append((outbuf[l], res["out"]))
        out["parity"] = parity_verdict(pairs)
    if ws.status() != 0:
        raise RuntimeError("device status set while timing %s" % name)
    del layers, xbuf, outbuf, ws
    return out


def run_ours(args, rank, world, local):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from routed_moe_decode_router_gb300 import synth
    wl0 = synth.WORKLOADS[args.workload]
    rows = args.rows or max(wl0.rows)
    n_layers = args.layers or wl0.layers
    t_layout = use_t_layout(args.down_layout, rows) and args.expert_fmt == "nvfp4"
    wl, shape, layers, xbuf, outbuf = build_workload(args.workload, rows, n_layers, dev, t_layout,
                                                     args.expert_fmt)
    from routed_moe_decode_router_gb300 import layer as L
    ws = L.Workspace(shape, device=dev, t_layout=t_layout)
    stream = torch.cuda.Stream(device=dev)

    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    g, elapsed, U = time_graph(layers, xbuf, outbuf, ws, rows, args.steps, args.warmup, stream,
                               args.gemv)
    clocks = sampler.stop()
    max_elapsed = max_over_ranks(elapsed)
    value = aggregate_us_per_unit(max_elapsed, args.steps * n_layers, world)
    ms_per_step = max_elapsed / args.steps

    # kernel timing pass: the same layers, events around each layer kernel
    kernel_ms = time_kernels(layers, xbuf, outbuf, ws, rows, max(1, min(args.steps, 20)), stream,
                             args.gemv)
    step_bytes = sum(layer_bytes(shape, rows, u) for u in U)
    peak, peak_kind = hbm_peak()
    achieved = step_bytes / n_layers / (kernel_ms * 1e-3) / 1e9
    traffic = committed_traffic("moe_layer_kernel", args.workload, rows, t_layout,
                                args.expert_fmt)

    # end to end through the public API with host buffers
    x_host = xbuf.cpu().pin_memory()
    out_host = torch.empty(outbuf.shape, dtype=outbuf.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 200))
    torch.cuda.synchronize()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(e2e_steps):
        xbuf.copy_(x_host, non_blocking=True)
        g.replay()
        out_host.copy_(outbuf, non_blocking=True)
    t1.record()
    t1.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1))
    e2e_value = aggregate_us_per_unit(e2e_ms, e2e_steps * n_layers, world)
    # the same end to end with one eager public-API call per layer (no
    # graph): the host side of every call (binding, argument checks, launch)
    # is inside the timed region too
    eager_steps = max(1, min(args.steps, 50))
    for l, dl in enumerate(layers):   # warm-up of the eager path
        L.forward(dl, xbuf[l], ws, out=outbuf[l], gemv=args.gemv)
    torch.cuda.synchronize()
    barrier()
    t0.record()
    for _ in range(eager_steps):
        xbuf.copy_(x_host, non_blocking=True)
        for l, dl in enumerate(layers):
            L.forward(dl, xbuf[l], ws, out=outbuf[l], gemv=args.gemv)
        out_host.copy_(outbuf, non_blocking=True)
    t1.record()
    t1.synchronize()
    eager_ms = max_over_ranks(t0.elapsed_time(t1))
    eager_value = aggregate_us_per_unit(eager_ms, eager_steps * n_layers, world)
    if ws.status() != 0:
        raise RuntimeError("device status set during the timed region")

    layer_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16" if args.expert_fmt == "bf16" else "f16")
                 + " mma / f32 accumulate (%s weights, bf16 activations)" % args.expert_fmt,
        "data": "synthetic (seeded N(0,0.02) weights encoded as %s, bf16 activations)"
                % args.expert_fmt.upper(),
        "config": workload_config(wl, shape, rows, n_layers, {
            "gemv_lever": int(args.gemv and rows == 1),
            "expert_fmt": args.expert_fmt,
            "down_layout": "t (input-major)" if t_layout else "output-major",
            "union_mean": round(sum(U) / len(U), 3),
            "l2": "no flush: each step streams %.2f GB of distinct weights (L2 129 MB)"
                  % (step_bytes / 1e9),
            "graph": "one CUDA graph of %d layers, one persistent kernel each, "
                     "PDL-chained" % n_layers,
            "parallelism": "replicas" if world > 1 else "single GPU"}),
        "weight_gbs": round(layer_gbs, 1),
        "weight_frac_of_peak": round(layer_gbs / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "moe_layer_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": int(step_bytes / n_layers),
                     "kernel_us": round(kernel_ms * 1000, 3),
                     "frac_graph_step": round(layer_gbs / peak, 4),
                     "note": "frac: the kernel timed alone (events around each launch, no "
                             "overlap with the previous layer); frac_graph_step: the same "
                             "bytes over the graph-replayed layer-step, where programmatic "
                             "dependent launch overlaps consecutive layers"},
        "e2e": {"value": round(e2e_value, 4), "unit": UNIT,
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(out_host.numel() * 2),
                "path": "graph replay of the public API calls",
                "eager_value": round(eager_value, 4),
                "eager_path": "one Python-level moe_forward per layer per step, no graph"},
        "gpu_launches": n_layers * args.steps * launches_per_layer(shape, rows, t_layout),
        "clocks": clocks,
    }
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if do_cpu:
        line["cpu_baseline"] = cpu_baseline(layers, xbuf, outbuf, rows, args.cpu_sample_s,
                                            os.cpu_count() or 1, args.cpu_1core_s)
    del layers, xbuf, outbuf, ws, g
    torch.cuda.empty_cache()
    if not args.no_extra and args.workload == "decode_h2048_e128" and not args.rows \
            and not args.layers:
        cache = {}
        line["rows_1_to_8"] = [
            measure_extra(ex, args.steps, args.warmup, dev, stream, peak, os.cpu_count() or 1,
                          do_cpu, cache)
            for ex in EXTRA_CONFIGS]
        line["variants"] = [
            measure_extra(ex, args.steps, args.warmup, dev, stream, peak, os.cpu_count() or 1,
                          do_cpu, cache)
            for ex in VARIANT_CONFIGS]
        cache.clear()
        torch.cuda.empty_cache()
    return line


def run_reference(args, rank, world):
    """The CPU oracle timed on the host cores on the same workload: each
    step is one whole layer forward (the layers in turn)."""
    if rank != 0:
        return None
    import torch
    from oracle import oracle
    from routed_moe_decode_router_gb300 import synth
    oracle.build()
    wl = synth.WORKLOADS[args.workload]
    shape = wl.shape
    rows = args.rows or max(wl.rows)
    n_layers = args.layers or wl.layers
    device = "cuda" if torch.cuda.is_available() else "cpu"
    nthreads = os.cpu_count() or 1
    budget_s = args.reference_budget_s
    need = min(n_layers, args.steps + args.warmup)
    prepared = []
    for l in range(need):
        weights = synth.make_layer(shape, wl.seed_base + l, device=device)
        x = synth.make_rows(shape, rows, seed=wl.seed_base + 500 + l, device=device,
                            corr=wl.corr).cpu()
        _, ids, _ = oracle.OracleLayer(weights, experts=()).route(x)
        prepared.append((oracle.OracleLayer(weights, experts=set(int(v) for v in ids.ravel())),
                         x))
        del weights
    for i in range(args.warmup):
        ol, x = prepared[i % len(prepared)]
        ol.forward(x, nthreads=nthreads)
    times = []
    t_start = time.perf_counter()
    for i in range(args.steps):
        ol, x = prepared[(args.warmup + i) % len(prepared)]
        t0 = time.perf_counter()
        ol.forward(x, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    value = sum(times) / len(times) * 1e6
    tasks = rows * (shape.top_k + (1 if shape.has_shared else 0))
    cores = min(nthreads, tasks)
    sample = ("%d timed whole-layer oracle forwards (%d row(s), %d distinct layers)"
              % (len(times), rows, len(prepared)))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": len(times), "steps_requested": args.steps,
        "warmup": args.warmup, "ms_per_step": round(value / 1000.0, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) weights quantised to NVFP4, bf16 activations)",
        "config": workload_config(wl, shape, rows, n_layers),
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_h2048_e128")
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-s", type=float, default=10.0)
    ap.add_argument("--cpu-1core-s", type=float, default=5.0)
    ap.add_argument("--gemv", action="store_true",
                    help="one-row layers on the CUDA-core GEMV variant (gemv_lever = 1)")
    ap.add_argument("--expert-fmt", choices=["nvfp4", "fp8", "bf16"], default="nvfp4",
                    help="expert matrix format (the t layout is NVFP4 only)")
    ap.add_argument("--down-layout", choices=["auto", "t", "output"], default="auto",
                    help="down projections in the t layout (the fused one-row form) or "
                         "output-major; auto = t for one-row workloads")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the extra rows=1..8 workloads beside the headline line")
    ap.add_argument("--reference-budget-s", type=float, default=150.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and world_env != args.gpus:
        ap.error("--gpus %d needs torch.distributed.run with %d processes"
                 % (args.gpus, args.gpus))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, rank, world_env)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    rank, world, local = dist_init("cuda")
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
