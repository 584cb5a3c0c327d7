"""Decode-step bench for the grouped-KV decode path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

One step = every layer of the workload: gqa_decode_step (the append fused
into the decode attention; --separate: gqa_kv_append then gqa_decode_attn)
through the C ABI, on one stream, with all inputs resident in HBM.  Timing:
W untimed steps, then K steps between a barrier + synchronize on both sides,
CUDA events on the launching stream, max over ranks.  Prints one JSON line
(rank 0).  Under torchrun each rank runs an independent replica on its own
GPU (the units are independent; no data-path collective): weak scaling.

The default workload is the Llama-3-70B-shaped decode step (80 layers,
b=32, h=64, g=8, d=128, 8192 cached tokens, bf16): 80 GiB of K/V, far
larger than L2, so no flush is needed between steps.

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload (the reference arm: there is no other implementation).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("decode-attn KV GB/s and % of GB300 HBM peak; layer-steps/sec at "
          "Llama-3-70B shape")
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; barrier and max-over-ranks only)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own replica of the workload."""
    return base_seed + 100 * rank


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


def smi_id(local_index: int) -> str:
    """nvidia-smi --id for torch's device index (through CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        items = [v.strip() for v in vis.split(",") if v.strip()]
        if local_index < len(items):
            return items[local_index]
    return str(local_index)


# ---------------------------------------------------------------------------
# byte counts
# ---------------------------------------------------------------------------
def step_bytes(cfg, lens, n: int = 1) -> dict:
    from gqa_kv_cache_append_gb300.inputs import layer_bytes
    attn = layer_bytes(cfg, lens, n)
    append = 2 * cfg.b * n * cfg.g * (cfg.d + cfg.dv) * cfg.elt  # read + write of the new rows
    return {"attn_per_layer": attn, "append_per_layer": append,
            "step": cfg.layers * (attn + append)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def profiled_traffic(kernel_src: str, workload: str, n: int = 1):
    """dram bytes per launch from the committed ncu summary of the kernel in
    `kernel_src` (profiles/<kernel>_<workload>.md), if it was taken on the
    current kernel source (matched by hash), else None."""
    tag = workload if n == 1 else f"{workload}_n{n}"
    kernel = os.path.splitext(os.path.basename(kernel_src))[0]
    path = os.path.join(ROOT, "profiles", f"{kernel}_{tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_hash and m_bytes):
        return None
    if kernel_source_hash(kernel_src) != m_hash.group(1):
        return None
    return int(m_bytes.group(1))


def kernel_source_hash(kernel_src: str) -> str:
    """sha256 of the kernel's source followed by the device header it
    includes (gqa_device.cuh, next to it: the tile walker, the merge
    protocol and the barrier helpers live there)."""
    h = hashlib.sha256(open(kernel_src, "rb").read())
    header = os.path.join(os.path.dirname(kernel_src), "gqa_device.cuh")
    if os.path.exists(header):
        h.update(open(header, "rb").read())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(cfg, target_s: float = 12.0, max_units: int = 4096, n: int = 1):
    """Time the float64 oracle's decode step on whole units (one sequence, one
    KV head, its r query heads; n new tokens each) of layer 0 of the
    workload, drawn on the CPU with the same generator recipe, until about
    target_s seconds of work.  Returns (GB/s of algorithmic bytes, seconds,
    units, bytes)."""
    import torch
    import oracle
    from gqa_kv_cache_append_gb300.inputs import make_layer, make_layer_multi, seq_lens_for
    import dataclasses

    lens = seq_lens_for(cfg)
    one = dataclasses.replace(cfg, b=1, layers=1)
    done_units, done_bytes, spent = 0, 0, 0.0
    i = 0
    while spent < target_s and done_units < max_units:
        L = int(lens[i % len(lens)])
        sub = dataclasses.replace(one, seed=cfg.seed * 7919 + i)
        if n == 1:
            x = make_layer(sub, 0, "cpu", lens=np.array([L], dtype=np.int32))
        else:
            x = make_layer_multi(sub, n, 0, "cpu", lens=np.array([L], dtype=np.int32))

        def np_(t):
            t = t.contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), "bf16"
            return t.numpy(), ("f16" if t.dtype == torch.float16 else "f32")
        tag = np_(x["q"])[1]
        arrs = [np_(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
        t0 = time.perf_counter()
        if n == 1:
            oracle.decode_step(*arrs, np.array([L]), cfg.g, cfg.scale, dtype=tag)
        else:
            oracle.decode_step_multi(*arrs, np.array([L]), cfg.g, cfg.scale, dtype=tag)
        spent += time.perf_counter() - t0
        done_units += cfg.g
        done_bytes += (L * cfg.g + n * cfg.h) * (cfg.d + cfg.dv) * cfg.elt
        i += 1
    return done_bytes / spent / 1e9, spent, done_units, done_bytes


def blas_threads() -> int:
    # numpy.einsum without `optimize` runs its own single-threaded loops
    return 1


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, local_rank, world):
    import torch
    from gqa_kv_cache_append_gb300 import binding as B
    from gqa_kv_cache_append_gb300.inputs import (make_layer, make_layer_multi,
                                                  make_layer_weights, projection_bytes,
                                                  seq_lens_for, to_paged, workload)
    import dataclasses

    n = args.tokens
    full_layer = args.layer
    paged = args.paged
    if (full_layer or paged) and n > 1:
        raise SystemExit("--layer and --paged run one new token per step")
    if full_layer and paged:
        raise SystemExit("--layer uses the contiguous cache")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    base = workload(args.workload)
    if args.g:
        base = dataclasses.replace(base, g=args.g)
    if args.h:
        base = dataclasses.replace(base, h=args.h)
    if args.b:
        base = dataclasses.replace(base, b=args.b)
    if args.cap:
        base = dataclasses.replace(base, cap=args.cap)
    if args.layers:
        base = dataclasses.replace(base, layers=min(args.layers, base.layers))
    if args.dtype:
        base = dataclasses.replace(base, dtype=args.dtype)
    if args.d:
        base = dataclasses.replace(base, d=args.d, scale=1.0 / math.sqrt(args.d))
    if args.dv:
        base = dataclasses.replace(base, d_v=args.dv)
    if (full_layer or paged) and base.dv != base.d:
        raise SystemExit("--layer and --paged use one head dim")
    if n > 1:
        # n new tokens per step: the workload's shapes with plain N(0, 1) data
        base = dataclasses.replace(base, kind="plain")
    lens = seq_lens_for(base)
    # a workload whose layers all fit in L2 is rotated through independent
    # replicas (extra layers of the same shape) until one step streams at
    # least 4x the L2 size, so every step reads K/V from HBM
    from gqa_kv_cache_append_gb300.inputs import layer_bytes as _lb, layer_flops
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_layer = _lb(base, lens, n) + (projection_bytes(base) if full_layer else 0)
    if base.layers * per_layer < 4 * l2 and not args.layers:
        base = dataclasses.replace(base, layers=-(-4 * l2 // per_layer))
    cfg = dataclasses.replace(base, seed=replica_seed(base.seed, rank))
    layers = [make_layer(cfg, l, dev) if n == 1 else make_layer_multi(cfg, n, l, dev)
              for l in range(cfg.layers)]
    if paged:
        # the caches become block pools with a shuffled block table
        for l, x in enumerate(layers):
            x["k_cache"], x["v_cache"], x["table"] = to_paged(
                x["k_cache"], x["v_cache"], paged, seed=cfg.seed * 1000 + l)
    if full_layer:
        # the layer's input is x; q / k_new / v_new come from the projections
        for l, x in enumerate(layers):
            for key in ("q", "k_new", "v_new"):
                del x[key]
            x.update(make_layer_weights(cfg, l, dev))
    # the step's per-layer inputs and outputs live in one packed buffer each
    # (layer-major), so the end-to-end leg moves them with one copy apiece
    packed = {}
    for key in (("x",) if full_layer else ("q", "k_new", "v_new")):
        packed[key] = torch.stack([x[key] for x in layers]).contiguous()
        for l, x in enumerate(layers):
            x[key] = packed[key][l]
    out_shape = (cfg.b, cfg.h, cfg.dv) if n == 1 else (cfg.b, n, cfg.h, cfg.dv)
    if full_layer:
        out_shape = (cfg.b, cfg.D)
    out_all = torch.empty((cfg.layers, *out_shape), dtype=cfg.torch_dtype, device=dev)
    outs = [out_all[l] for l in range(cfg.layers)]
    # --graph: the step is captured once in a CUDA graph and replayed; the
    # capture needs a stream of its own (and calls warmed up on it first)
    stream = torch.cuda.Stream(dev) if args.graph else torch.cuda.current_stream(dev)
    torch.cuda.set_stream(stream)
    sb = step_bytes(cfg, lens, n)
    if full_layer:
        sb["proj_per_layer"] = projection_bytes(cfg)
        sb["step"] += cfg.layers * sb["proj_per_layer"]
    early = 0 if args.ordered else B.GQA_STEP_EARLY_STREAM
    # --cuda-cores: the CUDA-core kernel on shapes the tensor-core kernel takes
    cuda_cores = B.GQA_STEP_CUDA_CORES if args.cuda_cores else 0
    if cuda_cores and (args.separate or full_layer):
        raise SystemExit("--cuda-cores applies to the fused step calls")

    def layer_call(l, x):
        if full_layer:
            B.gqa_decode_layer(x["x"], x["P_q"], x["P_k"], x["P_v"], x["P_o"], x["k_cache"],
                               x["v_cache"], x["seq_lens"], cfg.b, cfg.D, cfg.h, cfg.g, cfg.d,
                               cfg.d, cfg.scale, outs[l], flags=early, stream=stream)
        elif paged:
            B.gqa_decode_step_paged(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                    x["table"], x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.dv,
                                    cfg.scale, outs[l], flags=early | cuda_cores, stream=stream)
        elif n > 1:
            if args.separate:
                B.gqa_kv_append_multi(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                      x["seq_lens"], cfg.b, n, cfg.g, cfg.d, cfg.dv, stream=stream)
                B.gqa_decode_attn_multi(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b,
                                        n, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.scale, outs[l],
                                        stream=stream)
            else:
                B.gqa_decode_step_multi(x["q"], x["k_new"], x["v_new"], x["k_cache"],
                                        x["v_cache"], x["seq_lens"], cfg.b, n, cfg.h, cfg.g,
                                        cfg.d, cfg.dv, cfg.scale, outs[l],
                                        flags=early | cuda_cores, stream=stream)
        elif args.separate:
            B.gqa_kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"],
                            cfg.b, cfg.g, cfg.d, cfg.dv, stream=stream)
            B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b,
                              cfg.h, cfg.g, cfg.d, cfg.dv, cfg.scale, outs[l], stream=stream)
        else:
            # layers are independent buffers and seq_lens is fixed for the
            # step, so each layer may start streaming while the one before
            # finishes (GQA_STEP_EARLY_STREAM's contract)
            B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                              x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.scale,
                              outs[l], flags=early | cuda_cores, stream=stream)

    def step(ev=None):
        for l, x in enumerate(layers):
            if ev is not None:
                ev[l][0].record(stream)
            layer_call(l, x)
            if ev is not None:
                ev[l][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert B.gqa_device_status(stream) == 0
    run_step = step
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        run_step = graph.replay
        for _ in range(args.warmup):
            run_step()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing: K steps back to back, CUDA events on the
    # launching stream around the whole region.  Nothing is recorded between
    # the layer calls: an event between two launches would remove the
    # overlap their programmatic dependency allows.  Each step is only its
    # layer calls, so the time of one call is the step time / layers. ----
    clocks = ClockSampler(smi_id(dev.index))
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        run_step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(dist, dev)
    ms_local = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(dist, ms_local)
    attn_avg_ms = ms / cfg.layers
    # ---- the same calls one at a time, events around each (no overlap) ----
    n_iso = max(1, min(args.steps, 5))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)]
            for _ in range(cfg.layers)] for _ in range(n_iso)]
    for k in range(n_iso):
        step(evs[k])
    torch.cuda.synchronize(dev)
    iso_ms = max_over_ranks(dist, float(np.mean([e[0].elapsed_time(e[1])
                                                 for per in evs for e in per])))
    # ---- per-step spread: the same steps with an event between steps ----
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    sev[0].record(stream)
    for k in range(args.steps):
        run_step()
        sev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    step_times = [sev[k].elapsed_time(sev[k + 1]) for k in range(args.steps)]
    # ---- the append and the attention as separate calls (the one-token,
    # contiguous, projection-free step): each timed over all layers ----
    split = None
    if n == 1 and not paged and not full_layer:
        def timed(fn):
            for _ in range(2):
                for l, x in enumerate(layers):
                    fn(l, x)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                for l, x in enumerate(layers):
                    fn(l, x)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / (args.steps * cfg.layers)

        app_ms = timed(lambda l, x: B.gqa_kv_append(
            x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.g,
            cfg.d, cfg.dv, stream=stream))
        att_ms = timed(lambda l, x: B.gqa_decode_attn(
            x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.dv,
            cfg.scale, outs[l], stream=stream))
        split = {
            "append_us_per_call": round(app_ms * 1000, 3),
            "append_bytes_per_call": sb["append_per_layer"],
            "attn_only_us_per_call": round(att_ms * 1000, 3),
            "attn_only_gbs": round(sb["attn_per_layer"] / (att_ms * 1e-3) / 1e9, 2),
            "attn_only_frac_of_measured": None,  # filled below
            "how": "gqa_kv_append alone and gqa_decode_attn alone, each back to back over all "
                   "layers (no early streaming)",
        }
    status = B.gqa_device_status(stream)

    # ---- end to end: every step copies all layers' q, k_new, v_new in from
    # pinned host memory (one copy per tensor), runs the layers, and copies
    # all outputs back ----
    host_in = {k: v.cpu().pin_memory() for k, v in packed.items()}
    host_out = torch.empty_like(out_all, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for key, t in host_in.items():
            packed[key].copy_(t, non_blocking=True)
        for l, x in enumerate(layers):
            layer_call(l, x)
        host_out.copy_(out_all, non_blocking=True)

    run_e2e = e2e_step
    if args.graph:
        e2e_step()
        torch.cuda.synchronize(dev)
        graph_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_e2e, stream=stream):
            e2e_step()
        run_e2e = graph_e2e.replay
    for _ in range(max(1, args.warmup)):
        run_e2e()
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run_e2e()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps)
    status |= B.gqa_device_status(stream)

    if rank != 0:
        return None
    peaks = measured_peaks()
    call_bytes = sb["attn_per_layer"] + sb["append_per_layer"] + sb.get("proj_per_layer", 0)
    achieved = call_bytes / (attn_avg_ms * 1e-3) / 1e9
    plan = B.gqa_decode_plan(cfg.b, n, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.cap, cfg.dtype,
                             flags=cuda_cores)
    src = os.path.join(ROOT, "gqa_kv_cache_append_gb300", "csrc",
                       "decode_tc.cu" if plan["tensor_core"] else "decode_simt.cu")
    # the committed ncu summary covers the named workload's own shapes only
    reshaped = any(v is not None for v in (args.g, args.h, args.b, args.cap, args.d, args.dv,
                                           args.dtype)) or args.cuda_cores
    traffic = (None if (full_layer or reshaped)
               else profiled_traffic(src, args.workload + (f"_paged{paged}" if paged else ""), n))
    # per layer: the decode call's kernels (decode, plus combine when the
    # split partials are merged apart), + 2 projections or + 1 separate append
    launches_per_step = (plan["kernels"] + (2 if full_layer else (1 if args.separate else 0))
                         ) * cfg.layers
    value = world * sb["step"] / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded N(0,1), shapes of the workload)",
        "config": {
            "workload": cfg.name, "layers": cfg.layers, "b": cfg.b, "h": cfg.h, "g": cfg.g,
            "d_head": cfg.d, "d_v": cfg.dv, "seq_len": int(np.max(lens)), "cap": cfg.cap,
            "sum_seq_lens": int(np.sum(lens)),
            "kernel": "tensor cores" if plan["tensor_core"] else "CUDA cores",
            "l2": "inputs larger than L2: every step streams all layers' K/V "
                  f"({sb['step'] / 2**30:.2f} GiB, L2 {l2 / 2**20:.0f} MiB)",
            "parallelism": f"replicas x{world}",
            "launch": "CUDA graph" if args.graph else "stream",
            "tokens_per_step": n,
            "scope": "whole layer: projections + append + attention" if full_layer
                     else "append + attention",
            "kv_layout": f"paged, block {paged} rows, shuffled block table" if paged
                         else "contiguous",
        },
        "layer_steps_per_s": round(world * cfg.layers / (ms * 1e-3), 1),
        "attn_tflops_per_gpu": round(layer_flops(cfg, lens, n) / (attn_avg_ms * 1e-3) / 1e12, 2),
        "layer_call_gbs_per_gpu": round(achieved, 2),
        "pct_of_nominal_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": ("gqa_decode_layer (proj_tc_kernel x2 + " if full_layer else "")
                      + ("gqa_kv_append + gqa_decode_attn" if args.separate else "gqa_decode_step")
                      + ("_multi" if n > 1 else "") + ("_paged" if paged else "")
                      + (")" if full_layer else "")
                      + f" ({'decode_tc_kernel' if plan['tensor_core'] else 'decode_simt_kernel'})",
            "achieved": round(achieved, 2),
            "peak": peaks["hbm_gbs"],
            "peak_source": peaks["source"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": call_bytes,
            "avg_launch_ms": round(attn_avg_ms, 5),
            "avg_launch_ms_how": "timed region / layer calls (back-to-back launches)",
            "isolated_launch_ms": round(iso_ms, 5),
        },
        "e2e": {
            "value": round(world * sb["step"] / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
        },
        "step_ms_median": round(float(np.median(step_times)), 4),
        "step_ms_best": round(float(np.min(step_times)), 4),
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
        "device_status": status,
    }
    if split is not None:
        split["attn_only_frac_of_measured"] = round(split["attn_only_gbs"] / peaks["hbm_gbs"], 4)
        line["separate_calls"] = split
    if full_layer and not args.no_cpu_baseline:
        line["cpu_baseline"] = {"skipped": "the oracle baseline is timed on the step "
                                           "(run without --layer)"}
    elif not args.no_cpu_baseline:
        gbs, spent, units, nbytes = oracle_sample(base, target_s=args.cpu_seconds, n=n)
        line["cpu_baseline"] = {
            "value": round(gbs, 4), "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{units} (sequence, KV head) units of {cfg.name} layer-shaped data "
                      f"({nbytes / 2**20:.0f} MiB, {spent:.1f} s, float64 numpy oracle: "
                      "append + attention)"}
    return line


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores, timed per
    step on a bounded sample of the workload; rank 0 only."""
    from gqa_kv_cache_append_gb300.inputs import seq_lens_for, workload
    import dataclasses
    if rank != 0:
        return None
    cfg = workload(args.workload)
    n = args.tokens
    if n > 1:
        cfg = dataclasses.replace(cfg, kind="plain")
    # ~40 s of oracle work over the whole run: drawing each sample's inputs
    # costs about twice that again, so the run ends in about two minutes
    per_step_s = max(0.25, min(20.0, 40.0 / max(1, args.steps + args.warmup)))
    vals = []
    total_units = total_bytes = 0
    for k in range(args.warmup + args.steps):
        gbs, spent, units, nbytes = oracle_sample(cfg, target_s=per_step_s, n=n)
        if k >= args.warmup:
            vals.append(gbs)
            total_units += units
            total_bytes += nbytes
    value = float(np.mean(vals))
    lens = seq_lens_for(cfg)
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), shapes of the workload)",
        "config": {"workload": cfg.name, "layers": cfg.layers, "b": cfg.b, "h": cfg.h,
                   "g": cfg.g, "d_head": cfg.d, "seq_len": int(np.max(lens)),
                   "parallelism": "host cores", "tokens_per_step": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{total_units} (sequence, KV head) units over {args.steps} "
                                   f"steps, {total_bytes / 2**20:.0f} MiB"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama3_70b_b32_m8192")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--g", type=int, default=None, help="KV heads (for the g-knob sweep)")
    ap.add_argument("--h", type=int, default=None, help="query heads (shape studies)")
    ap.add_argument("--b", type=int, default=None, help="sequences (shape studies)")
    ap.add_argument("--cap", type=int, default=None,
                    help="cache capacity = length of full sequences (shape studies)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the step (and the end-to-end step) in a CUDA graph")
    ap.add_argument("--ordered", action="store_true",
                    help="no early streaming: each layer waits for the previous one")
    ap.add_argument("--separate", action="store_true",
                    help="time gqa_kv_append + gqa_decode_attn instead of gqa_decode_step")
    ap.add_argument("--tokens", type=int, default=1,
                    help="new tokens per sequence per step (causal; speculative / chunked decode)")
    ap.add_argument("--layer", action="store_true",
                    help="time the whole incremental layer (q/k/v projection, step, output "
                         "projection) through gqa_decode_layer")
    ap.add_argument("--dtype", choices=["bf16", "f16", "f32"], default=None,
                    help="storage type override (shape studies)")
    ap.add_argument("--d", type=int, default=None, help="head dim d_k (and d_v) override")
    ap.add_argument("--dv", type=int, default=None, help="head dim d_v override")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="the CUDA-core kernel where the tensor-core kernel would run")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK",
                    help="paged KV cache with this block size (rows per block)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (small profiling cases)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed steps
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, local_rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
