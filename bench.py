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


def copy_groups(nl: int):
    """The end-to-end step's copy schedule over `nl` layers, as half-open
    layer ranges: the inputs in three groups (the first layer, the next
    three, the rest), the outputs in groups of max(8, ceil(nl / 10)) layers
    with the last layer alone.  Each list covers 0..nl in order, without
    gaps or overlaps."""
    in_cuts = sorted({0, min(1, nl), min(4, nl), nl})
    in_groups = list(zip(in_cuts[:-1], in_cuts[1:]))
    og = max(8, -(-nl // 10))
    out_ends = sorted({e for e in range(og - 1, nl - 1, og)} |
                      {e for e in (nl - 2, nl - 1) if e >= 0})
    out_groups = list(zip([0] + [e + 1 for e in out_ends[:-1]], [e + 1 for e in out_ends]))
    return in_groups, out_groups


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
# ncu summary mode: --ncu-summary KERNEL profiles one launch of a kernel of
# this library on a small case of the workload and writes the summary that
# profiled_traffic reads (plus the launch list of a step)
# ---------------------------------------------------------------------------
NCU_KERNELS = {  # --ncu-summary name -> (kernel name regex, source file)
    "decode_tc": ("decode_tc_kernel", "decode_tc.cu"),
    "decode_simt": ("decode_simt_kernel", "decode_simt.cu"),
    "combine": ("combine_kernel", "gqa_api.cu"),
    "proj_tc": ("proj_tc_kernel", "proj_tc.cu"),
}
# the counters the summary quotes: one launch, a handful of hardware units
NCU_METRICS = [
    "gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
    "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed",
    "dram__bytes_read.sum.per_second",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
    "smsp__issue_active.avg.pct_of_peak_sustained_active",
    "sm__warps_active.avg.pct_of_peak_sustained_active",
    "lts__throughput.avg.pct_of_peak_sustained_elapsed",
    "launch__grid_size", "launch__block_size", "launch__registers_per_thread",
    "launch__shared_mem_per_block_dynamic", "gpc__cycles_elapsed.avg.per_second",
]
OUR_KERNELS = "regex:decode_tc|decode_simt|combine|kv_append|proj_tc|wait_selftest"


def ncu_case_args(args) -> list:
    """bench.py arguments of the small case profiled for args: the same
    workload and overrides, few enough layers to hold at most ~2.5 GB of
    cache on the device (one layer where a layer holds more) and at most 32,
    but where that allows at least 4 x L2 of K/V per step; two timed steps
    after three warm-up steps, nothing else."""
    from gqa_kv_cache_append_gb300.inputs import bench_layers, seq_lens_for, workload
    import dataclasses
    cfg = workload(args.workload)
    for k in ("g", "h", "b", "cap"):
        if getattr(args, k):
            cfg = dataclasses.replace(cfg, **{k: getattr(args, k)})
    if args.d:
        cfg = dataclasses.replace(cfg, d=args.d)
    if args.dv:
        cfg = dataclasses.replace(cfg, d_v=args.dv)
    if args.dtype:
        cfg = dataclasses.replace(cfg, dtype=args.dtype)
    lens = seq_lens_for(cfg)
    per_layer_cap = cfg.b * cfg.g * cfg.cap * (cfg.d + cfg.dv) * cfg.elt
    l2 = 129 << 20  # GB300's L2 as the device reports it (no CUDA call in this process)
    # (at most 32 layers: few launches before the profiled one)
    layers = args.layers or max(1, min(bench_layers(cfg, lens, l2, args.tokens),
                                       int(2.5e9 // per_layer_cap), 32))
    out = ["--workload", args.workload, "--layers", str(layers), "--steps", "2", "--warmup", "3",
           "--no-cpu-baseline", "--no-workloads"]
    for k in ("g", "h", "b", "cap", "d", "dv", "dtype"):
        v = getattr(args, k)
        if v:
            out += [f"--{k}", str(v)]
    if args.tokens != 1:
        out += ["--tokens", str(args.tokens)]
    if args.paged:
        out += ["--paged", str(args.paged)]
    for flag in ("layer", "cuda_cores", "separate", "ordered"):
        if getattr(args, flag):
            out.append("--" + flag.replace("_", "-"))
    return out


def ncu_tag(args) -> str:
    """Summary name suffix: the workload, then whatever differs from it."""
    tag = args.workload
    for k in ("g", "h", "b", "cap", "d", "dv", "dtype"):
        v = getattr(args, k)
        if v:
            tag += f"_{k}{v}"
    if args.tokens != 1:
        tag += f"_n{args.tokens}"
    if args.paged:
        tag += f"_paged{args.paged}"
    for flag in ("layer", "cuda_cores", "separate", "ordered"):
        if getattr(args, flag):
            tag += "_" + flag
    return tag


def _ncu_rows(csv_path: str) -> list:
    """Rows of an `ncu --page raw --csv --print-units base` table (the second
    line, the units, is skipped)."""
    import csv
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rows = list(csv.reader(lines))
    if len(rows) < 2:
        return []
    hdr = rows[0]
    return [dict(zip(hdr, r)) for r in rows[2:]]


def _num(row, key):
    try:
        return float(str(row.get(key, "")).replace(",", ""))
    except ValueError:
        return None


def run_ncu_summary(args) -> int:
    """Profile KERNEL (args.ncu_summary) on the small case of the workload:
    (1) run the case without ncu (it must exit 0); (2) the launch list of its
    steps (gpu__time_duration.sum of every launch of this library's kernels,
    one pass); (3) one launch of KERNEL in the third warm-up step with the
    summary's counters.  Raw output goes to --ncu-out; the summaries
    <kernel>_<tag>.md and launches_<tag>.md are written there too (copy them
    to profiles/).  Every ncu run keeps the GPU clocks as they are."""
    import shutil
    from gqa_kv_cache_append_gb300 import binding as B
    regex, src_name = NCU_KERNELS[args.ncu_summary]
    out_dir = os.path.abspath(args.ncu_out)
    os.makedirs(out_dir, exist_ok=True)
    case = ncu_case_args(args)
    tag = ncu_tag(args)
    py = [sys.executable, os.path.join(ROOT, "bench.py")] + case
    ncu = shutil.which("ncu") or "/usr/local/cuda/bin/ncu"
    # (1) the plain run
    with open(os.path.join(out_dir, f"ncu_plain_{tag}.log"), "w") as f:
        rc = subprocess.run(py, stdout=f, stderr=subprocess.STDOUT, cwd=ROOT).returncode
    if rc != 0:
        print(f"plain run failed (rc {rc}); not profiled", file=sys.stderr)
        return rc
    plain = open(os.path.join(out_dir, f"ncu_plain_{tag}.log")).read().strip().splitlines()
    line = json.loads(plain[-1])
    layers = int(line["config"]["layers"])
    per_step = int(line["gpu_launches_per_step"])
    # launches of KERNEL per step: the decode kernel runs once per layer call;
    # the combine kernel only where the plan says two kernels per call
    if args.ncu_summary in ("decode_tc", "decode_simt"):
        k_per_step = layers
    elif args.ncu_summary == "combine":
        k_per_step = max(0, per_step - layers)
    else:
        k_per_step = 2 * layers
    if k_per_step == 0:
        print(f"{regex} does not run in this case", file=sys.stderr)
        return 2
    # (2) launch list of the two timed steps (after the three warm-up steps)
    list_csv = os.path.join(out_dir, f"ncu_launches_{tag}.csv")
    cmd_list = [ncu, "--metrics", "gpu__time_duration.sum", "--clock-control", "none",
                "-k", OUR_KERNELS, "-s", str(3 * per_step), "-c", str(2 * per_step),
                "--csv", "--page", "raw", "--print-units", "base", "--log-file", list_csv] + py
    rc = subprocess.run(cmd_list, stdout=subprocess.DEVNULL, stderr=subprocess.STDOUT,
                        cwd=ROOT).returncode
    if rc != 0:
        return rc
    # (3) one launch of KERNEL (the third warm-up step's first)
    rep = os.path.join(out_dir, f"ncu_{args.ncu_summary}_{tag}")
    cmd_one = [ncu, "--clock-control", "none", "--metrics", ",".join(NCU_METRICS),
               "-k", f"regex:{regex}", "-s", str(2 * k_per_step), "-c", "1",
               "-o", rep, "-f"] + py
    rc = subprocess.run(cmd_one, stdout=subprocess.DEVNULL, stderr=subprocess.STDOUT,
                        cwd=ROOT).returncode
    if rc != 0:
        return rc
    one_csv = rep + ".raw.csv"
    with open(one_csv, "w") as f:
        rc = subprocess.run([ncu, "-i", rep + ".ncu-rep", "--page", "raw", "--csv",
                             "--print-units", "base"], stdout=f, cwd=ROOT).returncode
    if rc != 0:
        return rc
    rows = _ncu_rows(one_csv)
    if not rows:
        return 3
    r = rows[0]
    rd, wr = _num(r, "dram__bytes_read.sum"), _num(r, "dram__bytes_write.sum")
    traffic = int(rd + wr)
    src = os.path.join(ROOT, "gqa_kv_cache_append_gb300", "csrc", src_name)
    alg = line["roofline"]["algorithmic_bytes_per_launch"]
    pretty = " ".join(["python bench.py --ncu-summary", args.ncu_summary] +
                      [a for a in sys.argv[1:] if a not in ("--ncu-summary", args.ncu_summary)])
    shell = " ".join(["python bench.py"] + case)

    def pct(k):
        v = _num(r, k)
        return "-" if v is None else f"{v:.1f} %"
    md = [
        f"# {r.get('Kernel Name', regex).split('(')[0]} — {tag}",
        "",
        f"Made by `{pretty}` (raw reports in the --ncu-out folder).  Case profiled:",
        "",
        f"    {shell}",
        "",
        "It ran without ncu first (exit 0).  Then, every run with `--clock-control none`:",
        "",
        f"    ncu --metrics gpu__time_duration.sum -k {OUR_KERNELS} -s {3 * per_step} "
        f"-c {2 * per_step} --csv ... {shell}",
        f"    ncu --metrics <the rows below> -k regex:{regex} -s {2 * k_per_step} -c 1 ... {shell}",
        "",
        "| metric | value |",
        "|---|---|",
        f"| gpu__time_duration.sum (isolated, serialised) | {_num(r, 'gpu__time_duration.sum') / 1e3:.2f} us |",
        f"| dram__bytes_read.sum | {int(rd):,} B |",
        f"| dram__bytes_write.sum | {int(wr):,} B |",
        f"| read + write vs algorithmic bytes ({alg:,}) | {traffic / alg:.4f} |",
        f"| dram read throughput | {(_num(r, 'dram__bytes_read.sum.per_second') or 0) / 1e12:.2f} TB/s |",
        f"| gpu__dram_throughput (of peak, elapsed) | {pct('gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed')} |",
        f"| sm__pipe_tensor_cycles_active | {pct('sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed')} |",
        f"| smsp__issue_active | {pct('smsp__issue_active.avg.pct_of_peak_sustained_active')} |",
        f"| sm__warps_active | {pct('sm__warps_active.avg.pct_of_peak_sustained_active')} |",
        f"| lts__throughput | {pct('lts__throughput.avg.pct_of_peak_sustained_elapsed')} |",
        f"| grid x block, registers, dynamic smem | {r.get('launch__grid_size')} x "
        f"{r.get('launch__block_size')}, {r.get('launch__registers_per_thread')}, "
        f"{r.get('launch__shared_mem_per_block_dynamic')} B |",
        f"| SM clock | {(_num(r, 'gpc__cycles_elapsed.avg.per_second') or 0) / 1e9:.2f} GHz |",
        "",
        f"source_sha256: {kernel_source_hash(src)}",
        f"traffic_bytes_per_launch: {traffic}",
        "",
    ]
    with open(os.path.join(out_dir, f"{args.ncu_summary}_{tag}.md"), "w") as f:
        f.write("\n".join(md))
    # launch list: per kernel, launches, total time and share
    agg = {}
    for row in _ncu_rows(list_csv):
        name = row.get("Kernel Name", "?").split("(")[0]
        t = _num(row, "gpu__time_duration.sum") or 0.0
        n0, t0 = agg.get(name, (0, 0.0))
        agg[name] = (n0 + 1, t0 + t)
    total = sum(t for _, t in agg.values()) or 1.0
    lm = [f"# Launch list — {tag}", "",
          f"Made by `{pretty}`; ncu serialises launches with cold caches: compare SHARES.",
          "Two timed steps of:", "", f"    {shell}", "",
          "| kernel | launches | total (us) | share | avg (us) |", "|---|---|---|---|---|"]
    for name, (cnt, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        lm.append(f"| {name} | {cnt} | {t / 1e3:.1f} | {100 * t / total:.1f} % | "
                  f"{t / cnt / 1e3:.2f} |")
    with open(os.path.join(out_dir, f"launches_{tag}.md"), "w") as f:
        f.write("\n".join(lm) + "\n")
    print(json.dumps({"ncu_summary": args.ncu_summary, "tag": tag, "traffic": traffic,
                      "algorithmic": alg, "launch_list": agg}))
    return 0


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and reference arm), spread over
# every host core: one spawned worker process per core, each timing the
# float64 oracle on whole (sequence, all KV heads) units of the workload
# ---------------------------------------------------------------------------
_ORACLE_POOL = None


def host_cores() -> int:
    """Cores this process may run on (the oracle baseline uses all of them)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_pool(workers: int):
    """(executor, manager) with `workers` spawned processes, made once per
    run (spawn: safe after CUDA was initialised in this process)."""
    global _ORACLE_POOL
    if _ORACLE_POOL is None or _ORACLE_POOL[2] != workers:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        # one thread per worker process in any BLAS / OpenMP runtime it loads
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        ctx = mp.get_context("spawn")
        ex = ProcessPoolExecutor(max_workers=workers, mp_context=ctx,
                                 initializer=_oracle_worker_init)
        _ORACLE_POOL = (ex, ctx.Manager(), workers)
    return _ORACLE_POOL[0], _ORACLE_POOL[1]


def _oracle_worker_init():
    import torch
    torch.set_num_threads(1)


def _oracle_unit(cfg, n: int, i: int, L: int):
    """Host arrays (numpy, bf16 as uint16 patterns) of sample i: one sequence
    of length L with all its KV heads, drawn with the workload's recipe."""
    import dataclasses
    import torch
    from gqa_kv_cache_append_gb300.inputs import make_layer, make_layer_multi
    sub = dataclasses.replace(cfg, b=1, layers=1, seed=cfg.seed * 7919 + i)
    lens = np.array([L], dtype=np.int32)
    x = (make_layer(sub, 0, "cpu", lens=lens) if n == 1
         else make_layer_multi(sub, n, 0, "cpu", lens=lens))

    def np_(t):
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), "bf16"
        return t.numpy(), ("f16" if t.dtype == torch.float16 else "f32")
    tag = np_(x["q"])[1]
    return [np_(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")], tag


def _oracle_task(cfg, n: int, samples, reps: int, barrier):
    """One worker: draw its samples, wait for every worker, then run the
    oracle's step `reps` times over them.  Returns (bytes, units, t0, t1) on
    the system-wide monotonic clock."""
    import oracle
    data = [(_oracle_unit(cfg, n, i, L), L) for i, L in samples]
    barrier.wait(timeout=600)
    nbytes = units = 0
    t0 = time.monotonic()
    for k in range(reps):
        (arrs, tag), L = data[k % len(data)]
        if n == 1:
            oracle.decode_step(*arrs, np.array([L]), cfg.g, cfg.scale, dtype=tag)
        else:
            oracle.decode_step_multi(*arrs, np.array([L]), cfg.g, cfg.scale, dtype=tag)
        nbytes += (L * cfg.g + n * cfg.h) * (cfg.d + cfg.dv) * cfg.elt
        units += cfg.g
    return nbytes, units, t0, time.monotonic()


def oracle_sample(cfg, target_s: float = 12.0, n: int = 1, workers: int = 0):
    """Time the float64 oracle's decode step (append + attention) on whole
    units (one sequence, all its KV heads, n new tokens) of layer-0-shaped
    data of the workload, drawn on the host with the same recipe, on
    `workers` processes at once (0: every host core), for about target_s
    seconds of wall time.  Returns (GB/s of algorithmic bytes over the wall
    time of the timed window, seconds, units, bytes, workers)."""
    from gqa_kv_cache_append_gb300.inputs import seq_lens_for
    import oracle
    workers = workers or host_cores()
    lens = seq_lens_for(cfg)
    # one call here sizes the work: reps per worker for ~target_s of wall time
    (arrs, tag), L0 = _oracle_unit(cfg, n, 0, int(lens[0])), int(lens[0])
    t = time.perf_counter()
    if n == 1:
        oracle.decode_step(*arrs, np.array([L0]), cfg.g, cfg.scale, dtype=tag)
    else:
        oracle.decode_step_multi(*arrs, np.array([L0]), cfg.g, cfg.scale, dtype=tag)
    one = max(time.perf_counter() - t, 1e-4)
    reps = max(1, int(round(target_s / one)))
    per = min(reps, 4)  # distinct samples per worker (cycled)
    ex, mgr = _oracle_pool(workers)
    barrier = mgr.Barrier(workers)
    futs = []
    for w in range(workers):
        idx = [w * per + k for k in range(per)]
        samples = [(i, int(lens[i % len(lens)])) for i in idx]
        futs.append(ex.submit(_oracle_task, cfg, n, samples, reps, barrier))
    res = [f.result(timeout=900) for f in futs]
    nbytes = sum(r[0] for r in res)
    units = sum(r[1] for r in res)
    wall = max(r[3] for r in res) - min(r[2] for r in res)
    return nbytes / wall / 1e9, wall, units, nbytes, workers


# ---------------------------------------------------------------------------
# the other workloads, timed after the headline one in the same run
# ---------------------------------------------------------------------------
# (name, overrides): the long-context MQA step, the ragged Qwen-shaped batch,
# the four points of the g sweep and the fp32 MQA step
EXTRA_WORKLOADS = [
    ("long_mqa_b8_m131072", {}),
    ("qwen25_7b_b64_ragged", {}),
    ("gqa_sweep_b16_h32_d128_m4096", {"g": 32}),
    ("gqa_sweep_b16_h32_d128_m4096", {"g": 8}),
    ("gqa_sweep_b16_h32_d128_m4096", {"g": 4}),
    ("gqa_sweep_b16_h32_d128_m4096", {"g": 1}),
    ("mqa_f32_b1_h8_d64_m256", {}),
]


def time_workload(name, overrides, dev, stream, steps, warmup, dist, world, rank, peak_gbs):
    """The bench's default step (one gqa_decode_step per layer, early
    streaming, every layer back to back on one stream, inputs resident in
    HBM) on another workload: layers rotated as bench_layers says, W untimed
    steps, then K steps between CUDA events on the stream, max over ranks,
    clocks sampled during the timed region.  Returns a summary dict (rank 0)
    and frees the workload's memory."""
    import dataclasses
    import torch
    from gqa_kv_cache_append_gb300 import binding as B
    from gqa_kv_cache_append_gb300.inputs import bench_layers, make_layer, seq_lens_for, workload
    base = workload(name, **overrides)
    lens = seq_lens_for(base)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cfg = dataclasses.replace(base, layers=bench_layers(base, lens, l2),
                              seed=replica_seed(base.seed, rank))
    layers = [make_layer(cfg, l, dev) for l in range(cfg.layers)]
    outs = [torch.empty((cfg.b, cfg.h, cfg.dv), dtype=cfg.torch_dtype, device=dev)
            for _ in range(cfg.layers)]

    def step():
        for l, x in enumerate(layers):
            B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                              x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.scale,
                              outs[l], flags=B.GQA_STEP_EARLY_STREAM, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(smi_id(dev.index))
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(dist, dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1) / steps)
    status = B.gqa_device_status(stream)
    plan = B.gqa_decode_plan(cfg.b, 1, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.cap, cfg.dtype)
    sb = step_bytes(cfg, lens)
    del layers, outs
    torch.cuda.empty_cache()
    if rank != 0:
        return None
    call_ms = ms / cfg.layers
    call_bytes = sb["attn_per_layer"] + sb["append_per_layer"]
    gbs = call_bytes / (call_ms * 1e-3) / 1e9
    tag = name + "".join(f"_{k}{v}" for k, v in overrides.items())
    return tag, {
        "value": round(world * sb["step"] / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
        "us_per_call": round(call_ms * 1000, 3),
        "frac_of_measured": round(gbs / peak_gbs, 4),
        "pct_of_nominal_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
        "layer_steps_per_s": round(world * cfg.layers / (ms * 1e-3), 1),
        "bytes_per_call": call_bytes, "layers_rotated": cfg.layers, "steps": steps,
        "dtype": cfg.dtype, "b": cfg.b, "h": cfg.h, "g": cfg.g, "d": cfg.d,
        "sum_seq_lens": int(np.sum(lens)),
        "kernel": "tensor cores" if plan["tensor_core"] else "CUDA cores",
        "kernels_per_call": plan["kernels"], "ctas": plan["ctas"],
        "clocks": clk, "device_status": status,
    }


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
        # exactly N layers (past a workload's own: seeded replicas of its shape)
        base = dataclasses.replace(base, layers=args.layers)
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
    from gqa_kv_cache_append_gb300.inputs import bench_layers, layer_flops
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if not args.layers:
        base = dataclasses.replace(base, layers=bench_layers(
            base, lens, l2, n, projection_bytes(base) if full_layer else 0))
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
    # pinned host memory, runs the layers, and copies all outputs back.  The
    # copies run on a second stream beside the layers: the first layer's
    # inputs, then the next three layers', then the rest, each group waited
    # for by the first layer that reads it; the outputs go back in about ten
    # groups (at least eight layers each) as each group's last layer ends,
    # the last layer alone (an event between two launches costs host time,
    # which a step of short launches feels).
    # The step ends when its last copy has.  The serial form (all inputs,
    # the layers, all outputs, one stream) is timed beside it. ----
    host_in = {k: v.cpu().pin_memory() for k, v in packed.items()}
    host_out = torch.empty_like(out_all, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    in_groups, out_groups = copy_groups(cfg.layers)
    side = torch.cuda.Stream(dev)
    ev_start = torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in in_groups]
    ev_out = [torch.cuda.Event() for _ in out_groups]
    ev_done = torch.cuda.Event()

    def e2e_step():
        ev_start.record(stream)
        side.wait_event(ev_start)
        with torch.cuda.stream(side):
            for i, (a, z) in enumerate(in_groups):
                for key, t in host_in.items():
                    packed[key][a:z].copy_(t[a:z], non_blocking=True)
                ev_in[i].record(side)
        gi, go = 0, 0
        for l, x in enumerate(layers):
            if gi < len(in_groups) and l == in_groups[gi][0]:
                stream.wait_event(ev_in[gi])
                gi += 1
            layer_call(l, x)
            if l == out_groups[go][1] - 1:
                ev_out[go].record(stream)
                side.wait_event(ev_out[go])
                a, z = out_groups[go]
                with torch.cuda.stream(side):
                    host_out[a:z].copy_(out_all[a:z], non_blocking=True)
                go += 1
        ev_done.record(side)
        stream.wait_event(ev_done)

    def e2e_serial():
        for key, t in host_in.items():
            packed[key].copy_(t, non_blocking=True)
        for l, x in enumerate(layers):
            layer_call(l, x)
        host_out.copy_(out_all, non_blocking=True)

    def time_e2e(fn):
        run = fn
        if args.graph:
            fn()
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                fn()
            run = graph.replay
        for _ in range(max(1, args.warmup)):
            run()
        barrier(dist, dev)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        return max_over_ranks(dist, e0.elapsed_time(e1) / args.steps), run

    with torch.cuda.stream(stream):
        e2e_serial_ms, _ = time_e2e(e2e_serial)
        e2e_ms, run_e2e = time_e2e(e2e_step)
        assert torch.equal(host_out.to(dev), out_all), "end-to-end outputs differ"
    status |= B.gqa_device_status(stream)

    # ---- the other workloads (the default run only): the headline's
    # buffers are released first ----
    peaks = measured_peaks()
    extra = None
    if args.workloads:
        layers.clear()
        packed.clear()
        outs.clear()
        host_in.clear()
        out_all = host_out = None
        run_step = run_e2e = None
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        extra = {}
        for name, over in EXTRA_WORKLOADS:
            res = time_workload(name, over, dev, stream, args.workload_steps, args.warmup, dist,
                                world, rank, peaks["hbm_gbs"])
            if res is not None:
                extra[res[0]] = res[1]

    if rank != 0:
        return None
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
            "how": f"copies on a second stream beside the layers: inputs in {len(in_groups)} "
                   f"groups, outputs in {len(out_groups)}",
            "serial_ms_per_step": round(e2e_serial_ms, 4),
            "serial_value": round(world * sb["step"] / (e2e_serial_ms * 1e-3) / 1e9, 2),
        },
        "step_ms_median": round(float(np.median(step_times)), 4),
        "step_ms_best": round(float(np.min(step_times)), 4),
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clk,
        "device_status": status,
    }
    if extra is not None:
        line["workloads"] = extra
    if split is not None:
        split["attn_only_frac_of_measured"] = round(split["attn_only_gbs"] / peaks["hbm_gbs"], 4)
        line["separate_calls"] = split
    if full_layer and not args.no_cpu_baseline:
        line["cpu_baseline"] = {"skipped": "the oracle baseline is timed on the step "
                                           "(run without --layer)"}
    elif not args.no_cpu_baseline:
        gbs, spent, units, nbytes, cores = oracle_sample(base, target_s=args.cpu_seconds, n=n)
        line["cpu_baseline"] = {
            "value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{units} (sequence, KV head) units of {cfg.name} layer-shaped data "
                      f"({nbytes / 2**20:.0f} MiB in {spent:.1f} s of wall time on {cores} "
                      "worker processes, one per host core; float64 numpy oracle: "
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
    # --ref-seconds of timed oracle work (wall time, all host cores) over the
    # whole run; drawing each step's samples adds about as much again
    per_step_s = max(0.1, min(20.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    vals = []
    total_units = total_bytes = 0
    cores = host_cores()
    for k in range(args.warmup + args.steps):
        gbs, spent, units, nbytes, cores = oracle_sample(cfg, target_s=per_step_s, n=n)
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
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{total_units} (sequence, KV head) units over {args.steps} "
                                   f"steps, {total_bytes / 2**20:.0f} MiB, on {cores} worker "
                                   "processes (one per host core)"},
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
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall time of the oracle baseline (all host cores)")
    ap.add_argument("--ref-seconds", type=float, default=40.0,
                    help="--impl reference: timed oracle wall time over the whole run")
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
                    help="run exactly N layers (small profiling cases; past the workload's "
                         "own layers, seeded replicas of its shape)")
    ap.add_argument("--ncu-summary", choices=sorted(NCU_KERNELS), default=None,
                    help="profile one launch of this kernel on a small case of the workload "
                         "(ncu, clocks untouched) and write its summary and launch list")
    ap.add_argument("--ncu-out", default="ncu_reports",
                    help="--ncu-summary: folder for the raw reports and the summaries")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other workloads after the headline one")
    ap.add_argument("--workload-steps", type=int, default=20,
                    help="timed steps of each of the other workloads")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed steps
    # the other workloads are timed after a default run only (named
    # workload, no shape, layout or call overrides)
    default_run = (args.workload == "llama3_70b_b32_m8192" and not any(
        v for v in (args.g, args.h, args.b, args.cap, args.layers, args.dtype, args.d, args.dv,
                    args.paged)) and not (args.graph or args.ordered or args.separate or
                                          args.layer or args.cuda_cores) and args.tokens == 1)
    args.workloads = default_run and not args.no_workloads
    if args.ncu_summary:
        raise SystemExit(run_ncu_summary(args))
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, local_rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
