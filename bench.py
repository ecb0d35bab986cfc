#!/usr/bin/env python3
"""Bucket-flush bandwidth of the ZeRO-1 gradient-reduction path on GB300.

One step = one ZeRO-1 gradient flush of the 402.8M-parameter model at W=8:
the owner map, then the 7 reduce buckets (52,428,800-element capacity, reverse
layer order) flushed with reduce-to-owner, probe counters on.  The bf16
gradients of the 8 replicas ([8, 402,753,536], 6.4 GB) sit in HBM before the
timed region; every step reads all of them, so no step is served from L2.

Printed (rank 0, one JSON line): whole-job algorithmic HBM GB/s (value),
grad-elements/s, the roofline of the flush kernel, the same metric end to end
with host buffers (e2e), the CPU oracle baseline, clocks, and the other hot-path
rows (AllReduce form, deferred accumulation, ReduceScatter, AllGather) timed on
their own workloads.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bucket-flush achieved HBM GB/s and % of GB300 peak; grad-elems/s at W=8"
WORKLOAD = "zero1-bucket-flush 402.8M params W=8 bf16 reduce-to-owner (7 buckets of <=52,428,800 elems)"
FALLBACK_HBM_GBS = 6800.0
SEED, SIGMA, WORLD = 3, 1e-3, 8
KERNEL_SOURCES = ["flush_kernels.cuh", "flush_w8.cu", "common.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["dpred", "reference"], default="dpred")
    ap.add_argument("--max-buckets", type=int, default=0, help="flush only the first k buckets (small profiling case)")
    ap.add_argument("--no-rows", action="store_true", help="skip the other hot-path rows")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--flush-path", choices=["auto", "ldg", "tma"], default="auto",
                    help="kernel family of the flush (results are bit-identical)")
    ap.add_argument("--sweep", action="store_true",
                    help="flush sweep: bucket sizes 1 KB-1 GB per replica, W in {2,4,8,16}, bf16/fp32, eager and "
                         "CUDA-graph replay; one JSON line per case")
    ap.add_argument("--sweep-worlds", default="2,4,8,16", help="--sweep: world sizes to run (comma-separated)")
    ap.add_argument("--sweep-kb", default="1,16,256,4096,65536,1048576",
                    help="--sweep: bucket sizes per replica row in KB (comma-separated)")
    ap.add_argument("--row", choices=["allgather", "reduce_scatter", "accumulate"], default=None,
                    help="time one other hot-path row alone (small profiling cases) and print its JSON line")
    ap.add_argument("--row-nodes", type=int, default=8)
    ap.add_argument("--row-elems", type=int, default=1 << 29,
                    help="--row size: M (allgather / reduce_scatter) or n (accumulate, W=4)")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers ---

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(src: str) -> str:
    """C/C++ source without comments and blank lines: comment edits do not
    change the kernel, so they do not invalidate a traffic record."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "zero_collectives_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(bytes_per_launch: float):
    """DRAM read+write bytes per flush launch, from the committed ncu record of
    one bucket-0 launch (805 MB of gradients, one capture, one launch),
    scaled by the algorithmic bytes of a launch of this run over those of the
    captured one: every launch of the step streams its W rows once, so its
    traffic grows in proportion.  None when the kernel sources changed since
    the capture."""
    path = os.path.join(ROOT, "profiles", "flush_bucket0_w8_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_hash") != kernel_hash():
            return None
        return float(d["dram_bytes"]) * bytes_per_launch / float(d["algorithmic_bytes"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampling (every 50 ms) around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "mem_mhz": None, "mem_mhz_min": None,
                    "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mem = [float(r[9]) for r in rows if r[9].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "mem_mhz": statistics.median(mem) if mem else None, "mem_mhz_min": min(mem) if mem else None,
                "reasons": reasons, "samples": len(rows)}


def smi_gpu_id(logical: int) -> str:
    """nvidia-smi's id of a CUDA device (physical index or UUID under CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if logical < len(ids):
            return ids[logical]
    return str(logical)


def dist_setup(gpus: int):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device: str = "cuda") -> float:
    """The slowest rank's time: every rank's clock ran over the same barrier-bracketed region."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(ws: int, step_bytes: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return ws * step_bytes * steps / (elapsed_ms * 1e-3) / 1e9


# ----------------------------------------------------------- the workload ---

def flush_workload(max_buckets: int):
    from datagen import workloads
    tree = workloads.tree_402m()
    layout = workloads.arrival_layout(tree)
    buckets = layout.buckets if max_buckets <= 0 else layout.buckets[:max_buckets]
    return tree, layout, buckets


def flush_bytes(world, buckets, omap, holders_written_fn, in_size=2, out_size=2) -> int:
    """Algorithmic bytes of a flush: every row of every bucket read once, every
    delivered non-empty destination written once."""
    total = 0
    for b in buckets:
        total += world * b.size * in_size
        for t in b.tasks:
            total += int(t["numel"]) * out_size * holders_written_fn(int(t["param_id"]))
    return total


def owner_mode_writes(omap):
    def n(p):
        if omap.owner[p] >= 0:
            return 1
        return int(omap.holder_hi[p] - omap.holder_lo[p] + 1)
    return n


def events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def run_dpred(args):
    import numpy as np
    import torch

    import datagen
    import zero_collectives_gb300 as zc
    from datagen import BF16, NORMAL

    ws, rank, local = dist_setup(args.gpus)
    zc.set_flush_path({"auto": zc.PATH_AUTO, "ldg": zc.PATH_LDG, "tma": zc.PATH_TMA}[args.flush_path])
    tree, layout, buckets = flush_workload(args.max_buckets)
    n_rows = max(b.start + b.size for b in buckets)  # the whole row unless --max-buckets trims it
    stream = torch.cuda.current_stream()
    grads = torch.empty((WORLD, n_rows), dtype=torch.bfloat16, device="cuda")
    datagen.fill_device(grads.data_ptr(), WORLD, n_rows, n_rows, BF16, NORMAL, SEED, 0, 1, 0, SIGMA,
                        stream.cuda_stream)
    bucket_list = [(b.start, b.tasks) for b in buckets]
    # The executor object holds the owner map, the installed gradient buffers
    # (real on holders, empty elsewhere) and each bucket's destination table;
    # the timed step flushes through the per-call entry point, one
    # dpred_flush_bucket call per bucket as the buckets fill, with the probe
    # counters on and the overlap promise (consecutive buckets share no byte).
    ex = zc.Zero1Executor(WORLD, tree.numel, layout.row_offset, bucket_list, torch.bfloat16)
    step_bytes = flush_bytes(WORLD, buckets, ex.omap, owner_mode_writes(ex.omap))
    step_elems = sum(b.size for b in buckets)
    launches_per_step = len(buckets)
    calls = [(grads[:, s0:s0 + size], t, tab) for (s0, t), size, tab in zip(ex.buckets, ex.sizes, ex.tables)]
    owner = ex.omap.owner
    probes = []

    def step():
        zc.build_owner_map(WORLD, [(None, tree.numel)], True)   # the owner map (host, identical every time)
        probes.clear()
        for i, (g, t, tab) in enumerate(calls):
            probes.append(zc.flush_bucket(g, t, owner, tab, BF16, True, True, probe=True, flush_index=i,
                                          overlap=True))

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = Clocks(smi_gpu_id(torch.cuda.current_device()))
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    ev_start, ev_end = events(2)
    ev_start.record(stream)
    for _ in range(args.steps):
        step()
    ev_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    elapsed_ms = ev_start.elapsed_time(ev_end)
    # The timed region launches nothing but the flush kernel, so its mean
    # launch duration is the region time over the launches (gaps included).
    avg_launch_ms = elapsed_ms / (launches_per_step * args.steps)
    elapsed_max = max_over_ranks(elapsed_ms, ws)
    value_gbs = job_gbs(ws, step_bytes, args.steps, elapsed_max)
    elems_per_s = ws * step_elems * args.steps / (elapsed_max * 1e-3)

    peak, peak_src = peaks()
    bytes_per_launch = step_bytes / launches_per_step
    achieved = bytes_per_launch / (avg_launch_ms * 1e-3) / 1e9
    traffic = traffic_per_launch(bytes_per_launch)
    result = {
        "metric": METRIC, "value": round(value_gbs, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic (seeded Irwin-Hall normal, sigma 1e-3)",
        "config": {"workload": WORKLOAD, "world": WORLD, "params": tree.n_params, "elems_per_replica": step_elems,
                   "buckets": len(buckets), "bucket_capacity": 52_428_800, "reduce_to_owner": True, "pre_div": True,
                   "parallelism": f"{ws} independent replica(s), no inter-GPU exchange",
                   "l2": "inputs larger than L2: each step reads 6.4 GB of gradients"},
        "grad_elems_per_s": round(elems_per_s, 1),
        "pct_of_peak": round(100.0 * value_gbs / ws / peak, 2),
        "algorithmic_bytes_per_step": step_bytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
                     "kernel": "flush_kernel<8,1,bf16,bf16,FlushArgsInline,false>", "bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": round(avg_launch_ms, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    # Step-time distribution: a separate pass with one event pair per step (the
    # headline region above has no per-step events).
    evs = events(51)
    evs[0].record(stream)
    for i in range(50):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(50))
    result["step_ms_p10_p50_p90"] = [round(per[5], 4), round(per[25], 4), round(per[45], 4)]
    result["replica_elems_per_s"] = round(elems_per_s * WORLD, 1)
    step()
    torch.cuda.synchronize()
    result["probe_line"] = probes[0].line(0, zc.BF16, True)
    result["step_path"] = ("per bucket: dpred_flush_bucket (probe counters on, DPRED_FLUSH_OVERLAP); "
                           "the owner map rebuilt on the host every step")
    result["owner_map_report"] = ex.omap.report()

    if not args.no_e2e:
        result["e2e"] = e2e(args, ex, grads, step_bytes, ws)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(buckets, tree, layout, args.cpu_seconds)
        result["cpu_baseline_all_cores"] = cpu_baseline_all_cores(buckets, tree)
    if not args.no_rows:
        result["flush_paths"] = flush_path_ab(ex, grads, step_bytes, peak)
        result["flush_bucket_calls_step"] = flush_bucket_calls(ex, grads, step_bytes, peak)
        result["flush_bucket_per_call_overhead"] = per_call_overhead()
        mix = flush_mix_ceiling(grads, step_bytes, peak)
        mix["step_frac_of_step_mix"] = round(value_gbs / ws / mix["step_mix"]["GB/s"], 4)
        result["flush_mix_ceiling"] = mix
        del grads
        result["rows"] = rows(peak)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e(args, ex, grads, step_bytes, ws):
    """Same metric through the public API with host buffers: every step takes
    the gradients from pinned host memory and leaves the reduced gradients in
    pinned host memory.  Two forms of the step are timed: the mapped step
    (the flush kernels read and write the host buffers over the host link;
    the reported value) and the staged step (copy-engine copies into HBM,
    flush, copies back, pipelined over buckets)."""
    import torch
    import datagen
    from datagen import BF16, NORMAL
    host = torch.empty(grads.shape, dtype=torch.bfloat16, pin_memory=True)
    datagen.fill_host(host.view(torch.int16).numpy().view("uint16"), BF16, NORMAL, SEED, sigma=SIGMA)
    outs = [torch.empty(b.shape, dtype=b.dtype, pin_memory=True) for b in ex.grad.buf]
    stream = torch.cuda.current_stream()
    forms = {"mapped": lambda: ex.flush_all_mapped(host, outs, grads, probe=True),
             "staged": lambda: ex.flush_all_from_host(host, outs, grads, probe=True)}
    for f in forms.values():
        f()
    torch.cuda.synchronize()
    # the host link's own bandwidth in this run, for context: the median of
    # five plain copy-engine copies (single copies from pinned host memory
    # occasionally take two to three times as long on this platform)
    evs = events(6)
    evs[0].record(stream)
    for i in range(5):
        grads.copy_(host, non_blocking=True)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    copy_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(5))
    link_gbs = host.numel() * host.element_size() / (copy_ms[2] * 1e-3) / 1e9
    ms = {}
    for name, f in forms.items():
        barrier(ws)
        evs = events(args.e2e_steps + 1)
        evs[0].record(stream)
        for i in range(args.e2e_steps):
            f()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.e2e_steps)]
        ms[name] = (max_over_ranks(evs[0].elapsed_time(evs[-1]), ws), sorted(per))
    h2d = host.numel() * host.element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def gbs(name):
        return round(ws * step_bytes * args.e2e_steps / (ms[name][0] * 1e-3) / 1e9, 1)

    staged_per = ms["staged"][1]
    return {"value": gbs("mapped"), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": round(ms["mapped"][0] / args.e2e_steps, 3),
            "step_ms_min_max": [round(ms["mapped"][1][0], 3), round(ms["mapped"][1][-1], 3)],
            "host_link_h2d_GBps": round(link_gbs, 1),
            "path": "Zero1Executor.flush_all_mapped (dpred_executor_flush_all_mapped): kernels read and write "
                    "the pinned host buffers directly",
            "staged": {"value": gbs("staged"), "ms_per_step": round(ms["staged"][0] / args.e2e_steps, 3),
                       "step_ms_min_max": [round(staged_per[0], 3), round(staged_per[-1], 3)],
                       "path": "Zero1Executor.flush_all_from_host (dpred_executor_flush_all_from_host): "
                               "copy-engine copies pipelined with the flush"}}


def _cpu_flush_sample(buckets, tree, seconds):
    import numpy as np
    import datagen
    import oracle
    from datagen import BF16, NORMAL
    om = oracle.owner_map(WORLD, [(list(range(WORLD)), tree.numel)], True)
    done_bytes, done_s, done_elems, n_b = 0, 0.0, 0, 0
    for b in buckets:
        host = datagen.host_matrix(WORLD, b.size, BF16, NORMAL, SEED, col0=b.start, sigma=SIGMA)
        dst = [[None] * len(b.tasks) for _ in range(WORLD)]
        writes = 0
        for t, task in enumerate(b.tasks):
            p = int(task["param_id"])
            for r in range(om["holder_lo"][p], om["holder_hi"][p] + 1):
                dst[r][t] = np.empty(int(task["numel"]), np.uint16)
            writes += int(task["numel"]) * (1 if om["owner"][p] >= 0 else int(om["holder_hi"][p] - om["holder_lo"][p]) + 1)
        t0 = time.perf_counter()
        oracle.flush(WORLD, host, b.tasks, om["owner"], tree.n_params, dst, BF16, True, True)
        done_s += time.perf_counter() - t0
        done_bytes += WORLD * int(b.size) * 2 + int(writes) * 2
        done_elems += b.size
        n_b += 1
        if done_s >= seconds:
            break
    return done_bytes, done_s, done_elems, n_b


def cpu_baseline(buckets, tree, layout, seconds):
    """The oracle (single-threaded C) on the same workload: whole buckets in
    order until `seconds` of flush time have accumulated."""
    nbytes, secs, elems, nb = _cpu_flush_sample(buckets, tree, seconds)
    return {"value": round(nbytes / secs / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{nb} of {len(buckets)} buckets ({elems} elements per replica row), single-threaded C oracle",
            "seconds": round(secs, 2), "grad_elems_per_s": round(elems / secs, 1)}


def _cpu_worker(job):
    """One host core: the unchanged single-threaded oracle on a contiguous run of
    bucket 0's tasks, repeated until `seconds` have passed.  Runs in a spawned
    process; the start barrier lines all workers up before anyone times."""
    import numpy as np
    import datagen
    import oracle
    from datagen import BF16, NORMAL
    tasks, col0, n_params, numel, seconds, barrier = job
    om = oracle.owner_map(WORLD, [(list(range(WORLD)), numel)], True)
    base = int(tasks["offset"][0])
    tasks = tasks.copy()
    tasks["offset"] -= base
    width = int(tasks["offset"][-1] + tasks["numel"][-1])
    host = datagen.host_matrix(WORLD, width, BF16, NORMAL, SEED, col0=col0 + base, sigma=SIGMA)
    dst = [[None] * len(tasks) for _ in range(WORLD)]
    writes = 0
    for t, task in enumerate(tasks):
        p = int(task["param_id"])
        lo, hi = int(om["holder_lo"][p]), int(om["holder_hi"][p])
        for r in range(lo, hi + 1):
            dst[r][t] = np.empty(int(task["numel"]), np.uint16)
        writes += int(task["numel"]) * (1 if om["owner"][p] >= 0 else hi - lo + 1)
    per_pass = WORLD * width * 2 + writes * 2
    barrier.wait()
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.flush(WORLD, host, tasks, om["owner"], n_params, dst, BF16, True, True)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return t0, time.perf_counter(), passes * per_pass


def cpu_baseline_all_cores(buckets, tree, seconds=1.5):
    """The same single-threaded oracle run as one process per host core, each on
    its own contiguous share of bucket 0's tasks, all started together.  The
    figure is the bytes of all workers over the wall time from the first start
    to the last finish."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    b = buckets[0]
    cum = [0]
    for t in b.tasks:
        cum.append(cum[-1] + int(t["numel"]))
    groups, start = [], 0
    for c in range(1, cores + 1):
        target = b.size * c // cores
        end = start
        while end < len(b.tasks) and cum[end + 1] <= target:
            end += 1
        if c == cores:
            end = len(b.tasks)
        if end > start:
            groups.append(b.tasks[start:end])
        start = end
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        barrier = mgr.Barrier(len(groups))
        with ctx.Pool(len(groups)) as pool:
            res = pool.map(_cpu_worker, [(g, b.start, tree.n_params, tree.numel, seconds, barrier) for g in groups])
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    nbytes = sum(r[2] for r in res)
    return {"value": round(nbytes / wall / 1e9, 3), "unit": "GB/s", "cores": len(groups), "kind": "oracle",
            "sample": f"bucket 0 ({b.size} elements per replica row) split by tasks over {len(groups)} processes, "
                      f"each the single-threaded C oracle repeated for {seconds} s",
            "seconds": round(wall, 2)}


def flush_path_ab(ex, grads, step_bytes, peak):
    """The same flush step through the native executor (prebuilt plans, one
    call per step) with each kernel family (LDG streaming vs TMA staging), and
    with the launch overlap between buckets turned off."""
    import zero_collectives_gb300 as zc
    out = {}
    prev = zc.set_flush_path(zc.PATH_LDG)
    for name, path, overlap in (("ldg", zc.PATH_LDG, True), ("ldg_no_overlap", zc.PATH_LDG, False),
                                ("tma", zc.PATH_TMA, True)):
        zc.set_flush_path(path)
        was = ex.set_overlap(overlap)
        ms = timed(lambda: ex.flush_all(grads), 20, warm=3)
        ex.set_overlap(was)
        gbs = step_bytes / (ms * 1e-3) / 1e9
        out[name] = {"ms_per_step": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
    zc.set_flush_path(prev)
    return out


def flush_bucket_calls(ex, grads, step_bytes, peak):
    """The step as a caller of dpred_flush_bucket makes it: one call per bucket
    (7 on the 402.8M W=8 workload), probe counters on, with and without the
    overlap promise (consecutive buckets share no byte).  The executor's
    prebuilt plans are not used; every call goes through the per-call entry
    point (validation and planning are served by its plan cache after the
    first step)."""
    import zero_collectives_gb300 as zc
    out = {}
    calls = [(grads[:, s0:s0 + size], t, tab) for (s0, t), size, tab in zip(ex.buckets, ex.sizes, ex.tables)]
    owner = ex.omap.owner
    for overlap in (True, False):
        def step():
            for g, t, tab in calls:
                zc.flush_bucket(g, t, owner, tab, zc.BF16, True, True, probe=True, overlap=overlap)
        ms = timed(step, 20, warm=3)
        gbs = step_bytes / (ms * 1e-3) / 1e9
        out["overlap" if overlap else "no_overlap"] = {
            "ms_per_step": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "calls_per_step": len(calls)}
    return out


def flush_mix_ceiling(grads, step_bytes, peak):
    """HBM ceilings for the flush step's own traffic, measured by kernels that
    do nothing else (dpred_stream_mixed): the step's reads (the 6.44 GB of
    gradient rows) alone, and those reads together with its 1.02 GB of writes,
    spread evenly and with no store waiting for a load."""
    import torch
    import zero_collectives_gb300 as zc
    read_b = grads.numel() * grads.element_size()
    write_b = (step_bytes - read_b) // 16 * 16
    dst = torch.empty(write_b, dtype=torch.uint8, device="cuda")
    out = {}
    for name, wb in (("read_only", 0), ("step_mix", write_b)):
        ms = timed(lambda: zc.stream_mixed(grads, dst, read_bytes=read_b, write_bytes=wb), 10)
        gbs = (read_b + wb) / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "read_bytes": read_b, "write_bytes": wb}
    del dst
    return out


def per_call_overhead():
    """Host cost of one dpred_flush_bucket call on a small bucket (W=8, 16
    tasks, 256 KB of gradients): host time per call over 2000 back-to-back
    eager calls (perf_counter) through the Python binding, through a prepared
    per-bucket call (zc.BucketFlush, by its CPython module and by ctypes) with
    and without the probe, and through a pre-marshalled ctypes call; the first call (validation and planning)
    against a repeated one (plan cache); and the device time per call measured
    with CUDA events over the same loop."""
    import ctypes
    import time

    import numpy as np
    import torch

    import zero_collectives_gb300 as zc
    world, n_tasks, per = 8, 16, 1024
    grads = torch.randn((world, n_tasks * per), device="cuda").to(torch.bfloat16)
    tasks = np.zeros(n_tasks, dtype=zc.TASK_DTYPE)
    tasks["param_id"] = np.arange(n_tasks)
    tasks["offset"] = np.arange(n_tasks) * per
    tasks["numel"] = per
    owner = (np.arange(n_tasks) % world).astype(np.int32)
    bufs = [torch.empty(per, dtype=torch.bfloat16, device="cuda") for _ in range(n_tasks)]
    dst = zc.DstTable(world, n_tasks, [bufs[t].data_ptr() if owner[t] == r else 0
                                       for r in range(world) for t in range(n_tasks)])
    s = torch.cuda.current_stream()
    L = zc.lib()
    probe = zc._Probe()
    args = (world, zc.BF16, grads.data_ptr(), grads.stride(0), tasks.ctypes.data, n_tasks, owner.ctypes.data,
            n_tasks, zc.BF16, dst.c, 1, 1, 0, ctypes.byref(probe), None, 0, s.cuda_stream)
    out = {"bucket": f"W={world}, {n_tasks} tasks x {per} bf16 elements ({world * n_tasks * per * 2} bytes read)"}
    prepared = zc.BucketFlush(grads, tasks, owner, dst)
    prepared_ct = zc.BucketFlush(grads, tasks, owner, dst, fast=False)
    out["prepared_call_path"] = "cpython module" if prepared.fast else "ctypes (no Python headers on this host)"
    for name, fn in (("python_binding", lambda: zc.flush_bucket(grads, tasks, owner, dst, probe=True)),
                     ("python_prepared_call", lambda: prepared(probe=True)),
                     ("python_prepared_call_no_probe", lambda: prepared()),
                     ("python_prepared_call_ctypes", lambda: prepared_ct(probe=True)),
                     ("python_prepared_call_ctypes_no_probe", lambda: prepared_ct()),
                     ("ctypes_premarshalled", lambda: L.dpred_flush_bucket(*args))):
        for _ in range(50):
            fn()
        torch.cuda.synchronize()
        a, b = events(2)
        n = 2000
        a.record(s)
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        host_us = (time.perf_counter() - t0) / n * 1e6
        b.record(s)
        torch.cuda.synchronize()
        out[name] = {"host_us_per_call": round(host_us, 2), "device_us_per_call": round(a.elapsed_time(b) / n * 1e3, 2)}
    # first call of a new table (validation and planning) against a repeated one
    tasks2 = tasks.copy()
    firsts = []
    for k in range(20):
        tasks2["numel"] = per - 1 - k  # a new table every time: a plan-cache miss
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        L.dpred_flush_bucket(world, zc.BF16, grads.data_ptr(), grads.stride(0), tasks2.ctypes.data, n_tasks,
                             owner.ctypes.data, n_tasks, zc.BF16, dst.c, 1, 1, 0, ctypes.byref(probe), None, 0,
                             s.cuda_stream)
        firsts.append((time.perf_counter() - t0) * 1e6)
    torch.cuda.synchronize()
    out["ctypes_first_call_us_median"] = round(float(np.median(firsts)), 2)
    # the bare ctypes call: the same 17 arguments with an empty task table
    # (validated from the plan cache, nothing launched)
    empty = np.zeros(0, dtype=zc.TASK_DTYPE)
    noop = (world, zc.BF16, grads.data_ptr(), grads.stride(0), empty.ctypes.data, 0, None, 0, zc.BF16, None, 1, 1,
            0, ctypes.byref(probe), None, 0, s.cuda_stream)
    for _ in range(100):
        L.dpred_flush_bucket(*noop)
    t0 = time.perf_counter()
    for _ in range(20000):
        L.dpred_flush_bucket(*noop)
    out["ctypes_empty_call_us"] = round((time.perf_counter() - t0) / 20000 * 1e6, 2)
    out["c_side_and_launch_us"] = round(out["ctypes_premarshalled"]["host_us_per_call"] - out["ctypes_empty_call_us"], 2)
    return out


# -------------------------------------------------------- other hot rows ---

def timed(fn, reps, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = events(2)
    s = torch.cuda.current_stream()
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def rows(peak):
    import numpy as np
    import torch
    import datagen
    import zero_collectives_gb300 as zc
    from datagen import BF16, F32, NORMAL, UNIFORM, stream_id, workloads

    out = {}
    s = torch.cuda.current_stream().cuda_stream

    def entry(ms, nbytes, **kw):
        gbs = nbytes / (ms * 1e-3) / 1e9
        d = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "bytes": nbytes}
        d.update(kw)
        return d

    # AllReduce form vs reduce-to-owner, in place over the 8 bucket rows (the
    # collective as NCCL runs it: result delivered to every row / to one row).
    tree = workloads.tree_402m()
    layout = workloads.arrival_layout(tree)
    n = tree.total
    g = torch.empty((WORLD, n), dtype=torch.bfloat16, device="cuda")
    datagen.fill_device(g.data_ptr(), WORLD, n, n, BF16, NORMAL, SEED, 0, 1, 0, SIGMA, s)
    for rto, name in ((False, "flush_inplace_allreduce"), (True, "flush_inplace_owner")):
        ip = zc.InPlaceExecutor(WORLD, tree.numel, [(b.start, b.tasks) for b in layout.buckets], torch.bfloat16,
                                reduce_to_owner=rto)
        ms = timed(lambda: ip.flush_all(g), 5)
        om = ip.omap
        writes = sum(int(tree.numel[p]) * (1 if om.owner[p] >= 0 else WORLD) for p in range(tree.n_params))
        out[name] = entry(ms, WORLD * n * 2 + writes * 2, launches=len(layout.buckets),
                          workload="402.8M W=8 bf16, 7 buckets, in place (InPlaceExecutor: one call, overlapped)")
        ip.close()

    # The same model cut into small buckets (at most 4,194,304 elements, 8 MiB
    # per replica row): about a hundred launches per step, where the overlap of
    # consecutive flushes matters most.
    small = workloads.arrival_layout(tree, capacity=1 << 22)
    ex_s = zc.Zero1Executor(WORLD, tree.numel, small.row_offset, [(b.start, b.tasks) for b in small.buckets],
                            torch.bfloat16)
    sb = flush_bytes(WORLD, small.buckets, ex_s.omap, owner_mode_writes(ex_s.omap))
    for overlap, name in ((True, "flush_step_small_buckets"), (False, "flush_step_small_buckets_no_overlap")):
        ex_s.set_overlap(overlap)
        ms = timed(lambda: ex_s.flush_all(g), 20, warm=3)
        out[name] = entry(ms, sb, workload=f"402.8M W=8 bf16, {len(small.buckets)} buckets of <= 4,194,304 elements",
                          launches=len(small.buckets))
    ex_s.close()
    del ex_s

    # Partitioned flush (every rank gets exactly its partition slice) over the
    # 7 arrival-order buckets, and over the whole model as one bucket against
    # the two-pass relayout + ReduceScatter that ncclReduceScatter would need.
    flat = np.concatenate([[0], np.cumsum(tree.numel)[:-1]]).astype(np.int64)
    P = -(-n // WORLD)
    parts = [torch.empty(P, dtype=torch.bfloat16, device="cuda") for _ in range(WORLD)]
    wsf = torch.empty(zc.flush_workspace_bytes(WORLD, tree.n_params + WORLD), dtype=torch.uint8, device="cuda")

    def part7():
        for b in layout.buckets:
            zc.flush_bucket_partitioned(g[:, b.start:b.start + b.size], b.tasks, flat, P, parts, zc.BF16, True,
                                        workspace=wsf)

    ms = timed(part7, 5)
    out["flush_partitioned_step"] = entry(ms, WORLD * n * 2 + n * 2,
                                          workload="402.8M W=8 bf16, 7 buckets, each rank its partition slice")
    # the same through the partitioned executor (one native call, overlapped launches),
    # on the 7 buckets and on 98 small ones
    for lay, name in ((layout, "partitioned_executor_step"), (small, "partitioned_executor_step_small_buckets")):
        pex = zc.PartitionedExecutor(WORLD, tree.numel, lay.row_offset, [(b.start, b.tasks) for b in lay.buckets],
                                     torch.bfloat16, parts=parts)
        ms = timed(lambda: pex.flush_all(g), 20, warm=3)
        out[name] = entry(ms, WORLD * n * 2 + n * 2, workload=f"402.8M W=8 bf16, {len(lay.buckets)} buckets",
                          launches=len(lay.buckets))
        pex.close()
    one = workloads.arrival_layout(tree, capacity=None).buckets[0]
    ms = timed(lambda: zc.flush_bucket_partitioned(g, one.tasks, flat, P, parts, zc.BF16, True, workspace=wsf), 5)
    out["flush_partitioned_one_bucket"] = entry(ms, WORLD * n * 2 + n * 2, workload="402.8M W=8 bf16 as one bucket")
    relaid = torch.empty((WORLD, WORLD * P), dtype=torch.bfloat16, device="cuda")
    rs_out = torch.empty((WORLD, P), dtype=torch.bfloat16, device="cuda")
    wsr = torch.empty(zc.bucket_relayout_workspace_bytes(WORLD, len(one.tasks)), dtype=torch.uint8, device="cuda")

    def two_pass():
        zc.bucket_relayout(g, one.tasks, flat, P, P, relaid, workspace=wsr)
        zc.reduce_scatter(relaid, rs_out, pre_div=True)

    ms = timed(two_pass, 5)
    out["relayout_then_reduce_scatter_one_bucket"] = entry(
        ms, 2 * WORLD * n * 2 + WORLD * WORLD * P * 2 + WORLD * P * 2,
        workload="402.8M W=8 bf16 as one bucket: relayout pass + ReduceScatter", launches=2)
    del g, parts, relaid, rs_out

    # Accumulation on the 402.8M-parameter W=8 shape: bf16 micro-batch
    # gradients into an fp32 [8, n] accumulator, one add and the fused finalize.
    n = tree.total
    acc8 = torch.empty((WORLD, n), dtype=torch.float32, device="cuda")
    g8 = torch.empty((WORLD, n), dtype=torch.bfloat16, device="cuda")
    datagen.fill_device(g8.data_ptr(), WORLD, n, n, BF16, NORMAL, SEED, 0, 1, 0, SIGMA, s)
    zc.accumulate_microbatch(acc8, g8, first=True, finalize=False)
    tot8 = torch.empty(n, dtype=torch.float32, device="cuda")
    ms = timed(lambda: zc.accumulate_microbatch(acc8, g8, first=False, finalize=False), 5)
    out["accumulate_402m_w8_add"] = entry(ms, WORLD * n * (4 + 2 + 4),
                                          workload="402.8M W=8: fp32 acc += bf16 g (read acc, read g, write acc)")
    ms = timed(lambda: zc.accumulate_microbatch(acc8, g8, first=False, finalize=True, total=tot8), 5)
    out["accumulate_402m_w8_finalize"] = entry(ms, WORLD * n * (4 + 2) + 4 * n,
                                               workload="402.8M W=8: last micro-batch fused with the reduce")
    del acc8, g8, tot8

    # Deferred accumulation: W=4, 8 micro-batches, qwen3-0.6b tree, fp32.
    W, M = 4, 8
    n = workloads.tree_qwen3_06b().total
    acc = torch.empty((W, n), dtype=torch.float32, device="cuda")
    gb = [torch.empty((W, n), dtype=torch.float32, device="cuda") for _ in range(2)]
    for m, buf in enumerate(gb):
        datagen.fill_device(buf.data_ptr(), W, n, n, F32, NORMAL, 4, stream_id(0, m), 1, 0, SIGMA, s)
    total = torch.empty(n, dtype=torch.float32, device="cuda")

    def deferred():
        for m in range(M):
            last = m == M - 1
            zc.accumulate_microbatch(acc, gb[m % 2], first=(m == 0), finalize=last, total=total if last else None)

    ms = timed(deferred, 3, warm=1)
    nbytes = 8 * W * n + (M - 2) * 12 * W * n + 8 * W * n + 4 * n
    out["accumulate_deferred_step"] = entry(ms, nbytes, workload="qwen3-0.6b tree n=596,049,920, W=4, 8 micro-batches, fp32",
                                            launches=M)
    addm = lambda: zc.accumulate_microbatch(acc, gb[0], first=False, finalize=False)  # noqa: E731
    ms_add = timed(addm, 5)
    out["accumulate_one_microbatch"] = entry(ms_add, 12 * W * n, workload="one acc += g pass, W=4, fp32")
    fin = lambda: zc.accumulate_microbatch(acc, gb[0], first=False, finalize=True, total=total)  # noqa: E731
    ms_fin = timed(fin, 5)
    out["accumulate_finalize"] = entry(ms_fin, 8 * W * n + 4 * n, workload="last micro-batch fused with the reduce")
    # per-micro-batch all-reduce (the status quo): reduce each micro-batch, then sum
    red = torch.empty((1, n), dtype=torch.float32, device="cuda")
    s_m = torch.empty(n, dtype=torch.float32, device="cuda")

    def per_mb():
        for m in range(M):
            zc.accumulate_microbatch(acc, gb[m % 2], first=True, finalize=True, total=s_m)
            zc.accumulate_microbatch(red, s_m.view(1, n), first=(m == 0), finalize=False)

    ms_pm = timed(per_mb, 3, warm=1)
    out["accumulate_per_microbatch_step"] = entry(ms_pm, M * (4 * W * n + 4 * n) + 4 * n + (M - 1) * 12 * n,
                                                  workload="status quo: reduce every micro-batch", launches=2 * M)
    # accumulator checkpoints (row f2): save reduces the W rows to the total a
    # checkpoint holds; restore puts a total back as row 0 with the rest zero
    ms_save = timed(lambda: zc.accumulator_save(acc, total), 5)
    out["accumulator_save"] = entry(ms_save, 4 * W * n + 4 * n, workload="qwen3 W=4: W fp32 rows -> total")
    ms_rest = timed(lambda: zc.accumulator_restore(acc, total), 5)
    out["accumulator_restore"] = entry(ms_rest, 4 * n + 4 * W * n, workload="qwen3 W=4: total -> row 0, zeros elsewhere")
    del acc, gb, total, red, s_m

    # HBM ceilings measured by kernels that do nothing else (no AllGather
    # involved): a write-only fill (the best of 16-byte, 32-byte and bulk
    # stores over 4 GiB) and, for the AllGather's own mix of reads and writes
    # (M read, N*M written), a stream of exactly that mix in which no store
    # waits for a load.
    wbuf = torch.empty(4 << 30, dtype=torch.uint8, device="cuda")
    fills = {}
    for method in (0, 1, 2):
        fills[method] = timed(lambda: zc.fill_pattern(wbuf, 0x3F803F80, method, 0 if method < 2 else 1), 10)
    best = min(fills, key=fills.get)
    out["hbm_write_ceiling"] = entry(fills[best], 4 << 30, workload="write-only fill of 4 GiB (dpred_fill_pattern)",
                                     method=best, ms_by_method={m: round(v, 4) for m, v in fills.items()})
    write_gbs = out["hbm_write_ceiling"]["GB/s"]
    ms = timed(lambda: wbuf.zero_(), 10)
    out["torch_zero_fill_4GiB"] = entry(ms, 4 << 30, workload="write-only reference (torch zero_)")
    del wbuf
    Mel = 1 << 29
    mixed_ms = {}
    src = torch.empty(Mel, dtype=torch.bfloat16, device="cuda")
    for N in (8, 4):
        dstm = torch.empty(N * Mel, dtype=torch.bfloat16, device="cuda")
        mixed_ms[N] = timed(lambda: zc.stream_mixed(src, dstm), 10)
        out[f"hbm_mixed_ceiling_1r{N}w"] = entry(mixed_ms[N], Mel * 2 + N * Mel * 2,
                                                 workload=f"1 GiB read + {N} GiB written, no dependency (dpred_stream_mixed)")
        del dstm
    del src

    # ReduceScatter / AllGather, M = 1 GiB bf16.
    for N in (8, 4):
        S = Mel // N
        x = torch.empty((N, Mel), dtype=torch.bfloat16, device="cuda")
        datagen.fill_device(x.data_ptr(), N, Mel, Mel, BF16, UNIFORM, 5, 0, 1, 0, 1.0, s)
        rs = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
        ms = timed(lambda: zc.reduce_scatter(x, rs), 10)
        out[f"reduce_scatter_N{N}"] = entry(ms, N * Mel * 2 + Mel * 2, workload=f"N={N}, M=1 GiB bf16")
        prev = zc.set_flush_path(zc.PATH_TMA)
        ms = timed(lambda: zc.reduce_scatter(x, rs), 10)
        zc.set_flush_path(prev)
        out[f"reduce_scatter_N{N}_tma"] = entry(ms, N * Mel * 2 + Mel * 2, workload=f"N={N}, M=1 GiB bf16, TMA path")
        del x
        ag = torch.empty((N, Mel), dtype=torch.bfloat16, device="cuda")
        model_ms = (N * Mel * 2 / (write_gbs * 1e9) + Mel * 2 / (peak * 1e9)) * 1e3
        for order, name in ((0, "canonical"), (1, "ring")):
            for form, suffix, what in ((zc.AG_AUTO, "", "default form"), (zc.AG_TMA1, "_tma1", "bulk copies, unskewed"),
                                       (zc.AG_REGISTER, "_ldg", "register-streaming form")):
                prev = zc.set_allgather_form(form)
                ms = timed(lambda: zc.allgather(rs, ag, order), 10)
                zc.set_allgather_form(prev)
                r = entry(ms, Mel * 2 + N * Mel * 2, workload=f"N={N}, M=1 GiB bf16, {what}")
                r["frac_of_write_model"] = round(model_ms / ms, 4)
                r["frac_of_mixed_ceiling"] = round(mixed_ms[N] / ms, 4)
                out[f"allgather_{name}_N{N}{suffix}"] = r
        del ag, rs
    # the restore writes W rows for one read (1 read : 4 writes at W=4): the
    # N=4 mixed stream has the same mix
    out["accumulator_restore"]["frac_of_mixed_ceiling"] = round(
        out["accumulator_restore"]["GB/s"] / out["hbm_mixed_ceiling_1r4w"]["GB/s"], 4)
    out["allgather_schedules_N8"] = schedule_fit(8, Mel)
    torch.cuda.empty_cache()
    return out


def schedule_fit(N, M):
    """Ring, bidirectional ring and recursive doubling run step by step (one
    copy launch per step) on N node buffers; per-step CUDA-event times fitted to
    t = alpha + bytes / beta, and the page's closed forms (eqs. ring-ag,
    ag-bidir-ring, rd-ag) evaluated with that alpha and the per-node
    beta' = beta / (2N) (every step moves N chunks in and out of one HBM)."""
    import numpy as np
    import torch
    import datagen
    import zero_collectives_gb300 as zc
    from datagen import BF16, UNIFORM
    S = M // N
    s = torch.cuda.current_stream()
    x = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
    datagen.fill_device(x.data_ptr(), N, S, S, BF16, UNIFORM, 5, 0, 1, 0, 1.0, s.cuda_stream)
    bufs = torch.empty((N, N * S), dtype=torch.bfloat16, device="cuda")
    cb = S * 2
    pts, totals = [], {}
    names = {zc.SCHED_RING: "ring", zc.SCHED_BIDIR_RING: "bidir_ring", zc.SCHED_RECURSIVE_DOUBLING: "recursive_doubling"}
    for sched, name in names.items():
        steps = zc.allgather_schedule_steps(sched, N)
        best = None
        for rep in range(4):
            zc.allgather_schedule_init(sched, x, bufs)
            ev = events(steps + 1)
            ev[0].record(s)
            for k in range(1, steps + 1):
                zc.allgather_schedule_step(sched, bufs, k)
                ev[k].record(s)
            torch.cuda.synchronize()
            t = [ev[k - 1].elapsed_time(ev[k]) for k in range(1, steps + 1)]
            if rep and (best is None or sum(t) < sum(best)):
                best = t
        for k, tk in enumerate(best, start=1):
            if sched == zc.SCHED_RING:
                chunks = N
            elif sched == zc.SCHED_BIDIR_RING:
                chunks = N * (1 if (N % 2 == 0 and k == N // 2) else 2)
            else:
                chunks = N * (1 << (k - 1))
            pts.append((2 * chunks * cb, tk * 1e-3))
        totals[name] = {"steps": steps, "measured_ms": round(sum(best), 4), "step_ms": [round(v, 4) for v in best]}
    b = np.array([p[0] for p in pts], dtype=np.float64)
    t = np.array([p[1] for p in pts], dtype=np.float64)
    A = np.stack([np.ones_like(b), b], axis=1)
    (alpha, inv_beta), *_ = np.linalg.lstsq(A, t, rcond=None)
    beta = 1.0 / inv_beta
    beta_node = beta / (2 * N)
    Mb = M * 2
    from zero_collectives_gb300 import costs
    model = {"ring": costs.ring(N, Mb, alpha, beta_node),
             "bidir_ring": costs.bidirectional_ring(N, Mb, alpha, beta_node),
             "recursive_doubling": costs.recursive_doubling(N, Mb, alpha, beta_node)}
    for name in totals:
        totals[name]["model_ms"] = round(model[name] * 1e3, 4)
    del x, bufs
    return {"alpha_us": round(alpha * 1e6, 2), "beta_GBps": round(beta / 1e9, 1),
            "beta_per_node_GBps": round(beta_node / 1e9, 1), "M_bytes": Mb, "schedules": totals}


# ------------------------------------------------------ reference (oracle) ---

def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import datagen
    import oracle
    from datagen import BF16, NORMAL
    tree, layout, buckets = flush_workload(args.max_buckets)
    b = buckets[0]
    om = oracle.owner_map(WORLD, [(list(range(WORLD)), tree.numel)], True)
    # Sample per step: the leading tasks of the first bucket, sized so that
    # warm-up plus timed steps take about two minutes of oracle time.
    calib = _sub_bucket(b, 1 << 20)
    host_c = datagen.host_matrix(WORLD, int(calib["offset"][-1] + calib["numel"][-1]), BF16, NORMAL, SEED,
                                 col0=b.start, sigma=SIGMA)
    t0 = time.perf_counter()
    _oracle_step(host_c, calib, om, tree)
    rate = (1 << 20) / (time.perf_counter() - t0)
    total_steps = args.steps + max(args.warmup, 1)
    elems = int(max(8192, min(b.size, rate * 120.0 / total_steps)))
    tasks = _sub_bucket(b, elems)
    width = int(tasks["offset"][-1] + tasks["numel"][-1])
    host = datagen.host_matrix(WORLD, width, BF16, NORMAL, SEED, col0=b.start, sigma=SIGMA)
    for _ in range(max(args.warmup, 1)):
        _oracle_step(host, tasks, om, tree)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += _oracle_step(host, tasks, om, tree)
    secs = time.perf_counter() - t0
    gbs = nbytes / secs / 1e9
    sample = f"first {width} elements per replica row of bucket 0 (of 402,753,536), per step; single-threaded C oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic (seeded Irwin-Hall normal, sigma 1e-3)",
        "config": {"workload": WORKLOAD, "world": WORLD, "sample_elems_per_step": width},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _sub_bucket(b, elems):
    import numpy as np
    keep = []
    acc = 0
    for t in b.tasks:
        if acc >= elems:
            break
        t = t.copy()
        t["numel"] = min(int(t["numel"]), elems - acc)
        keep.append(t)
        acc += int(t["numel"])
    return np.array(keep, dtype=b.tasks.dtype)


def _oracle_step(host, tasks, om, tree):
    import numpy as np
    import oracle
    from datagen import BF16
    dst = [[None] * len(tasks) for _ in range(WORLD)]
    writes = 0
    for t, task in enumerate(tasks):
        p = int(task["param_id"])
        for r in range(om["holder_lo"][p], om["holder_hi"][p] + 1):
            dst[r][t] = np.empty(int(task["numel"]), np.uint16)
        writes += int(task["numel"]) * (1 if om["owner"][p] >= 0 else int(om["holder_hi"][p] - om["holder_lo"][p]) + 1)
    oracle.flush(WORLD, host, tasks, om["owner"], tree.n_params, dst, BF16, True, True)
    return WORLD * host.shape[1] * 2 + writes * 2


def single_row(args):
    """One row alone, e.g. for an ncu capture of a small case."""
    import torch
    import datagen
    import zero_collectives_gb300 as zc
    from datagen import F32, NORMAL, UNIFORM, BF16, stream_id
    torch.cuda.set_device(0)
    zc.set_flush_path({"auto": zc.PATH_AUTO, "ldg": zc.PATH_LDG, "tma": zc.PATH_TMA}[args.flush_path])
    s = torch.cuda.current_stream().cuda_stream
    peak, _ = peaks()
    N, M = args.row_nodes, args.row_elems
    if args.row in ("allgather", "reduce_scatter"):
        S = M // N
        if args.row == "allgather":
            x = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
            datagen.fill_device(x.data_ptr(), N, S, S, BF16, UNIFORM, 5, 0, 1, 0, 1.0, s)
            out = torch.empty((N, N * S), dtype=torch.bfloat16, device="cuda")
            fn = lambda: zc.allgather(x, out, 0)  # noqa: E731
            nbytes = N * S * 2 + N * N * S * 2
        else:
            x = torch.empty((N, N * S), dtype=torch.bfloat16, device="cuda")
            datagen.fill_device(x.data_ptr(), N, N * S, N * S, BF16, UNIFORM, 5, 0, 1, 0, 1.0, s)
            out = torch.empty((N, S), dtype=torch.bfloat16, device="cuda")
            fn = lambda: zc.reduce_scatter(x, out)  # noqa: E731
            nbytes = N * N * S * 2 + N * S * 2
    else:
        W, n = 4, M
        acc = torch.empty((W, n), dtype=torch.float32, device="cuda")
        g = torch.empty((W, n), dtype=torch.float32, device="cuda")
        datagen.fill_device(g.data_ptr(), W, n, n, F32, NORMAL, 4, stream_id(0, 0), 1, 0, SIGMA, s)
        acc.zero_()
        fn = lambda: zc.accumulate_microbatch(acc, g, first=False, finalize=False)  # noqa: E731
        nbytes = 12 * W * n
    ms = timed(fn, max(args.steps, 1), warm=max(args.warmup, 3))
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"row": args.row, "nodes": N, "elems": M, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                      "frac_of_peak": round(gbs / peak, 4), "bytes": nbytes}), flush=True)


def sweep(args):
    """Config 5: one bucket of W-1 straddlers plus an excluded 3-parameter
    group, bucket bytes per replica 1 KB .. 1 GB (x16), W in {2, 4, 8, 16},
    bf16 and fp32, reduce-to-owner.  Eager executor flushes and the same step
    replayed from a CUDA graph; inputs above ~2x L2 need no flush between
    launches, smaller ones rotate over enough copies to exceed it."""
    import numpy as np
    import torch
    import datagen
    import zero_collectives_gb300 as zc
    from datagen import BF16, F32, NORMAL, workloads
    torch.cuda.set_device(0)
    zc.set_flush_path({"auto": zc.PATH_AUTO, "ldg": zc.PATH_LDG, "tma": zc.PATH_TMA}[args.flush_path])
    peak, _ = peaks()
    s = torch.cuda.current_stream()
    l2 = 129 * 2**20
    for W in [int(w) for w in args.sweep_worlds.split(",")]:
        for dt, code in ((torch.bfloat16, BF16), (torch.float32, F32)):
            esize = 2 if code == BF16 else 4
            for kb in [int(k) for k in args.sweep_kb.split(",")]:
                elems = max(kb * 1024 // esize, 64 * W)
                tree = workloads.straddle_tree(W, elems, W - 1, pieces=2)
                ex_sizes = np.array([96, 64, 32], np.int64)
                numel = np.concatenate([tree.numel, ex_sizes])
                groups = [(None, tree.numel), (list(range(max(1, W // 2))), ex_sizes)]
                full = workloads.Tree([f"p{i}" for i in range(len(numel))], numel)
                layout = workloads.arrival_layout(full, capacity=None)
                copies = max(1, -(-2 * l2 // (W * full.total * esize)))
                gs = []
                for c in range(copies):
                    g = torch.empty((W, full.total), dtype=dt, device="cuda")
                    datagen.fill_device(g.data_ptr(), W, full.total, full.total, code, NORMAL, 6 + c, 0, 1, 0, 1e-3,
                                        s.cuda_stream)
                    gs.append(g)
                exs = [zc.Zero1Executor(W, numel, layout.row_offset, [(b.start, b.tasks) for b in layout.buckets], dt,
                                        groups=groups) for _ in range(copies)]
                for e, g in zip(exs, gs):
                    e.flush_all(g)
                nbytes = W * full.total * esize + sum(
                    int(full.numel[p]) * esize * (1 if exs[0].omap.owner[p] >= 0 else
                                                  int(exs[0].omap.holder_hi[p] - exs[0].omap.holder_lo[p]) + 1)
                    for p in range(full.n_params))
                reps = int(min(2000, max(20, 0.05 / max(nbytes / (peak * 1e9), 1e-6))))
                reps = max(copies, reps - reps % copies)

                def eager():
                    for e, g in zip(exs, gs):
                        e.flush_all(g)

                # the same flushes as direct dpred_flush_bucket calls, each
                # bucket's arguments marshalled once (zc.BucketFlush, as a
                # training loop keeps them; the plan cache serves the plan),
                # with and without the overlap promise (the copies share no byte)
                calls = {ov: [zc.BucketFlush(g[:, s0:s0 + size], t, e.omap.owner, tab, code, overlap=ov)
                              for e, g in zip(exs, gs) for (s0, t), size, tab in zip(e.buckets, e.sizes, e.tables)]
                         for ov in (False, True)}

                def per_call(overlap):
                    for c in calls[overlap]:
                        c()

                side = torch.cuda.Stream()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=side):
                    eager()
                # the per-call flushes with the overlap promise, captured once
                # (programmatic launch dependencies become graph edges)
                per_call(True)
                torch.cuda.synchronize()
                graph_o = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph_o, stream=side):
                    per_call(True)
                clocks = Clocks(smi_gpu_id(torch.cuda.current_device()))
                clocks.start()
                ms_e = timed(eager, reps // copies, warm=3) / copies
                ms_g = timed(graph.replay, reps // copies, warm=3) / copies
                ms_c = timed(lambda: per_call(False), reps // copies, warm=3) / copies
                ms_o = timed(lambda: per_call(True), reps // copies, warm=3) / copies
                ms_go = timed(graph_o.replay, reps // copies, warm=3) / copies
                clk = clocks.stop()
                line = {"sweep": True, "flush_path": args.flush_path, "world": W, "dtype": "bf16" if code == BF16 else "f32",
                        "bucket_bytes_per_replica": full.total * esize, "elems": full.total, "copies": copies,
                        "bytes": nbytes, "eager_us": round(ms_e * 1e3, 2), "graph_us": round(ms_g * 1e3, 2),
                        "eager_GBps": round(nbytes / (ms_e * 1e-3) / 1e9, 1),
                        "graph_GBps": round(nbytes / (ms_g * 1e-3) / 1e9, 1),
                        "graph_frac_of_peak": round(nbytes / (ms_g * 1e-3) / 1e9 / peak, 4),
                        "eager_frac_of_peak": round(nbytes / (ms_e * 1e-3) / 1e9 / peak, 4),
                        "per_call_us": round(ms_c * 1e3, 2),
                        "per_call_frac_of_peak": round(nbytes / (ms_c * 1e-3) / 1e9 / peak, 4),
                        "per_call_overlap_us": round(ms_o * 1e3, 2),
                        "per_call_overlap_frac_of_peak": round(nbytes / (ms_o * 1e-3) / 1e9 / peak, 4),
                        "graph_overlap_us": round(ms_go * 1e3, 2),
                        "graph_overlap_frac_of_peak": round(nbytes / (ms_go * 1e-3) / 1e9 / peak, 4),
                        "sm_mhz": clk["sm_mhz"], "mem_mhz_min": clk["mem_mhz_min"], "clock_reasons": clk["reasons"]}
                print(json.dumps(line), flush=True)
                for e in exs:
                    e.close()
                del gs, exs, graph, graph_o
                torch.cuda.empty_cache()


def main():
    args = parse()
    if args.sweep:
        sweep(args)
    elif args.row is not None:
        single_row(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_dpred(args)


if __name__ == "__main__":
    main()
