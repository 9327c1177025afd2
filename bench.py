#!/usr/bin/env python3
"""KV page backup (D2H) / restore (H2D) throughput on one GB300 (or N replicas).

Default workload: the Llama-8B-shaped pool (32 layers x {K,V} x 8 KV heads x
head_dim 128 bf16, page 16 tokens, 4096 pages, layer-first NHD; 8 GiB) with a
page-contiguous pinned host tier of 512 slots (1 GiB).  One step = back up 512
seeded-random pages to slots 0..511, then restore all 512 into 512 other
random pages: 1 GiB each way across the host link.  Inputs are synthetic
(seeded random bytes; bf16 values are opaque bytes on this path).

Printed (rank 0, one JSON line): device-timed throughput of the step
(``value``), the same through the C ABI on the host clock (``e2e``), the host
link's pinned-memcpy peak measured in the same run, per-direction GB/s and %
of that peak, the roofline of the dominant kernel, SM clocks sampled during
the timed region, and the CPU oracle timed on the host cores as a baseline.
``--impl reference`` times the CPU oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

METRIC = "KV page backup/restore GB/s (D2H, H2D, 1 GB300) and % of measured host-link peak"
GB = 1e9


def parse():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["llama8b", "mla_fp8", "trtllm_ipc"], default="llama8b")
    p.add_argument("--mode", choices=["zero_copy", "staged", "copy_engine"], default="zero_copy")
    p.add_argument("--max-ctas", type=int, default=0)
    p.add_argument("--staging-mib", type=int, default=0,
                   help="STAGED mode: device staging buffer in MiB (0 = library default)")
    p.add_argument("--cta-threads", type=int, default=0, choices=[0, 256, 1024],
                   help="threads per CTA of host-link moves (0 = library default)")
    p.add_argument("--no-bulk", action="store_true",
                   help="HBM-only moves use the register kernel instead of bulk copies")
    p.add_argument("--no-pdl", action="store_true",
                   help="host-link moves launch without programmatic dependent launch")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def dist_max(x: float, dist, device=None) -> float:
    """Max of a per-rank time over all ranks (the job is as slow as its slowest rank)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, steps: int, ranks: int, max_elapsed_s: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return ranks * bytes_per_rank_step * steps / max_elapsed_s / GB


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_sha():
    """Hash of the kernels' code (comments and blank space removed), so that
    recorded profiler figures stay attached to the code they were taken on."""
    import re

    h = hashlib.sha256()
    for rel in ("hierarchical_kv_cache_backup_gb300/csrc/kvb_kernels.cu",
                "hierarchical_kv_cache_backup_gb300/csrc/kvb_internal.h"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch from a committed ncu summary, if taken on this kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except OSError:
        return None
    if t.get("kernel_sha") != kernel_sha():
        return None
    return t.get(key)


class ClockSampler:
    """nvidia-smi clock / throttle samples over the timed region.  nvidia-smi is
    started before the warm-up (its start-up touches the driver) and every line
    is timestamped; summary() keeps the samples taken between mark() and
    stop()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.1

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(int(1000 * self.PERIOD_S))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            atexit.register(self._kill)   # an exception before stop() leaves no sampler behind
        except OSError:
            self.proc = None
        return self

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self):
        self.t0 = time.monotonic()

    def stop(self):
        self.t1 = time.monotonic()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def window_lines(self):
        t0 = self.t0 if self.t0 is not None else 0.0
        t1 = (self.t1 if self.t1 is not None else time.monotonic()) + self.PERIOD_S
        inside = [ln for ts, ln in self.lines if t0 <= ts <= t1]
        if not inside:   # a window shorter than one period: the first sample after it began
            inside = [ln for ts, ln in self.lines if ts >= t0][:1]
        return inside

    def summary(self):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not found"}
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.window_lines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"unavailable": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(pw), "reasons": sorted(reasons)}


def _exporter(q, done, device, seed, pool_offset):
    """Second process of the TRT-LLM workload: owns the pool allocation (a raw
    allocation with the pool at a byte offset), exports it over CUDA IPC and
    keeps it alive until the benchmark is done with it."""
    import torch

    sys.path.insert(0, ROOT)
    from hierarchical_kv_cache_backup_gb300 import kvb as k

    torch.cuda.set_device(device)
    g = wl.TRTLLM.geom
    alloc = torch.empty(pool_offset + g.pool_bytes, dtype=torch.uint8, device=f"cuda:{device}")
    wl.fill_random_(alloc, seed)
    torch.cuda.synchronize()
    lay = k.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    pool = k.kv_pool_register(lay, alloc.data_ptr(), pool_offset, instance_id=os.getpid(),
                              generation=1)
    q.put(k.desc_to_bytes(k.kv_pool_export(pool)))
    done.wait(3600)
    k.kv_pool_close(pool)


# ------------------------------------------------------------- CPU oracle leg

def oracle_sample(cpu_seconds: float, steps: int | None = None, n_sample: int = 512,
                  pool_pages: int = 1024, threads: int | None = None):
    """Times the CPU oracle (as it stands) on the host cores: backup of n_sample
    random pages of the Llama-8B geometry, then restore into n_sample others, on a
    pool of ``pool_pages`` pages, with ``threads`` threads (all cores by default).
    Returns (GB/s, threads, sample text, per-step s)."""
    import oracle

    g = wl.LLAMA8B.geom.with_(P=pool_pages)
    og = oracle.geom(g.L, g.C, g.P, g.T, g.H, g.B)
    pool = np.full(g.pool_bytes, 7, dtype=np.uint8)
    host = np.full(n_sample * g.page_bytes, 3, dtype=np.uint8)
    cores = threads or len(os.sched_getaffinity(0))
    r = wl.rng(wl.LLAMA8B.seed)
    per_step = 2 * n_sample * g.page_bytes
    times = []
    used = 1
    t_all = time.perf_counter()
    k = 0
    while True:
        src = wl.distinct_pages(r, g.P, n_sample)
        dst = wl.distinct_pages(r, g.P, n_sample, exclude=src)
        slots = np.arange(n_sample, dtype=np.int32)
        t0 = time.perf_counter()
        used = oracle.backup(og, pool, host, src, slots, threads=cores)
        oracle.restore(og, pool, host, slots, dst, threads=cores)
        times.append(time.perf_counter() - t0)
        k += 1
        if steps is not None:
            if k >= steps:
                break
        elif (time.perf_counter() - t_all >= cpu_seconds and k >= 2) or k >= 200:
            break
    total = sum(times)
    sample = (f"{k} x (backup {n_sample} random pages + restore {n_sample}) of the Llama-8B "
              f"geometry on a {pool_pages}-page host pool ({per_step / 2**20:.0f} MiB per step)")
    return per_step * k / total / GB, used, sample, times


def numpy_statement_sample(cpu_seconds: float, n_sample: int = 64, pool_pages: int = 128):
    """Times the oracle's numpy statement (views and fancy indexing, one thread)
    as it stands on the Llama-8B geometry: backup of n_sample random pages, then
    restore into n_sample others.  Each call returns a new array, so a restore
    also copies the whole pool: the figure depends on the pool's size, stated in
    the sample.  Returns (GB/s, sample text)."""
    from oracle import numpy_statement as nps

    g = wl.LLAMA8B.geom.with_(P=pool_pages)
    pool = np.full(g.pool_bytes, 7, dtype=np.uint8)
    host = np.full(n_sample * g.page_bytes, 3, dtype=np.uint8)
    r = wl.rng(wl.LLAMA8B.seed + 1)
    per_step = 2 * n_sample * g.page_bytes
    times = []
    t_all = time.perf_counter()
    while not times or (time.perf_counter() - t_all < cpu_seconds and len(times) < 200):
        src = wl.distinct_pages(r, g.P, n_sample)
        dst = wl.distinct_pages(r, g.P, n_sample, exclude=src)
        slots = np.arange(n_sample, dtype=np.int32)
        t0 = time.perf_counter()
        host = nps.backup(pool, g, g.order, g.dev_heads, host, n_sample, g.host_heads, src, slots)
        pool = nps.restore(pool, g, g.order, g.dev_heads, host, n_sample, g.host_heads, slots,
                           dst, -1)
        times.append(time.perf_counter() - t0)
    sample = (f"{len(times)} x (backup {n_sample} random pages + restore {n_sample}) of the "
              f"Llama-8B geometry on a {pool_pages}-page host pool ({per_step / 2**20:.0f} MiB "
              f"moved per step; each restore also copies the {g.pool_bytes / 2**20:.0f} MiB pool)")
    return per_step * len(times) / sum(times) / GB, sample


def run_reference(args):
    rank, _, ws = dist_env()
    if rank != 0:
        return
    w = wl.LLAMA8B
    # the reference arm: the oracle on the host cores, a bounded sample per step
    n_sample = 64
    oracle_sample(0, steps=max(1, args.warmup), n_sample=n_sample)
    gbs, used, sample, times = oracle_sample(0, steps=max(1, args.steps), n_sample=n_sample)
    ms = 1000 * statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    g = w.geom
    return {"workload": f"{w.name}: L{g.L} x C{g.C} x H{g.H} x T{g.T} x {g.B} B per head vector, "
                        f"{g.P} pages ({g.pool_bytes / 2**30:.1f} GiB) "
                        f"{'page' if g.order else 'layer'}-first "
                        f"{'HND' if g.dev_heads else 'NHD'}, host tier "
                        f"{'HND' if g.host_heads else 'NHD'}",
            "pages_per_op": w.n, "page_bytes": g.page_bytes,
            "cache": "inputs larger than L2: 1 GiB+ per direction from random pages of a "
                     "multi-GiB pool; no flush needed"}


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    from hierarchical_kv_cache_backup_gb300 import build as kbuild

    kbuild.build_library()
    from hierarchical_kv_cache_backup_gb300 import kvb

    rank, local, ws = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mode = {"zero_copy": kvb.KV_MODE_ZERO_COPY, "staged": kvb.KV_MODE_STAGED,
            "copy_engine": kvb.KV_MODE_COPY_ENGINE}[args.mode]
    kvb.kv_config_set(mode, args.max_ctas, args.staging_mib << 20,
                      (kvb.KV_CFG_NO_BULK if args.no_bulk else 0) |
                      (kvb.KV_CFG_NO_PDL if args.no_pdl else 0), args.cta_threads)

    w = {"llama8b": wl.LLAMA8B, "mla_fp8": wl.MLA_FP8, "trtllm_ipc": wl.TRTLLM}[args.workload]
    g = w.geom
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    exporter = None
    host = torch.empty(w.host_slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    if w is wl.TRTLLM:
        # the pool lives in a second process and is imported over CUDA IPC
        import multiprocessing as mp

        ctx = mp.get_context("spawn")
        q, done_ev = ctx.Queue(), ctx.Event()
        exporter = ctx.Process(target=_exporter,
                               args=(q, done_ev, local, w.seed + 100 * rank, w.pool_offset))
        exporter.start()
        pool = kvb.kv_pool_import(kvb.desc_from_bytes(q.get(timeout=900)))
        alloc = torch.empty(2 << 30, dtype=torch.uint8, device=dev)   # probe buffer only
        wl.fill_random_(alloc, w.seed + 7)
        for lo in range(0, host.numel(), alloc.numel()):
            hi = min(host.numel(), lo + alloc.numel())
            host[lo:hi].copy_(alloc[:hi - lo])
    else:
        alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8, device=dev)
        wl.fill_random_(alloc, w.seed + 100 * rank)
        host.copy_(alloc[:host.numel()])
        pool = kvb.kv_pool_register(lay, alloc.data_ptr(), w.pool_offset)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), w.host_slots, g.host_heads, lay)
    s_a = torch.cuda.Stream(device=dev)
    s_b = torch.cuda.Stream(device=dev)
    R = 8
    idsets = [wl.op_ids(w, seed=w.seed + 17 * k + 1000 * rank) for k in range(R)]

    # ---- host-link peak, measured in this run: pinned cudaMemcpyAsync, 2 GiB, best of 10
    link = {}
    probe_n = 2 << 30
    pin = torch.empty(probe_n, dtype=torch.uint8, pin_memory=True)
    dbuf = alloc[:probe_n] if alloc.numel() >= probe_n else torch.empty(probe_n, dtype=torch.uint8,
                                                                          device=dev)
    pin2 = torch.empty(probe_n // 2, dtype=torch.uint8, pin_memory=True)
    dbuf2 = torch.empty(probe_n // 2, dtype=torch.uint8, device=dev)

    def best_of(fn, nbytes, reps=10):
        ts = []
        for i in range(reps + 3):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_a)
            fn()
            e1.record(s_a)
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) / 1000)
        return nbytes / min(ts) / GB

    with torch.cuda.stream(s_a):
        link["d2h"] = best_of(lambda: pin.copy_(dbuf, non_blocking=True), probe_n)
        link["h2d"] = best_of(lambda: dbuf.copy_(pin, non_blocking=True), probe_n)

    def bidir():
        ev = torch.cuda.Event()
        ev.record(s_a)
        s_b.wait_event(ev)
        with torch.cuda.stream(s_a):
            pin[:probe_n // 2].copy_(dbuf[:probe_n // 2], non_blocking=True)
        with torch.cuda.stream(s_b):
            dbuf2.copy_(pin2, non_blocking=True)
        ev2 = torch.cuda.Event()
        ev2.record(s_b)
        s_a.wait_event(ev2)
    link["bidir"] = best_of(bidir, probe_n)
    del pin, pin2, dbuf2
    torch.cuda.empty_cache()

    # ---- one step of the workload (through the C ABI; ids are host arrays)
    bytes_b = bytes_r = 0
    if w is wl.LLAMA8B:
        bytes_b = bytes_r = w.n * g.page_bytes
    elif w is wl.MLA_FP8:
        bytes_r = g.L * w.n * g.layer_page_bytes
    else:
        bytes_b = bytes_r = w.n * g.page_bytes

    def step(k, evs=None):
        ids = idsets[k % R]
        if w is wl.LLAMA8B:
            if evs:
                evs[0].record(s_a)
            kvb.kv_backup(pool, tier, ids.backup_src, ids.backup_slots, s_a.cuda_stream)
            if evs:
                evs[1].record(s_a)
            f = kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, -1, s_a.cuda_stream)
            if evs:
                evs[2].record(s_a)
            return [f]   # same stream: the restore's fence follows the backup
        if w is wl.MLA_FP8:
            if evs:
                evs[0].record(s_a)
            f = None
            for l in range(g.L):
                f = kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, l,
                                   s_a.cuda_stream)
            if evs:
                evs[1].record(s_a)
                evs[2].record(s_a)
            return [f]
        # trtllm: backup on stream A and restore on stream B at the same time
        ev = torch.cuda.Event()
        ev.record(s_a)
        s_b.wait_event(ev)
        if evs:
            evs[0].record(s_a)
        fb = kvb.kv_backup(pool, tier, ids.backup_src, ids.backup_slots, s_a.cuda_stream)
        if evs:
            evs[1].record(s_a)
        if evs:
            evs[3].record(s_b)
        fr = kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, -1, s_b.cuda_stream)
        if evs:
            evs[4].record(s_b)
        ev2 = torch.cuda.Event()
        ev2.record(s_b)
        s_a.wait_event(ev2)
        if evs:
            evs[2].record(s_a)
        return [fb, fr]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local).start()   # before the warm-up: its start-up is not timed
    for k in range(args.warmup):
        step(k)
    barrier()

    # ---- timed region: device clock (CUDA events on the launching stream)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    l0 = kvb.kv_launch_count()
    barrier()
    clk.mark()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(s_a)
    for k in range(args.steps):
        step(k, evs[k])
    t_end.record(s_a)
    barrier()
    clk.stop()
    launches = kvb.kv_launch_count() - l0
    elapsed = dist_max(t_start.elapsed_time(t_end) / 1000, dist, dev)
    b_ms = [e[0].elapsed_time(e[1]) for e in evs]
    r_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if w is wl.TRTLLM:   # the restore ran on stream B, bracketed by its own events
        r_ms = [e[3].elapsed_time(e[4]) for e in evs]
    step_bytes = bytes_b + bytes_r
    value = job_gbs(step_bytes, args.steps, ws, elapsed)

    # ---- end to end through the C ABI, host clock, fence wait every step
    barrier()
    t0 = time.perf_counter()
    for k in range(args.steps):
        for f in step(k):
            kvb.kv_fence_wait(f, 60_000_000_000)
    e2e_s = dist_max(time.perf_counter() - t0, dist, dev)
    e2e = job_gbs(step_bytes, args.steps, ws, e2e_s)

    # ---- device-side layout-transform gather (staged half) against HBM
    peaks, peak_src = measured_peaks()
    hbm = None
    if w is not wl.MLA_FP8:
        n = w.n
        buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device=dev)
        gathers = 10      # back to back, so each launch is issued while the GPU is busy

        def gather_gbs(with_fence):
            ts = []
            for i in range(4):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(s_a)
                for k in range(gathers):
                    kvb.kv_device_gather(pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                         idsets[(i + k) % R].backup_src, s_a.cuda_stream,
                                         fence=with_fence)
                e1.record(s_a)
                e1.synchronize()
                if i >= 1:
                    ts.append(e0.elapsed_time(e1) / 1000 / gathers)
            return 2 * n * g.page_bytes / statistics.median(ts) / GB

        gb_s = gather_gbs(True)          # the roofline: with its fence, as a backup has
        gb_s_ordered = gather_gbs(False)  # stream order only (fence = NULL)
        hbm = {"bound": "hbm", "kernel": ("kv_move_kernel" if args.no_bulk else
                                          "kv_tsp_kernel" if g.dev_heads != g.host_heads else
                                          "kv_bulk_kernel") +
                         " (device gather, pool -> device buffer in host layout)",
               "achieved": round(gb_s, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
               "frac": round(gb_s / peaks["hbm_gbs"], 4),
               "traffic": recorded_traffic("device_gather_transposed_dram_bytes_per_launch"
                                           if g.dev_heads != g.host_heads else
                                           "device_gather_dram_bytes_per_launch"),
               "algorithmic_bytes_per_launch": 2 * n * g.page_bytes,
               "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_src})",
               "achieved_without_fence": round(gb_s_ordered, 1),
               "frac_without_fence": round(gb_s_ordered / peaks["hbm_gbs"], 4)}
        del buf

    # ---- MLA: the same 61 layers restored by one progressive call per step
    progressive = None
    if w is wl.MLA_FP8:
        ts = []
        for k in range(args.warmup + args.steps):
            ids = idsets[k % R]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_a)
            kvb.kv_restore_layers(pool, tier, ids.restore_slots, ids.restore_dst, 0, g.L,
                                  s_a.cuda_stream)
            e1.record(s_a)
            if k >= args.warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        sec = statistics.mean(a.elapsed_time(b) for a, b in ts) / 1000
        progressive = {"call": "kv_restore_layers: 61 layers x 64 pages in one call, per-layer "
                               "fences published as the restored prefix grows",
                       "gbs": round(bytes_r / sec / GB, 2), "ms_per_step": round(1000 * sec, 4)}

    # ---- MLA: overlap of the layer-wise restore with each layer's forward.  A
    # stand-in forward (one bf16 GEMM per layer, sized near one layer's transfer
    # time) runs on a compute stream that waits, on the GPU, for that layer's
    # fence; exposed transfer = pipelined time - compute-only time.
    overlap = None
    if w is wl.MLA_FP8:
        comp = torch.cuda.Stream(device=dev)
        M = 3456
        A = torch.randn(M, M, dtype=torch.bfloat16, device=dev)
        Bm = torch.randn(M, M, dtype=torch.bfloat16, device=dev)
        Cm = torch.empty(M, M, dtype=torch.bfloat16, device=dev)

        def timed(fn, stream, reps=5):
            out = []
            for i in range(reps + 2):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(i)
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    out.append(e0.elapsed_time(e1))
            return statistics.median(out)

        def compute_only(i):
            with torch.cuda.stream(comp):
                for _ in range(g.L):
                    torch.matmul(A, Bm, out=Cm)

        def restore_only(i):
            ids = idsets[i % R]
            for l in range(g.L):
                kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, l, s_a.cuda_stream)

        def pipelined(i, progressive):
            ids = idsets[i % R]
            ev = torch.cuda.Event()
            ev.record(comp)
            s_a.wait_event(ev)
            if progressive:
                fences = kvb.kv_restore_layers(pool, tier, ids.restore_slots, ids.restore_dst, 0,
                                               g.L, s_a.cuda_stream)
            else:
                fences = [kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, l,
                                         s_a.cuda_stream) for l in range(g.L)]
            with torch.cuda.stream(comp):
                for l in range(g.L):
                    kvb.kv_fence_stream_wait(fences[l], comp.cuda_stream)
                    torch.matmul(A, Bm, out=Cm)
            ev2 = torch.cuda.Event()
            ev2.record(comp)
            s_a.wait_event(ev2)

        t_c = timed(compute_only, comp)
        t_r = timed(restore_only, s_a)
        t_p1 = timed(lambda i: pipelined(i, False), s_a)
        t_p2 = timed(lambda i: pipelined(i, True), s_a)
        overlap = {"forward_stand_in": f"bf16 GEMM {M}^3 per layer on a compute stream, 61 layers",
                   "compute_only_ms": round(t_c, 3), "restore_only_ms": round(t_r, 3),
                   "pipelined_per_layer_calls_ms": round(t_p1, 3),
                   "pipelined_progressive_ms": round(t_p2, 3),
                   "exposed_transfer_ms_per_layer_calls": round(t_p1 - t_c, 3),
                   "exposed_transfer_ms_progressive": round(t_p2 - t_c, 3)}

        # ---- the SM budget that saturates the host link: the progressive
        # restore (H2D) and a backup of the same 64 pages (D2H) on k whole SMs
        # (k CTAs of 1024 threads, one per SM), alone and, for the restore,
        # pipelined with the stand-in forward above
        def restore_prog(i):
            ids = idsets[i % R]
            kvb.kv_restore_layers(pool, tier, ids.restore_slots, ids.restore_dst, 0, g.L,
                                  s_a.cuda_stream)

        def backup_pages(i):
            ids = idsets[i % R]
            kvb.kv_backup(pool, tier, ids.restore_dst, ids.restore_slots, s_a.cuda_stream)

        cfg0 = kvb.kv_config_get()
        budget = []
        try:
            for k in (1, 2, 3, 4, 6, 8, 12, 16):
                kvb.kv_config_set(cfg0.mode, k, cfg0.staging_bytes, cfg0.flags, 1024)
                t_rk = timed(restore_prog, s_a)
                t_bk = timed(backup_pages, s_a)
                t_pk = timed(lambda i: pipelined(i, True), s_a)
                t_lk = timed(restore_only, s_a)
                t_qk = timed(lambda i: pipelined(i, False), s_a)
                budget.append({"sms": k,
                               "restore_gbs": round(bytes_r / t_rk * 1000 / GB, 2),
                               "restore_pct_h2d": round(100 * bytes_r / t_rk * 1000 / GB /
                                                        link["h2d"], 1),
                               "backup_gbs": round(bytes_r / t_bk * 1000 / GB, 2),
                               "backup_pct_d2h": round(100 * bytes_r / t_bk * 1000 / GB /
                                                       link["d2h"], 1),
                               "pipelined_progressive_ms": round(t_pk, 3),
                               "per_layer_calls_gbs": round(bytes_r / t_lk * 1000 / GB, 2),
                               "pipelined_per_layer_calls_ms": round(t_qk, 3)})
        finally:
            kvb.kv_config_set(cfg0.mode, cfg0.max_ctas, cfg0.staging_bytes, cfg0.flags,
                              cfg0.cta_threads)
        overlap["sm_budget"] = {
            "what": "k CTAs of 1024 threads (k whole SMs): kv_restore_layers of 61 layers x 64 "
                    "pages (H2D), kv_backup of the same 64 pages (D2H) and the 61 one-layer "
                    "kv_restore calls, each alone (median of 5), and both restores pipelined "
                    "with the per-layer GEMMs",
            "rows": budget}
        del A, Bm, Cm

        # ---- the 61 one-layer restores as ring descriptors (one per layer, 64
        # pages each), all submitted at once, served by a host thread and by the
        # GPU-resident server; host clock from the first submit to the last
        # ticket, median of 5 steps after one.  The resident server launches
        # nothing per descriptor.
        ring_layers = {}
        steps_l = 6
        for kind in ("host", "device"):
            name = f"/kvbbenchly_{os.getpid()}_{kind}"
            sub = kvb.kv_ring_create(name, 64)
            srv = kvb.kv_ring_attach(name)
            rs = torch.cuda.Stream(device=dev)
            stop = threading.Event()
            served = [0]

            def serve_layers():
                while not stop.is_set() and served[0] < g.L * steps_l:
                    served[0] += kvb.kv_ring_serve(srv, [pool], tier, rs.cuda_stream, 64,
                                                   200_000_000)

            th, fence = None, None
            if kind == "host":
                th = threading.Thread(target=serve_layers, daemon=True)
                th.start()
            else:
                fence = kvb.kv_ring_serve_device(srv, [pool], tier, rs.cuda_stream,
                                                 g.L * steps_l, 5_000_000_000)
            times = []
            for i in range(steps_l):
                ids = idsets[i % R]
                ops = [kvb.make_ring_op(1, ids.restore_slots, ids.restore_dst, layer=l)
                       for l in range(g.L)]
                t0 = time.perf_counter()
                tks = [kvb.kv_ring_submit(sub, op) for op in ops]
                sts = [kvb.kv_ring_wait(sub, tk, 30_000_000_000) for tk in tks]
                times.append(time.perf_counter() - t0)
                if any(sts):
                    raise RuntimeError(f"ring {kind} layer step {i}: statuses {sts}")
            if fence is not None:
                kvb.kv_fence_wait(fence, 30_000_000_000)
            stop.set()
            if th is not None:
                th.join(10)
            rs.synchronize()
            kvb.kv_ring_close(srv)
            kvb.kv_ring_close(sub)
            t_med = statistics.median(times[1:])
            ring_layers[f"{kind}_served_gbs"] = round(bytes_r / t_med / GB, 2)
            ring_layers[f"{kind}_served_us_per_layer"] = round(1e6 * t_med / g.L, 2)
        ring_layers["workload"] = ("61 one-layer restore descriptors of 64 pages (9,437,184 B "
                                   "each) submitted at once, host clock from the first submit "
                                   "to the last ticket, median of 5 steps after one")
        overlap["ring_one_layer_descriptors"] = ring_layers

    # ---- Llama-8B: write-through backup beside the prefill that fills the pages.
    # The step's 512 pages are written by 8 chunks of a stand-in forward (bf16
    # GEMMs on a compute stream, sized near one chunk's backup time); each chunk's
    # 64 pages are backed up on the copy stream once that chunk's forward is done
    # (a GPU-side event wait), so the backup of chunk k runs beside the forward of
    # chunk k + 1.  Exposed backup = pipelined - compute-only; the last chunk's
    # backup can never overlap and is reported beside it.
    write_through = None
    if w is wl.LLAMA8B:
        comp = torch.cuda.Stream(device=dev)
        M, per_chunk, chunks = 3456, 16, 8
        A = torch.randn(M, M, dtype=torch.bfloat16, device=dev)
        Bm = torch.randn(M, M, dtype=torch.bfloat16, device=dev)
        Cm = torch.empty(M, M, dtype=torch.bfloat16, device=dev)
        cp = w.n // chunks

        def wt_timed(fn, reps=5):
            out = []
            for i in range(reps + 2):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s_a)
                ev = torch.cuda.Event()
                ev.record(s_a)
                comp.wait_event(ev)
                fn(i)
                ev2 = torch.cuda.Event()
                ev2.record(comp)
                s_a.wait_event(ev2)
                e1.record(s_a)
                e1.synchronize()
                if i >= 2:
                    out.append(e0.elapsed_time(e1))
            return statistics.median(out)

        def wt_compute(i):
            with torch.cuda.stream(comp):
                for _ in range(chunks * per_chunk):
                    torch.matmul(A, Bm, out=Cm)

        def wt_backup(i, last_only=False):
            ids = idsets[i % R]
            for c in range(chunks - 1 if last_only else 0, chunks):
                sl = slice(c * cp, (c + 1) * cp)
                kvb.kv_backup(pool, tier, ids.backup_src[sl], ids.backup_slots[sl],
                              s_a.cuda_stream)

        def wt_pipelined(i):
            ids = idsets[i % R]
            for c in range(chunks):
                with torch.cuda.stream(comp):
                    for _ in range(per_chunk):
                        torch.matmul(A, Bm, out=Cm)
                done = torch.cuda.Event()
                done.record(comp)
                s_a.wait_event(done)
                sl = slice(c * cp, (c + 1) * cp)
                kvb.kv_backup(pool, tier, ids.backup_src[sl], ids.backup_slots[sl],
                              s_a.cuda_stream)

        t_c = wt_timed(wt_compute)
        t_b = wt_timed(wt_backup)
        t_last = wt_timed(lambda i: wt_backup(i, True))
        t_p = wt_timed(wt_pipelined)
        write_through = {
            "forward_stand_in": f"bf16 GEMM {M}^3 x {per_chunk} per chunk on a compute stream",
            "chunks": chunks, "pages_per_chunk": cp,
            "compute_only_ms": round(t_c, 3), "backup_only_ms": round(t_b, 3),
            "pipelined_ms": round(t_p, 3), "exposed_backup_ms": round(t_p - t_c, 3),
            "last_chunk_backup_ms": round(t_last, 3),
            "exposed_beyond_last_chunk_ms": round(t_p - t_c - t_last, 3)}
        del A, Bm, Cm

    # ---- Llama-8B: the hop below the host tier.  The step's 512 backed-up host
    # slots (1 GiB) are put into 512 records of a memfd and got back, on the
    # host cores (host memory bandwidth bound; no GPU work).
    l3 = None
    if w is wl.LLAMA8B and hasattr(os, "memfd_create"):
        fd = os.memfd_create("kvb_bench_l3")
        threads = min(16, len(os.sched_getaffinity(0)))
        store = kvb.kv_l3_open(fd, 0, g.page_bytes, w.n, threads)
        ids = idsets[0]
        recs = np.arange(w.n, dtype=np.int32)
        kvb.kv_l3_put(store, host.data_ptr(), w.host_slots, ids.backup_slots, recs)  # grows it
        tp, tg = [], []
        for _ in range(5):
            t0 = time.perf_counter()
            kvb.kv_l3_put(store, host.data_ptr(), w.host_slots, ids.backup_slots, recs)
            t1 = time.perf_counter()
            kvb.kv_l3_get(store, host.data_ptr(), w.host_slots, recs, ids.backup_slots)
            tp.append(t1 - t0)
            tg.append(time.perf_counter() - t1)
        l3 = {"store": f"memfd, {w.n} records of {g.page_bytes} bytes, host clock",
              "threads": threads,
              "put_gbs": round(w.n * g.page_bytes / statistics.median(tp) / GB, 2),
              "get_gbs": round(w.n * g.page_bytes / statistics.median(tg) / GB, 2)}
        kvb.kv_l3_close(store)
        os.close(fd)

    # ---- small-op latency: the tiny workload (8 pages of 16 KiB) through the C ABI
    latency = None
    if w is wl.LLAMA8B:
        t = wl.TINY
        tg = t.geom
        tlay = kvb.make_layout(tg.L, tg.C, tg.P, tg.T, tg.H, tg.B, tg.order, tg.dev_heads,
                               tg.elem_bytes)
        talloc = torch.empty(tg.pool_bytes, dtype=torch.uint8, device=dev)
        wl.fill_random_(talloc, t.seed)
        thost = torch.empty(t.host_slots * tg.page_bytes, dtype=torch.uint8, pin_memory=True)
        tpool = kvb.kv_pool_register(tlay, talloc.data_ptr(), 0)
        ttier = kvb.kv_host_register(thost.data_ptr(), thost.numel(), t.host_slots, 0, tlay)
        # four disjoint source sets, four disjoint destination sets, two slot sets,
        # and L2 flushed before every op (the whole tiny pool would sit in L2)
        perm = wl.rng(t.seed).permutation(tg.P).astype(np.int32)
        srcs = [perm[8 * k:8 * k + 8] for k in range(4)]
        dsts = [perm[32 + 8 * k:40 + 8 * k] for k in range(4)]
        slot_sets = [np.arange(0, 8, dtype=np.int32), np.arange(8, 16, dtype=np.int32)]
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        lat_b, lat_r = [], []
        for i in range(250):
            sl = slot_sets[i % 2]
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            kvb.kv_fence_wait(kvb.kv_backup(tpool, ttier, srcs[i % 4], sl, s_a.cuda_stream),
                              10_000_000_000)
            t1 = time.perf_counter()
            flush.zero_()
            torch.cuda.synchronize()
            t2 = time.perf_counter()
            kvb.kv_fence_wait(kvb.kv_restore(tpool, ttier, sl, dsts[i % 4], -1, s_a.cuda_stream),
                              10_000_000_000)
            t3 = time.perf_counter()
            if i >= 50:
                lat_b.append(t1 - t0)
                lat_r.append(t3 - t2)
        del flush
        latency = {"workload": "tiny: 8 pages x 16 KiB (128 KiB) per op, host clock from the "
                               "C-ABI call to the fence wait returning; 4 disjoint page sets "
                               "in rotation, L2 flushed (256 MiB write) before every op",
                   "backup_us_median": round(1e6 * statistics.median(lat_b), 1),
                   "restore_us_median": round(1e6 * statistics.median(lat_r), 1),
                   "backup_us_p99": round(1e6 * sorted(lat_b)[int(0.99 * len(lat_b))], 1)}
        # ---- descriptor ring round trip (submit -> ticket complete) for the same
        # tiny backups, served by a host thread (kv_ring_serve: pop, validate,
        # launch, GPU completion) and by the GPU-resident server
        # (kv_ring_serve_device: no host thread, no launch per descriptor)
        ring_lat = {}
        iters = 400
        ops = [kvb.make_ring_op(0, srcs[i % 4], slot_sets[i % 2], operation_id=i)
               for i in range(iters)]
        for kind in ("host", "device"):
            name = f"/kvbbench_{os.getpid()}_{kind}"
            sub = kvb.kv_ring_create(name, 64)
            srv = kvb.kv_ring_attach(name)
            rs = torch.cuda.Stream(device=dev)
            stop = threading.Event()
            served = [0]

            def serve_loop():
                while not stop.is_set() and served[0] < iters:
                    served[0] += kvb.kv_ring_serve(srv, [tpool], ttier, rs.cuda_stream, 64,
                                                   200_000_000)

            th, fence = None, None
            if kind == "host":
                th = threading.Thread(target=serve_loop, daemon=True)
                th.start()
            else:
                fence = kvb.kv_ring_serve_device(srv, [tpool], ttier, rs.cuda_stream, iters,
                                                 2_000_000_000)
            lat = []
            half = iters // 2
            for i in range(half):
                t0 = time.perf_counter()
                tk = kvb.kv_ring_submit(sub, ops[i])
                st = kvb.kv_ring_wait(sub, tk, 10_000_000_000)
                lat.append(time.perf_counter() - t0)
                if st != kvb.KV_OK:
                    raise RuntimeError(f"ring {kind} op {i}: status {st}")
            # the other half back to back, up to 32 in flight: descriptors per second
            t0 = time.perf_counter()
            tks = []
            for i in range(half, iters):
                if len(tks) >= 32:
                    if kvb.kv_ring_wait(sub, tks.pop(0), 10_000_000_000) != kvb.KV_OK:
                        raise RuntimeError(f"ring {kind}: a streamed descriptor failed")
                tks.append(kvb.kv_ring_submit(sub, ops[i]))
            for tk in tks:
                if kvb.kv_ring_wait(sub, tk, 10_000_000_000) != kvb.KV_OK:
                    raise RuntimeError(f"ring {kind}: a streamed descriptor failed")
            ring_lat[f"{kind}_served_descriptors_per_s"] = round((iters - half) /
                                                                 (time.perf_counter() - t0))
            if fence is not None:
                kvb.kv_fence_wait(fence, 30_000_000_000)
            stop.set()
            if th is not None:
                th.join(10)
            rs.synchronize()
            kvb.kv_ring_close(srv)
            kvb.kv_ring_close(sub)
            lat = lat[20:]
            ring_lat[f"{kind}_served_us_median"] = round(1e6 * statistics.median(lat), 1)
            ring_lat[f"{kind}_served_us_p99"] = round(1e6 * sorted(lat)[int(0.99 * len(lat))], 1)
        ring_lat["workload"] = ("tiny: 8 pages x 16 KiB (128 KiB) backup per descriptor, submit "
                                "to ticket complete on the host clock, one descriptor in flight "
                                "(180 timed after 20), then 200 back to back with up to 32 in "
                                "flight (descriptors per second); 4 page sets in rotation, L2 warm")
        latency["ring_round_trip"] = ring_lat
        # ---- descriptor ring throughput: each step is the Llama-8B step as 8
        # descriptors (4 backups of 128 pages, then 4 restores of 128 pages), all
        # submitted at once, host clock from the first submit to the last ticket
        ring_tp = {}
        steps_r = 6
        per = w.n // 4
        for kind in ("host", "device"):
            name = f"/kvbbenchtp_{os.getpid()}_{kind}"
            sub = kvb.kv_ring_create(name, 16)
            srv = kvb.kv_ring_attach(name)
            rs = torch.cuda.Stream(device=dev)
            stop = threading.Event()
            served = [0]

            def serve_loop():
                while not stop.is_set() and served[0] < 8 * steps_r:
                    served[0] += kvb.kv_ring_serve(srv, [pool], tier, rs.cuda_stream, 64,
                                                   200_000_000)

            th, fence = None, None
            if kind == "host":
                th = threading.Thread(target=serve_loop, daemon=True)
                th.start()
            else:
                fence = kvb.kv_ring_serve_device(srv, [pool], tier, rs.cuda_stream, 8 * steps_r,
                                                 5_000_000_000)
            times = []
            for i in range(steps_r):
                ids = idsets[i % R]
                ops = [kvb.make_ring_op(0, ids.backup_src[c * per:(c + 1) * per],
                                        ids.backup_slots[c * per:(c + 1) * per]) for c in range(4)]
                ops += [kvb.make_ring_op(1, ids.restore_slots[c * per:(c + 1) * per],
                                         ids.restore_dst[c * per:(c + 1) * per]) for c in range(4)]
                t0 = time.perf_counter()
                tks = [kvb.kv_ring_submit(sub, op) for op in ops]
                sts = [kvb.kv_ring_wait(sub, tk, 30_000_000_000) for tk in tks]
                times.append(time.perf_counter() - t0)
                if any(sts):
                    raise RuntimeError(f"ring {kind} step {i}: statuses {sts}")
            if fence is not None:
                kvb.kv_fence_wait(fence, 30_000_000_000)
            stop.set()
            if th is not None:
                th.join(10)
            rs.synchronize()
            kvb.kv_ring_close(srv)
            kvb.kv_ring_close(sub)
            ring_tp[f"{kind}_served_gbs"] = round(2 * w.n * g.page_bytes /
                                                  statistics.median(times[1:]) / GB, 2)
        # two rings, each with its own resident server: 4 x 64-page backups into
        # slots 0..255 through one, 4 x 64-page restores from slots 256..511
        # through the other (disjoint pages and slots), both directions at once;
        # with the default 32 movers per server and with 64 (kv_config.max_ctas)
        def two_rings_gbs(movers):
            old_cfg = kvb.kv_config_get()
            kvb.kv_config_set(old_cfg.mode, movers, old_cfg.staging_bytes, old_cfg.flags,
                              old_cfg.cta_threads)
            names = [f"/kvbbenchbi_{os.getpid()}_{x}{movers}" for x in "ab"]
            subs = [kvb.kv_ring_create(nm, 16) for nm in names]
            srvs = [kvb.kv_ring_attach(nm) for nm in names]
            streams = [torch.cuda.Stream(device=dev) for _ in names]
            fences = [kvb.kv_ring_serve_device(sv, [pool], tier, st.cuda_stream, 4 * steps_r,
                                               5_000_000_000) for sv, st in zip(srvs, streams)]
            times = []
            q = w.n // 8
            for i in range(steps_r):
                ids = idsets[i % R]
                ops_a = [kvb.make_ring_op(0, ids.backup_src[c * q:(c + 1) * q],
                                          np.arange(c * q, (c + 1) * q)) for c in range(4)]
                ops_b = [kvb.make_ring_op(1, np.arange(w.n // 2 + c * q, w.n // 2 + (c + 1) * q),
                                          ids.restore_dst[c * q:(c + 1) * q]) for c in range(4)]
                t0 = time.perf_counter()
                tks = []
                for oa, ob in zip(ops_a, ops_b):
                    tks.append((0, kvb.kv_ring_submit(subs[0], oa)))
                    tks.append((1, kvb.kv_ring_submit(subs[1], ob)))
                sts = [kvb.kv_ring_wait(subs[j], tk, 30_000_000_000) for j, tk in tks]
                times.append(time.perf_counter() - t0)
                if any(sts):
                    raise RuntimeError(f"two-ring step {i}: statuses {sts}")
            for f in fences:
                kvb.kv_fence_wait(f, 30_000_000_000)
            for h in srvs + subs:
                kvb.kv_ring_close(h)
            kvb.kv_config_set(old_cfg.mode, old_cfg.max_ctas, old_cfg.staging_bytes,
                              old_cfg.flags, old_cfg.cta_threads)
            return round(w.n * g.page_bytes / statistics.median(times[1:]) / GB, 2)

        ring_tp["device_served_two_rings_gbs"] = two_rings_gbs(0)
        ring_tp["device_served_two_rings_64_movers_gbs"] = two_rings_gbs(64)
        ring_tp["workload"] = ("Llama-8B step as 8 ring descriptors (4 x 128-page backups, then "
                               "4 x 128-page restores; 2 GiB), all submitted at once, host clock "
                               "from the first submit to the last ticket, median of 5 steps; "
                               "two_rings: 4 x 64-page backups and 4 x 64-page restores on two "
                               "rings with a resident server each (32 movers, or 64), at once "
                               "(1 GiB per step)")
        latency["ring_throughput"] = ring_tp
        kvb.kv_pool_close(tpool)
        kvb.kv_host_close(ttier)
        del talloc, thost

    # ---- dominant kernel: the backup (D2H) move, or the restore for MLA
    if w is wl.MLA_FP8:
        dom_ms = statistics.mean(b_ms) / g.L
        dom_bytes = w.n * g.layer_page_bytes
        dom_peak, dom_dir = link["h2d"], "h2d"
        kern = "kv_move_kernel (restore of one layer, zero-copy H2D)"
    else:
        dom_ms = statistics.mean(b_ms)
        dom_bytes = bytes_b
        dom_peak, dom_dir = link["d2h"], "d2h"
        kern = {0: "kv_move_kernel (backup, zero-copy D2H)",
                1: "kv_move_kernel + cudaMemcpyAsync (backup, staged D2H)",
                2: "cudaMemcpy2DAsync per page (backup, copy engine D2H)"}[mode]
    achieved = dom_bytes / (dom_ms / 1000) / GB
    roofline = {"bound": "host_link", "kernel": kern, "achieved": round(achieved, 2),
                "peak": round(dom_peak, 2), "unit": "GB/s", "frac": round(achieved / dom_peak, 4),
                # captured on the Llama-8B backup launch only; other workloads: none taken
                "traffic": recorded_traffic("backup_dram_bytes_per_launch")
                if w is wl.LLAMA8B else None,
                "algorithmic_bytes_per_launch": dom_bytes,
                "peak_source": f"pinned cudaMemcpyAsync {dom_dir} of 2 GiB measured in this run, "
                               "best of 10 (host link peak; not in MEASURED_PEAKS.json)"}
    # per-direction device times: the backup on stream A; the restore on stream A
    # after it (llama8b), on stream B beside it (trtllm), or the 61 one-layer calls
    op_b, op_r = (None, b_ms) if w is wl.MLA_FP8 else (b_ms, r_ms)
    backup_gbs = bytes_b / (statistics.mean(op_b) / 1000) / GB if op_b else None
    restore_gbs = bytes_r / (statistics.mean(op_r) / 1000) / GB

    def op_stats(ms, pages):
        return {"median_ms": round(statistics.median(ms), 4), "best_ms": round(min(ms), 4),
                "pages_per_s": round(pages / (statistics.mean(ms) / 1000), 1)}

    per_op = {"restore": op_stats(op_r, w.n)}
    if op_b:
        per_op["backup"] = op_stats(op_b, w.n)
    if w is wl.MLA_FP8:
        per_op["restore"]["per_layer_call_us"] = round(1000 * statistics.mean(op_r) / g.L, 2)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * elapsed / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random bytes; bf16/fp8 KV are opaque bytes)",
        "config": dict(config_of(w), mode=args.mode,
                       step=("backup n pages then restore n pages, one stream"
                             if w is wl.LLAMA8B else
                             "61 one-layer restores of 64 pages on a copy stream"
                             if w is wl.MLA_FP8 else
                             "backup n pages (stream A) while restoring n others (stream B) on "
                             "a pool imported over CUDA IPC from a second process")),
        "backup_gbs": round(backup_gbs, 2) if backup_gbs else None,
        "restore_gbs": round(restore_gbs, 2) if restore_gbs else None,
        "pages_per_s": round(ws * (w.n * (2 if bytes_b else 1)) * args.steps / elapsed, 1),
        "per_op": per_op,
        "host_link_peak_gbs": {k: round(v, 2) for k, v in link.items()},
        "pct_of_host_link_peak": {
            "d2h": round(100 * backup_gbs / link["d2h"], 2) if backup_gbs else None,
            "h2d": round(100 * restore_gbs / link["h2d"], 2) if restore_gbs else None,
            **({"step_vs_bidir_peak": round(100 * value / ws / link["bidir"], 2),
                "note": "d2h / h2d: each direction while the other runs, against its solo peak"}
               if w is wl.TRTLLM else
               {"step_vs_sequential_peak": round(
                   100 * value / ws / (step_bytes / ((bytes_b / link["d2h"] if bytes_b else 0) +
                                                     bytes_r / link["h2d"])), 2)})},
        "roofline": roofline,
        "roofline_hbm": hbm,
        "e2e": {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": bytes_r +
                8 * w.n * (2 if bytes_b else g.L), "d2h_bytes_per_step": bytes_b + 8,
                "note": "host clock around kv_backup/kv_restore with host id arrays and a fence "
                        "wait every step; payload crosses the host link inside the region"},
        "gpu_launches": launches,
        "latency_small_ops": latency,
        "layerwise_progressive": progressive,
        "overlap_with_compute": overlap,
        "write_through": write_through,
        "l3_hop": l3,
        "clocks": clk.summary(),
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        del alloc
        torch.cuda.empty_cache()
        gbs, used, sample, _ = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 3), "unit": "GB/s", "cores": used,
                                "kind": "oracle", "sample": sample}
        gbs1, _, sample1, _ = oracle_sample(max(1.0, args.cpu_seconds / 4), n_sample=64,
                                            threads=1)
        line["cpu_baseline_single_thread"] = {"value": round(gbs1, 3), "unit": "GB/s",
                                              "cores": 1, "kind": "oracle", "sample": sample1}
        gbs2, sample2 = numpy_statement_sample(max(1.0, args.cpu_seconds / 4))
        line["cpu_baseline_numpy_statement"] = {"value": round(gbs2, 3), "unit": "GB/s",
                                                "cores": 1, "kind": "oracle (numpy statement)",
                                                "sample": sample2}
    else:
        line["cpu_baseline"] = None
    kvb.kv_pool_close(pool)
    kvb.kv_host_close(tier)
    if exporter is not None:
        done_ev.set()
        exporter.join(120)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
