#!/usr/bin/env python3
"""KV page backup (D2H) / restore (H2D) throughput on one GB300 (or N replicas).

Headline workload: the Llama-8B-shaped pool (32 layers x {K,V} x 8 KV heads x
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
At N = 1 the line also carries one record per other workload of the pages
(``mla_fp8``: the 16,384-token MLA prefix restored layer by layer, beside a
stand-in forward; ``trtllm_ipc``: backup || restore on a TRT-LLM pool imported
from a second process; ``sweep``: a summary grid of page sizes, batches and
id patterns), each with its own roofline, clocks and CPU baseline.

Other uses:
  --impl reference   the CPU oracle alone, timed on the headline step (the
                     reference arm).
  --profile-case C   one kind of transfer repeated on a small case, for
                     profiler captures (see profiles/).
  --sweep            the full bandwidth sweep (page bytes x batch x ids x
                     direction x mode), written to --out as JSON.
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
WAIT_NS = 60_000_000_000


def parse(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["llama8b", "mla_fp8", "trtllm_ipc"], default="llama8b",
                   help="the headline workload (mla_fp8 adds the SM-budget table and the "
                        "ring-descriptor figures)")
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
    p.add_argument("--overlap", action="store_true",
                   help="KV_CFG_OVERLAP_RESTORES: consecutive disjoint restores may overlap")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-subrecords", action="store_true",
                   help="headline workload only (no mla_fp8 / trtllm_ipc / sweep records)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the headline's oracle baseline sample")
    # profiler cases
    p.add_argument("--profile-case", choices=["backup", "restore", "gather", "scatter",
                                              "restore_layer", "restore_layers"])
    p.add_argument("--geometry", choices=["llama8b", "trtllm", "mla"], default="llama8b")
    p.add_argument("--pool-pages", type=int, default=512)
    p.add_argument("--pages", type=int, default=128)
    p.add_argument("--reps", type=int, default=3)
    # the full sweep
    p.add_argument("--sweep", action="store_true")
    p.add_argument("--out", default="sweep.json")
    p.add_argument("--quick", action="store_true", help="sweep: every other page size and batch")
    p.add_argument("--sweep-pages", type=int, default=8192)
    p.add_argument("--page-bytes", type=int, nargs="*", help="sweep: only these page sizes")
    p.add_argument("--batches", type=int, nargs="*", help="sweep: only these batch sizes")
    return p.parse_args(argv)


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
    """nvidia-smi clock / throttle samples, timestamped.  nvidia-smi is started
    once, before any warm-up (its start-up touches the driver), and runs until
    stop(); summary(t0, t1) keeps the samples taken inside one timed window."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.1

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

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

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self, t0, t1):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not found"}
        lines = list(self.lines)
        inside = [ln for ts, ln in lines if t0 <= ts <= t1 + self.PERIOD_S]
        if not inside:   # a window shorter than one period: the first sample after it began
            inside = [ln for ts, ln in lines if ts >= t0][:1]
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
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


class Window:
    """A timed region on the host clock.  Records hold the Window itself under
    "clocks"; resolve_clocks() replaces it with the samples taken inside it once
    the sampler has stopped (a short region's first sample may arrive later)."""

    def __enter__(self):
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *exc):
        self.t1 = time.monotonic()


def resolve_clocks(obj, clk):
    """Replaces every Window in a (nested) record with its clock summary."""
    if isinstance(obj, dict):
        for k, v in obj.items():
            if isinstance(v, Window):
                obj[k] = clk.summary(v.t0, v.t1)
            else:
                resolve_clocks(v, clk)
    elif isinstance(obj, list):
        for v in obj:
            resolve_clocks(v, clk)


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

def oracle_sample(g: wl.Geometry, n: int, pool_pages: int, cpu_seconds: float,
                  steps: int | None = None, threads: int | None = None, layerwise: bool = False,
                  seed: int = 0, max_steps: int = 200, warmup: int = 0):
    """Times the CPU oracle (as it stands) on the host cores.  One step: backup of
    n random pages into slots 0..n-1, then restore of those slots into n other
    random pages (whole pages), or -- layerwise -- the restore of n slots into n
    random pages one layer per call, every layer.  The pool holds pool_pages pages
    of geometry g.  After `warmup` untimed steps, runs `steps` steps, or until
    cpu_seconds have passed.  Returns (GB/s, threads used, sample text, per-step
    seconds)."""
    import oracle

    gp = g.with_(P=pool_pages)
    og = oracle.geom(gp.L, gp.C, gp.P, gp.T, gp.H, gp.B, page_first=gp.order == wl.PAGE_FIRST,
                     dev_hnd=gp.dev_heads == wl.HND, host_hnd=gp.host_heads == wl.HND)
    pool = np.full(gp.pool_bytes, 7, dtype=np.uint8)
    host = np.full(n * gp.page_bytes, 3, dtype=np.uint8)
    cores = threads or len(os.sched_getaffinity(0))
    r = wl.rng(seed)
    slots = np.arange(n, dtype=np.int32)
    per_step = n * gp.L * gp.layer_page_bytes if layerwise else 2 * n * gp.page_bytes
    times, used, k = [], 1, 0

    def one_step():
        src = wl.distinct_pages(r, gp.P, n)
        dst = wl.distinct_pages(r, gp.P, n, exclude=src)
        t0 = time.perf_counter()
        u = 1
        if layerwise:
            for layer in range(gp.L):
                u = oracle.restore(og, pool, host, slots, dst, layer=layer, threads=cores)
        else:
            u = oracle.backup(og, pool, host, src, slots, threads=cores)
            oracle.restore(og, pool, host, slots, dst, threads=cores)
        return time.perf_counter() - t0, u

    for _ in range(warmup):
        one_step()
    t_all = time.perf_counter()
    while True:
        dt, used = one_step()
        times.append(dt)
        k += 1
        if steps is not None:
            if k >= steps:
                break
        elif (time.perf_counter() - t_all >= cpu_seconds and k >= 2) or k >= max_steps:
            break
    what = (f"{gp.L} one-layer restores of {n} random pages" if layerwise else
            f"backup {n} random pages + restore {n}")
    sample = (f"{k} x ({what}) of the {g.L}x{g.C}x{g.H}x{g.T}x{g.B} B geometry on a "
              f"{pool_pages}-page host pool ({per_step / 2**20:.0f} MiB per step)")
    return per_step * k / sum(times) / GB, used, sample, times


def cpu_record(g, n, pool_pages, seconds, layerwise=False, seed=0):
    gbs, used, sample, _ = oracle_sample(g, n, pool_pages, seconds, layerwise=layerwise, seed=seed)
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": sample}


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


STEP_TEXT = {
    "llama8b": "backup n pages then restore n pages, one stream",
    "mla_fp8": "61 one-layer restores of 64 pages on a copy stream",
    "trtllm_ipc": "backup n pages (stream A) while restoring n others (stream B) on a pool "
                  "imported over CUDA IPC from a second process",
}


def config_of(w):
    """The workload's description: identical in both arms' lines."""
    g = w.geom
    return {"workload": f"{w.name}: L{g.L} x C{g.C} x H{g.H} x T{g.T} x {g.B} B per head vector, "
                        f"{g.P} pages ({g.pool_bytes / 2**30:.1f} GiB) "
                        f"{'page' if g.order else 'layer'}-first "
                        f"{'HND' if g.dev_heads else 'NHD'}, host tier "
                        f"{'HND' if g.host_heads else 'NHD'}",
            "pages_per_op": w.n, "page_bytes": g.page_bytes, "step": STEP_TEXT[w.name],
            "cache": "inputs larger than L2: 1 GiB+ per direction from random pages of a "
                     "multi-GiB pool; no flush needed"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores, timed
    on the headline step itself (backup of 512 random pages of the Llama-8B
    pool into slots 0..511, restore of those slots into 512 other random pages,
    on a 4,096-page pool), `warmup` untimed steps then `steps` timed ones."""
    rank, _, ws = dist_env()
    if rank != 0:
        return
    w = wl.LLAMA8B
    g = w.geom
    gbs, used, sample, times = oracle_sample(g, w.n, g.P, 0, steps=max(1, args.steps),
                                             seed=w.seed + 1, warmup=max(0, args.warmup))
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


# ---------------------------------------------------------------- our arm

class Ctx:
    """What every section of our arm shares: the library, the device, two
    streams, the in-run host-link peaks and the clock sampler."""

    def __init__(self, args):
        import torch

        from hierarchical_kv_cache_backup_gb300 import build as kbuild

        kbuild.build_library()
        from hierarchical_kv_cache_backup_gb300 import kvb

        self.torch, self.kvb, self.args = torch, kvb, args
        self.rank, self.local, self.ws = dist_env()
        self.dist = None
        if self.ws > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
            self.dist = dist
        torch.cuda.set_device(self.local)
        self.dev = torch.device("cuda", self.local)
        self.s_a = torch.cuda.Stream(device=self.dev)
        self.s_b = torch.cuda.Stream(device=self.dev)
        self.peaks, self.peak_src = measured_peaks()
        self.clk = None
        self.link = None
        self.probe_bufs = None   # set by measure_link: 1 GiB each way for bidir_nearby

    def set_config(self, overlap=None, mode=None, max_ctas=None, cta_threads=None):
        a, kvb = self.args, self.kvb
        m = {"zero_copy": kvb.KV_MODE_ZERO_COPY, "staged": kvb.KV_MODE_STAGED,
             "copy_engine": kvb.KV_MODE_COPY_ENGINE}[a.mode] if mode is None else mode
        flags = ((kvb.KV_CFG_NO_BULK if a.no_bulk else 0) | (kvb.KV_CFG_NO_PDL if a.no_pdl else 0)
                 | (kvb.KV_CFG_OVERLAP_RESTORES if (a.overlap if overlap is None else overlap)
                    else 0))
        kvb.kv_config_set(m, a.max_ctas if max_ctas is None else max_ctas, a.staging_mib << 20,
                          flags, a.cta_threads if cta_threads is None else cta_threads)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def timed(self, fn, stream, reps=5, warm=2):
        """Median CUDA-event time (ms) of fn(i) on `stream` after `warm` calls."""
        out = []
        for i in range(reps + warm):
            self.torch.cuda.synchronize()
            e0, e1 = self.event(), self.event()
            e0.record(stream)
            fn(i)
            e1.record(stream)
            e1.synchronize()
            if i >= warm:
                out.append(e0.elapsed_time(e1))
        return statistics.median(out)


def measure_link(ctx, probe_alloc=None):
    """Host-link peaks measured in this run: pinned cudaMemcpyAsync of 2 GiB D2H,
    H2D and both at once (two streams, 1 GiB each way), best of 10."""
    torch = ctx.torch
    probe_n = 2 << 30
    pin = torch.empty(probe_n, dtype=torch.uint8, pin_memory=True)
    dbuf = (probe_alloc[:probe_n] if probe_alloc is not None and probe_alloc.numel() >= probe_n
            else torch.empty(probe_n, dtype=torch.uint8, device=ctx.dev))
    pin2 = torch.empty(probe_n // 2, dtype=torch.uint8, pin_memory=True)
    dbuf2 = torch.empty(probe_n // 2, dtype=torch.uint8, device=ctx.dev)
    s_a, s_b = ctx.s_a, ctx.s_b

    def best_of(fn, nbytes, reps=10):
        ts = []
        for i in range(reps + 3):
            torch.cuda.synchronize()
            e0, e1 = ctx.event(), ctx.event()
            e0.record(s_a)
            fn()
            e1.record(s_a)
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) / 1000)
        return nbytes / min(ts) / GB

    link = {}
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
    # kept for bidir_nearby(): 1 GiB each way
    ctx.probe_bufs = (pin[:probe_n // 2], dbuf[:probe_n // 2], pin2, dbuf2)
    return link


def bidir_nearby(ctx):
    """The bidirectional pinned-memcpy rate (1 GiB each way, best of 3) measured
    right beside a concurrent measurement: the host link's capacity at that
    moment.  Other tenants of the same host can take some of it, and concurrent
    figures taken seconds apart then differ for that reason alone."""
    torch = ctx.torch
    pin, dbuf, pin2, dbuf2 = ctx.probe_bufs
    s_a, s_b = ctx.s_a, ctx.s_b
    ts = []
    for i in range(4):
        torch.cuda.synchronize()
        e0, e1 = ctx.event(), ctx.event()
        e0.record(s_a)
        ev = torch.cuda.Event()
        ev.record(s_a)
        s_b.wait_event(ev)
        with torch.cuda.stream(s_a):
            pin.copy_(dbuf, non_blocking=True)
        with torch.cuda.stream(s_b):
            dbuf2.copy_(pin2, non_blocking=True)
        ev2 = torch.cuda.Event()
        ev2.record(s_b)
        s_a.wait_event(ev2)
        e1.record(s_a)
        e1.synchronize()
        if i >= 1:
            ts.append(e0.elapsed_time(e1) / 1000)
    return round((pin.numel() + pin2.numel()) / min(ts) / GB, 2)


class Setup:
    """A workload's pool (registered, or imported from a second process for
    TRT-LLM), its pinned host tier filled with random bytes, and R id sets."""

    def __init__(self, ctx, w, R=8):
        torch, kvb = ctx.torch, ctx.kvb
        self.ctx, self.w = ctx, w
        g = self.g = w.geom
        self.lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads,
                                   g.elem_bytes)
        self.exporter = self.done_ev = None
        self.host = torch.empty(w.host_slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
        rank = ctx.rank
        if w is wl.TRTLLM:
            import multiprocessing as mp

            mpc = mp.get_context("spawn")
            q, self.done_ev = mpc.Queue(), mpc.Event()
            self.exporter = mpc.Process(target=_exporter, args=(q, self.done_ev, ctx.local,
                                                                w.seed + 100 * rank,
                                                                w.pool_offset))
            self.exporter.daemon = True   # never outlives the benchmark, whatever happens
            self.exporter.start()
            self.pool = kvb.kv_pool_import(kvb.desc_from_bytes(q.get(timeout=900)))
            self.alloc = None
            fill = torch.empty(2 << 30, dtype=torch.uint8, device=ctx.dev)
            wl.fill_random_(fill, w.seed + 7)
            for lo in range(0, self.host.numel(), fill.numel()):
                hi = min(self.host.numel(), lo + fill.numel())
                self.host[lo:hi].copy_(fill[:hi - lo])
            del fill
        else:
            self.alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8,
                                     device=ctx.dev)
            wl.fill_random_(self.alloc, w.seed + 100 * rank)
            for lo in range(0, self.host.numel(), 2 << 30):
                hi = min(self.host.numel(), lo + (2 << 30))
                self.host[lo:hi].copy_(self.alloc[lo:hi])
            self.pool = kvb.kv_pool_register(self.lay, self.alloc.data_ptr(), w.pool_offset)
        self.tier = kvb.kv_host_register(self.host.data_ptr(), self.host.numel(), w.host_slots,
                                         g.host_heads, self.lay)
        self.R = R
        self.idsets = [wl.op_ids(w, seed=w.seed + 17 * k + 1000 * rank) for k in range(R)]
        torch.cuda.synchronize()

    def ids(self, k):
        return self.idsets[k % self.R]

    def close(self):
        kvb = self.ctx.kvb
        kvb.kv_pool_close(self.pool)
        kvb.kv_host_close(self.tier)
        if self.exporter is not None:
            self.done_ev.set()
            self.exporter.join(120)
            if self.exporter.is_alive():
                self.exporter.terminate()
                self.exporter.join(10)
        self.alloc = self.host = None
        self.ctx.torch.cuda.empty_cache()


def step_fn(ctx, su):
    """One step of the workload through the C ABI (ids are host arrays).
    Returns (step(k, evs) -> fences, backup bytes, restore bytes).  evs (five
    events) bracket: [0] backup start, [1] backup end / restore start, [2] step
    end on stream A, [3]/[4] the restore on stream B (TRT-LLM)."""
    kvb, torch = ctx.kvb, ctx.torch
    w, g = su.w, su.g
    s_a, s_b = ctx.s_a, ctx.s_b
    if w is wl.MLA_FP8:
        def step(k, evs=None):
            ids = su.ids(k)
            if evs:
                evs[0].record(s_a)
            f = None
            for layer in range(g.L):
                f = kvb.kv_restore(su.pool, su.tier, ids.restore_slots, ids.restore_dst, layer,
                                   s_a.cuda_stream)
            if evs:
                evs[1].record(s_a)
                evs[2].record(s_a)
            return [f]
        return step, 0, g.L * w.n * g.layer_page_bytes
    if w is wl.TRTLLM:
        def step(k, evs=None):
            ids = su.ids(k)
            ev = torch.cuda.Event()
            ev.record(s_a)
            s_b.wait_event(ev)
            if evs:
                evs[0].record(s_a)
            fb = kvb.kv_backup(su.pool, su.tier, ids.backup_src, ids.backup_slots, s_a.cuda_stream)
            if evs:
                evs[1].record(s_a)
                evs[3].record(s_b)
            fr = kvb.kv_restore(su.pool, su.tier, ids.restore_slots, ids.restore_dst, -1,
                                s_b.cuda_stream)
            if evs:
                evs[4].record(s_b)
            ev2 = torch.cuda.Event()
            ev2.record(s_b)
            s_a.wait_event(ev2)
            if evs:
                evs[2].record(s_a)
            return [fb, fr]
        return step, w.n * g.page_bytes, w.n * g.page_bytes

    def step(k, evs=None):
        ids = su.ids(k)
        if evs:
            evs[0].record(s_a)
        kvb.kv_backup(su.pool, su.tier, ids.backup_src, ids.backup_slots, s_a.cuda_stream)
        if evs:
            evs[1].record(s_a)
        f = kvb.kv_restore(su.pool, su.tier, ids.restore_slots, ids.restore_dst, -1,
                           s_a.cuda_stream)
        if evs:
            evs[2].record(s_a)
        return [f]   # same stream: the restore's fence follows the backup
    return step, w.n * g.page_bytes, w.n * g.page_bytes


def timed_steps(ctx, step, steps, warmup):
    """warmup untimed steps, then `steps` timed on the device clock (CUDA events
    on the launching stream, a barrier and a synchronize on both sides).
    Returns (max-over-ranks seconds, per-step events, launches, Window)."""
    kvb = ctx.kvb
    for k in range(warmup):
        step(k)
    ctx.barrier()
    evs = [[ctx.event() for _ in range(5)] for _ in range(steps)]
    l0 = kvb.kv_launch_count()
    ctx.barrier()
    with Window() as win:
        t_start, t_end = ctx.event(), ctx.event()
        t_start.record(ctx.s_a)
        for k in range(steps):
            step(k, evs[k])
        t_end.record(ctx.s_a)
        ctx.barrier()
    launches = kvb.kv_launch_count() - l0
    elapsed = dist_max(t_start.elapsed_time(t_end) / 1000, ctx.dist, ctx.dev)
    return elapsed, evs, launches, win


def e2e_gbs(ctx, step, steps, step_bytes):
    """The same step end to end through the C ABI on the host clock, a fence
    wait every step (payload crosses the host link inside the region)."""
    ctx.barrier()
    t0 = time.perf_counter()
    for k in range(steps):
        for f in step(k):
            ctx.kvb.kv_fence_wait(f, WAIT_NS)
    return job_gbs(step_bytes, steps, ctx.ws, dist_max(time.perf_counter() - t0, ctx.dist,
                                                        ctx.dev))


def hbm_gather(ctx, su):
    """Device-side layout-transform gather of the step's pages (pool -> device
    buffer in host layout) against the HBM peak: 10 launches back to back."""
    torch, kvb, g, w = ctx.torch, ctx.kvb, su.g, su.w
    n = w.n
    buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device=ctx.dev)
    gathers = 10      # back to back, so each launch is issued while the GPU is busy

    def gather_gbs(with_fence):
        ts = []
        for i in range(4):
            e0, e1 = ctx.event(), ctx.event()
            e0.record(ctx.s_a)
            for k in range(gathers):
                kvb.kv_device_gather(su.pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                     su.ids(i + k).backup_src, ctx.s_a.cuda_stream,
                                     fence=with_fence)
            e1.record(ctx.s_a)
            e1.synchronize()
            if i >= 1:
                ts.append(e0.elapsed_time(e1) / 1000 / gathers)
        return 2 * n * g.page_bytes / statistics.median(ts) / GB

    with Window() as win:
        gb_s = gather_gbs(True)          # the roofline: with its fence, as a backup has
        gb_s_ordered = gather_gbs(False)  # stream order only (fence = NULL)
    transposed = g.dev_heads != g.host_heads
    kern = ("kv_move_kernel" if ctx.args.no_bulk else
            "kv_tsp_kernel" if transposed else "kv_bulk_kernel")
    peak = ctx.peaks["hbm_gbs"]
    del buf
    return {"bound": "hbm", "kernel": kern + " (device gather, pool -> device buffer in host "
                                             "layout)",
            "achieved": round(gb_s, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gb_s / peak, 4),
            "traffic": recorded_traffic("device_gather_transposed_dram_bytes_per_launch"
                                        if transposed else "device_gather_dram_bytes_per_launch"),
            "algorithmic_bytes_per_launch": 2 * n * g.page_bytes,
            "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({ctx.peak_src}); of measured",
            "achieved_without_fence": round(gb_s_ordered, 1),
            "frac_without_fence": round(gb_s_ordered / peak, 4),
            "clocks": win}


def op_stats(ms, pages):
    return {"median_ms": round(statistics.median(ms), 4), "best_ms": round(min(ms), 4),
            "pages_per_s": round(pages / (statistics.mean(ms) / 1000), 1)}


def link_roofline(kernel, nbytes, seconds, peak, direction, traffic=None):
    a = nbytes / seconds / GB
    return {"bound": "host_link", "kernel": kernel, "achieved": round(a, 2),
            "peak": round(peak, 2), "unit": "GB/s", "frac": round(a / peak, 4),
            "traffic": traffic, "algorithmic_bytes_per_launch": nbytes,
            "peak_source": f"pinned cudaMemcpyAsync {direction} of 2 GiB measured in this run, "
                           "best of 10 (host link peak; not in MEASURED_PEAKS.json)"}


# --------------------------------------------------------------- the headline

def headline(ctx):
    """The headline workload's line (value, e2e, roofline, per-op figures)."""
    args, kvb = ctx.args, ctx.kvb
    w = {"llama8b": wl.LLAMA8B, "mla_fp8": wl.MLA_FP8, "trtllm_ipc": wl.TRTLLM}[args.workload]
    ctx.set_config()
    su = Setup(ctx, w)
    g = su.g
    step, bytes_b, bytes_r = step_fn(ctx, su)
    elapsed, evs, launches, win = timed_steps(ctx, step, args.steps, args.warmup)
    b_ms = [e[0].elapsed_time(e[1]) for e in evs]
    r_ms = ([e[3].elapsed_time(e[4]) for e in evs] if w is wl.TRTLLM else
            [e[1].elapsed_time(e[2]) for e in evs])
    step_bytes = bytes_b + bytes_r
    value = job_gbs(step_bytes, args.steps, ctx.ws, elapsed)
    e2e = e2e_gbs(ctx, step, args.steps, step_bytes)
    link = ctx.link
    mode = kvb.kv_config_get().mode
    if w is wl.MLA_FP8:
        dom_ms = statistics.mean(b_ms) / g.L
        roofline = link_roofline("kv_move_kernel (restore of one layer, zero-copy H2D)",
                                 w.n * g.layer_page_bytes, dom_ms / 1000, link["h2d"], "h2d")
    elif w is wl.TRTLLM:
        step_s = elapsed / args.steps
        a = step_bytes / step_s / GB
        roofline = {"bound": "host_link_bidirectional",
                    "kernel": "kv_move_kernel x 2 (backup D2H || restore H2D)",
                    "achieved": round(a, 2), "peak": round(link["bidir"], 2), "unit": "GB/s",
                    "frac": round(a / link["bidir"], 4), "traffic": None,
                    "algorithmic_bytes_per_launch": step_bytes,
                    "peak_source": "pinned cudaMemcpyAsync D2H || H2D (two streams, 1 GiB each "
                                   "way) measured in this run, best of 10"}
    else:
        kern = {0: "kv_move_kernel (backup, zero-copy D2H)",
                1: "kv_move_kernel + cudaMemcpyAsync (backup, staged D2H)",
                2: "cudaMemcpy2DAsync per page (backup, copy engine D2H)"}[mode]
        roofline = link_roofline(kern, bytes_b, statistics.mean(b_ms) / 1000, link["d2h"], "d2h",
                                 recorded_traffic("backup_dram_bytes_per_launch")
                                 if w is wl.LLAMA8B and mode == 0 else None)
    op_b, op_r = (None, b_ms) if w is wl.MLA_FP8 else (b_ms, r_ms)
    backup_gbs = bytes_b / (statistics.mean(op_b) / 1000) / GB if op_b else None
    restore_gbs = bytes_r / (statistics.mean(op_r) / 1000) / GB
    per_op = {"restore": op_stats(op_r, w.n)}
    if op_b:
        per_op["backup"] = op_stats(op_b, w.n)
    if w is wl.MLA_FP8:
        per_op["restore"]["per_layer_call_us"] = round(1000 * statistics.mean(op_r) / g.L, 2)
    pct = {"d2h": round(100 * backup_gbs / link["d2h"], 2) if backup_gbs else None,
           "h2d": round(100 * restore_gbs / link["h2d"], 2)}
    if w is wl.TRTLLM:
        pct["step_vs_bidir_peak"] = round(100 * value / ctx.ws / link["bidir"], 2)
        pct["note"] = "d2h / h2d: each direction while the other runs, against its solo peak"
    else:
        seq_peak = step_bytes / ((bytes_b / link["d2h"] if bytes_b else 0) +
                                 bytes_r / link["h2d"])
        pct["step_vs_sequential_peak"] = round(100 * value / ctx.ws / seq_peak, 2)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ctx.ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * elapsed / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random bytes; bf16/fp8 KV are opaque bytes)",
        "config": config_of(w),
        "mode": args.mode + (" + overlap_restores" if args.overlap else ""),
        "backup_gbs": round(backup_gbs, 2) if backup_gbs else None,
        "restore_gbs": round(restore_gbs, 2),
        "pages_per_s": round(ctx.ws * (w.n * (2 if bytes_b else 1)) * args.steps / elapsed, 1),
        "per_op": per_op,
        "host_link_peak_gbs": {k: round(v, 2) for k, v in link.items()},
        "pct_of_host_link_peak": pct,
        "roofline": roofline,
        "e2e": {"value": round(e2e, 2), "unit": "GB/s",
                "h2d_bytes_per_step": bytes_r + 8 * w.n * (2 if bytes_b else g.L),
                "d2h_bytes_per_step": bytes_b + 8,
                "note": "host clock around kv_backup/kv_restore with host id arrays and a fence "
                        "wait every step; payload crosses the host link inside the region"},
        "gpu_launches": launches,
        "clocks": win,
    }
    if w is not wl.MLA_FP8:
        line["roofline_hbm"] = hbm_gather(ctx, su)
    return line, su


# -------------------------------------------------- MLA: layer-wise restores

def mla_layerwise(ctx, su, detail=False):
    """The MLA prefix (61 layers x 64 pages) restored one layer per call (plain,
    and with overlapped calls), and by one progressive call; each pipelined with
    a stand-in forward (one bf16 GEMM per layer on a compute stream that waits
    on the GPU for that layer's fence).  detail adds the SM-budget table and
    the ring-descriptor figures."""
    torch, kvb, args = ctx.torch, ctx.kvb, ctx.args
    w, g = su.w, su.g
    s_a = ctx.s_a
    link = ctx.link
    steps, warmup = max(5, min(args.steps, 20)), max(3, args.warmup)
    nbytes = g.L * w.n * g.layer_page_bytes
    call_bytes = w.n * g.layer_page_bytes

    def layer_calls(i, stream=s_a):
        ids = su.ids(i)
        return [kvb.kv_restore(su.pool, su.tier, ids.restore_slots, ids.restore_dst, layer,
                               stream.cuda_stream) for layer in range(g.L)]

    def progressive(i, stream=s_a):
        ids = su.ids(i)
        return kvb.kv_restore_layers(su.pool, su.tier, ids.restore_slots, ids.restore_dst, 0,
                                     g.L, stream.cuda_stream)

    def run_timed(fn):
        for i in range(warmup):
            fn(i)
        ctx.barrier()
        evs = []
        l0 = kvb.kv_launch_count()
        for i in range(steps):
            e0, e1 = ctx.event(), ctx.event()
            e0.record(s_a)
            fn(warmup + i)
            e1.record(s_a)
            evs.append((e0, e1))
        ctx.barrier()
        return statistics.mean(a.elapsed_time(b) for a, b in evs) / 1000, \
            kvb.kv_launch_count() - l0

    rec = {"workload": config_of(w)["workload"] + "; prefix of 16,384 tokens = 64 pages",
           "step": STEP_TEXT["mla_fp8"], "steps": steps, "warmup": warmup,
           "bytes_per_step": nbytes, "bytes_per_call": call_bytes}
    with Window() as win:
        ctx.set_config(overlap=False)
        t_plain, launches = run_timed(layer_calls)
        ctx.set_config(overlap=True)
        c0 = kvb.kv_overlap_count()
        t_ov, launches_ov = run_timed(layer_calls)
        overlapped = kvb.kv_overlap_count() - c0
        ctx.set_config(overlap=False)
        t_prog, launches_p = run_timed(progressive)
    # end to end through the C ABI on the host clock: the overlapped calls with a
    # wait on the last layer's fence every step (host ids, payload over the link)
    ctx.set_config(overlap=True)
    ctx.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        kvb.kv_fence_wait(layer_calls(i)[-1], WAIT_NS)
    e2e_s = time.perf_counter() - t0
    ctx.set_config(overlap=False)
    rec["clocks"] = win
    # the record's figure: one restore per layer the way the library runs that
    # pattern best (overlapped calls); the default configuration beside it
    rec["config"] = ("kv_config.flags = KV_CFG_OVERLAP_RESTORES (zero-copy, library default "
                     "grid under the flag: 6 CTAs of 1,024 threads): each one-layer restore "
                     "starts while the previous one (another layer: disjoint bytes) finishes; "
                     "fences still complete in call order")
    rec["value"] = round(nbytes / t_ov / GB, 2)
    rec["unit"] = "GB/s"
    rec["per_layer_call_us"] = round(1e6 * t_ov / g.L, 2)
    rec["overlapped_restores"] = overlapped
    rec["gpu_launches"] = launches_ov
    rec["e2e"] = {"value": round(nbytes * steps / e2e_s / GB, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": nbytes + 8 * w.n * g.L, "d2h_bytes_per_step": 8,
                  "note": "host clock around the 61 kv_restore calls (overlapped) with a wait "
                          "on the last layer's fence every step"}
    rec["roofline"] = link_roofline("kv_move_kernel (restore of one layer, zero-copy H2D, one "
                                    "launch per call, overlapped calls)", call_bytes,
                                    t_ov / g.L, link["h2d"], "h2d")
    rec["plain_calls"] = {
        "config": "library defaults (no overlap flag): each call waits for the previous "
                  "kernel on the stream to finish",
        "gbs": round(nbytes / t_plain / GB, 2), "per_layer_call_us": round(1e6 * t_plain / g.L, 2),
        "gpu_launches": launches,
        "roofline": link_roofline("kv_move_kernel (restore of one layer, one launch per call)",
                                  call_bytes, t_plain / g.L, link["h2d"], "h2d")}
    rec["progressive_call"] = {
        "call": "kv_restore_layers: 61 layers x 64 pages in one call, per-layer fences "
                "published as the restored prefix grows",
        "gbs": round(nbytes / t_prog / GB, 2), "ms_per_step": round(1000 * t_prog, 4),
        "gpu_launches": launches_p,
        "roofline": link_roofline("kv_move_kernel (61 layers in one progressive launch)",
                                  nbytes, t_prog, link["h2d"], "h2d")}

    # overlap with a stand-in forward: one bf16 GEMM (3456^3) per layer on a compute
    # stream that waits, on the GPU, for that layer's fence; exposed = pipelined - compute
    comp = torch.cuda.Stream(device=ctx.dev)
    M = 3456
    A = torch.randn(M, M, dtype=torch.bfloat16, device=ctx.dev)
    Bm = torch.randn(M, M, dtype=torch.bfloat16, device=ctx.dev)
    Cm = torch.empty(M, M, dtype=torch.bfloat16, device=ctx.dev)

    def compute_only(i):
        with torch.cuda.stream(comp):
            for _ in range(g.L):
                torch.matmul(A, Bm, out=Cm)

    def pipelined(i, prog):
        ev = torch.cuda.Event()
        ev.record(comp)
        s_a.wait_event(ev)
        fences = progressive(i) if prog else layer_calls(i)
        with torch.cuda.stream(comp):
            for layer in range(g.L):
                kvb.kv_fence_stream_wait(fences[layer], comp.cuda_stream)
                torch.matmul(A, Bm, out=Cm)
        ev2 = torch.cuda.Event()
        ev2.record(comp)
        s_a.wait_event(ev2)

    with Window() as win2:
        t_c = ctx.timed(compute_only, comp)
        ctx.set_config(overlap=False)
        t_r = ctx.timed(layer_calls, s_a)
        t_p1 = ctx.timed(lambda i: pipelined(i, False), s_a)
        t_p2 = ctx.timed(lambda i: pipelined(i, True), s_a)
        ctx.set_config(overlap=True)
        t_r3 = ctx.timed(layer_calls, s_a)
        t_p3 = ctx.timed(lambda i: pipelined(i, False), s_a)
        ctx.set_config(overlap=False)
    rec["overlap_with_compute"] = {
        "forward_stand_in": f"bf16 GEMM {M}^3 per layer on a compute stream, 61 layers",
        "compute_only_ms": round(t_c, 3),
        "restore_only_ms": {"per_layer_calls": round(t_r, 3),
                            "overlapped_calls": round(t_r3, 3)},
        "pipelined_ms": {"per_layer_calls": round(t_p1, 3), "progressive": round(t_p2, 3),
                         "overlapped_calls": round(t_p3, 3)},
        "exposed_transfer_ms": {"per_layer_calls": round(t_p1 - t_c, 3),
                                "progressive": round(t_p2 - t_c, 3),
                                "overlapped_calls": round(t_p3 - t_c, 3)},
        "clocks": win2}
    if detail:
        rec["overlap_with_compute"]["sm_budget"] = mla_sm_budget(ctx, su, layer_calls,
                                                                 progressive, pipelined)
        rec["ring_one_layer_descriptors"] = mla_ring_layers(ctx, su)
    del A, Bm, Cm
    ctx.set_config()
    return rec


def mla_sm_budget(ctx, su, layer_calls, progressive, pipelined):
    """The SM budget that saturates the host link: the progressive restore (H2D)
    and a backup of the same 64 pages (D2H) on k whole SMs (k CTAs of 1024
    threads), alone and pipelined with the stand-in forward."""
    kvb, g, link, s_a = ctx.kvb, su.g, ctx.link, ctx.s_a
    nbytes = g.L * su.w.n * g.layer_page_bytes

    def backup_pages(i):
        ids = su.ids(i)
        kvb.kv_backup(su.pool, su.tier, ids.restore_dst, ids.restore_slots, s_a.cuda_stream)

    rows = []
    try:
        for k in (1, 2, 3, 4, 6, 8, 12, 16):
            ctx.set_config(overlap=False, max_ctas=k, cta_threads=1024)
            t_rk = ctx.timed(progressive, s_a)
            t_bk = ctx.timed(backup_pages, s_a)
            t_pk = ctx.timed(lambda i: pipelined(i, True), s_a)
            t_lk = ctx.timed(layer_calls, s_a)
            t_qk = ctx.timed(lambda i: pipelined(i, False), s_a)
            rows.append({"sms": k,
                         "restore_gbs": round(nbytes / t_rk * 1000 / GB, 2),
                         "restore_pct_h2d": round(100 * nbytes / t_rk * 1000 / GB / link["h2d"],
                                                  1),
                         "backup_gbs": round(nbytes / t_bk * 1000 / GB, 2),
                         "backup_pct_d2h": round(100 * nbytes / t_bk * 1000 / GB / link["d2h"],
                                                 1),
                         "pipelined_progressive_ms": round(t_pk, 3),
                         "per_layer_calls_gbs": round(nbytes / t_lk * 1000 / GB, 2),
                         "pipelined_per_layer_calls_ms": round(t_qk, 3)})
    finally:
        ctx.set_config()
    return {"what": "k CTAs of 1024 threads (k whole SMs): kv_restore_layers of 61 layers x 64 "
                    "pages (H2D), kv_backup of the same 64 pages (D2H) and the 61 one-layer "
                    "kv_restore calls, each alone (median of 5), and both restores pipelined "
                    "with the per-layer GEMMs", "rows": rows}


def mla_ring_layers(ctx, su):
    """The 61 one-layer restores as ring descriptors (one per layer, 64 pages
    each), all submitted at once, served by a host thread and by the
    GPU-resident server; host clock from the first submit to the last ticket,
    median of 5 steps after one."""
    torch, kvb, g, w = ctx.torch, ctx.kvb, su.g, su.w
    nbytes = g.L * w.n * g.layer_page_bytes
    out = {}
    steps_l = 6
    for kind in ("host", "device"):
        name = f"/kvbbenchly_{os.getpid()}_{kind}"
        sub = kvb.kv_ring_create(name, 64)
        srv = kvb.kv_ring_attach(name)
        rs = torch.cuda.Stream(device=ctx.dev)
        stop = threading.Event()
        served = [0]

        def serve_layers():
            while not stop.is_set() and served[0] < g.L * steps_l:
                served[0] += kvb.kv_ring_serve(srv, [su.pool], su.tier, rs.cuda_stream, 64,
                                               200_000_000)

        th, fence = None, None
        if kind == "host":
            th = threading.Thread(target=serve_layers, daemon=True)
            th.start()
        else:
            fence = kvb.kv_ring_serve_device(srv, [su.pool], su.tier, rs.cuda_stream,
                                             g.L * steps_l, 5_000_000_000)
        times = []
        for i in range(steps_l):
            ids = su.ids(i)
            ops = [kvb.make_ring_op(1, ids.restore_slots, ids.restore_dst, layer=layer)
                   for layer in range(g.L)]
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
        out[f"{kind}_served_gbs"] = round(nbytes / t_med / GB, 2)
        out[f"{kind}_served_us_per_layer"] = round(1e6 * t_med / g.L, 2)
    out["workload"] = ("61 one-layer restore descriptors of 64 pages (9,437,184 B each) "
                       "submitted at once, host clock from the first submit to the last ticket, "
                       "median of 5 steps after one")
    return out


def mla_record(ctx):
    """The MLA fp8 workload as a record of its own (17.2 GiB pool), with the 61
    one-layer restores also sent as ring descriptors (overlapped restores on)."""
    su = Setup(ctx, wl.MLA_FP8)
    try:
        rec = mla_layerwise(ctx, su)
        ctx.set_config(overlap=True)
        ring = mla_ring_layers(ctx, su)
        ring["config"] = "kv_config.flags = KV_CFG_OVERLAP_RESTORES"
        rec["ring_one_layer_descriptors"] = ring
        ctx.set_config()
    finally:
        su.close()
    g, w = wl.MLA_FP8.geom, wl.MLA_FP8
    rec["cpu_baseline"] = cpu_record(g, w.n, 128, 3.0, layerwise=True, seed=w.seed)
    return rec


# --------------------------------------------------- TRT-LLM over CUDA IPC

def trtllm_record(ctx):
    """Backup of 512 pages on stream A while 512 others are restored on stream B,
    on the TRT-LLM pool ([2048, 40, 2, 8*32*128] bf16, page-first HND, at byte
    offset 2 MiB + 48 in its allocation) imported over CUDA IPC from a second
    process; host tier NHD.  The bound is the host link both ways at once."""
    args, link = ctx.args, ctx.link
    w = wl.TRTLLM
    ctx.set_config(overlap=False)
    su = Setup(ctx, w)
    g = su.g
    steps, warmup = max(5, min(args.steps, 20)), max(3, args.warmup)
    try:
        step, bytes_b, bytes_r = step_fn(ctx, su)
        near0 = bidir_nearby(ctx)
        elapsed, evs, launches, win = timed_steps(ctx, step, steps, warmup)
        near1 = bidir_nearby(ctx)
        b_ms = [e[0].elapsed_time(e[1]) for e in evs]
        r_ms = [e[3].elapsed_time(e[4]) for e in evs]
        step_bytes = bytes_b + bytes_r
        value = step_bytes * steps / elapsed / GB
        e2e = e2e_gbs(ctx, step, steps, step_bytes)
        hbm = hbm_gather(ctx, su)
    finally:
        su.close()
    d2h = bytes_b / (statistics.mean(b_ms) / 1000) / GB
    h2d = bytes_r / (statistics.mean(r_ms) / 1000) / GB
    rec = {"workload": config_of(w)["workload"] + f", pool at byte offset {w.pool_offset} of "
                                                  "an allocation owned by a second process",
           "step": STEP_TEXT["trtllm_ipc"], "steps": steps, "warmup": warmup,
           "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(1000 * elapsed / steps,
                                                                           4),
           "bytes_per_step": step_bytes, "gpu_launches": launches,
           "roofline": {"bound": "host_link_bidirectional",
                        "kernel": "kv_move_kernel x 2 at once (backup D2H || restore H2D, HND pool "
                                  "<-> NHD tier)",
                        "achieved": round(value, 2), "peak": round(link["bidir"], 2),
                        "unit": "GB/s", "frac": round(value / link["bidir"], 4), "traffic": None,
                        "algorithmic_bytes_per_launch": step_bytes,
                        "peak_source": "pinned cudaMemcpyAsync D2H || H2D (two streams, 1 GiB "
                                       "each way) measured in this run, best of 10",
                        "bidir_memcpy_nearby_gbs": [near0, near1],
                        "frac_of_nearby": round(value / max(near0, near1), 4)},
           "per_direction": {
               "note": "each direction while the other runs; secondary to the bidirectional "
                       "roofline",
               "d2h": {"gbs": round(d2h, 2), "pct_of_solo_d2h": round(100 * d2h / link["d2h"], 2),
                       **op_stats(b_ms, w.n)},
               "h2d": {"gbs": round(h2d, 2), "pct_of_solo_h2d": round(100 * h2d / link["h2d"], 2),
                       **op_stats(r_ms, w.n)}},
           "e2e": {"value": round(e2e, 2), "unit": "GB/s"},
           "roofline_hbm": hbm,
           "clocks": win}
    rec["cpu_baseline"] = cpu_record(g, 64, 256, 3.0, seed=w.seed)
    return rec


# ------------------------------------------------------------ sweep summary

SUMMARY_SIZES = [4096, 65536, 1 << 20]
SUMMARY_BATCHES = [1, 32, 1024]


def sweep_points(ctx, sizes, batches, modes, reps, warmup, pages):
    """Times backup (D2H), restore (H2D) and both at once (two streams, disjoint
    pages and slots) for every page size x batch x id pattern x mode, with CUDA
    events on the launching stream (median of `reps` after `warmup`; every rep
    uses another page set so small batches do not run from L2)."""
    torch, kvb = ctx.torch, ctx.kvb
    P = pages
    max_pb, max_n = max(sizes), max(batches)
    alloc = torch.empty(P * max_pb, dtype=torch.uint8, device=ctx.dev)
    wl.fill_random_(alloc, 4004)
    host = torch.empty(2 * max_n * max_pb, dtype=torch.uint8, pin_memory=True)
    host.copy_(alloc[:host.numel()])
    sa, sb = ctx.s_a, ctx.s_b
    r = wl.rng(1004)
    records = []
    for pb in sizes:
        lay = kvb.make_layout(1, 1, P, 1, 1, pb, 0, 0, 1)
        pool = kvb.kv_pool_register(lay, alloc.data_ptr(), 0)
        slots_total = 2 * max_n
        tier = kvb.kv_host_register(host.data_ptr(), slots_total * pb, slots_total, 0, lay)
        for n in batches:
            for pattern in ("seq", "random"):
                sets = []
                for k in range(warmup + reps):
                    if pattern == "seq":
                        base = (k * 2 * n) % max(1, P - 2 * n + 1)
                        src = np.arange(base, base + n, dtype=np.int32)
                        dst = np.arange(base + n, base + 2 * n, dtype=np.int32) % P
                    else:
                        src = wl.distinct_pages(r, P, n)
                        dst = wl.distinct_pages(r, P, n, exclude=src)
                    sets.append((src, dst))
                slots_b = np.arange(n, dtype=np.int32)
                slots_r = np.arange(n, 2 * n, dtype=np.int32)
                for mode_name, mode in modes:
                    kvb.kv_config_set(mode, 0, 0)
                    for direction in ("d2h", "h2d", "both"):
                        ts = []
                        for k, (src, dst) in enumerate(sets):
                            e0, e1 = ctx.event(), ctx.event()
                            torch.cuda.synchronize()
                            e0.record(sa)
                            if direction == "both":
                                ev = torch.cuda.Event()
                                ev.record(sa)
                                sb.wait_event(ev)
                            if direction in ("d2h", "both"):
                                kvb.kv_backup(pool, tier, src, slots_b, sa.cuda_stream)
                            if direction in ("h2d", "both"):
                                s = sb if direction == "both" else sa
                                kvb.kv_restore(pool, tier, slots_r, dst, -1, s.cuda_stream)
                            if direction == "both":
                                ev2 = torch.cuda.Event()
                                ev2.record(sb)
                                sa.wait_event(ev2)
                            e1.record(sa)
                            e1.synchronize()
                            if k >= warmup:
                                ts.append(e0.elapsed_time(e1) / 1000)
                        t = statistics.median(ts)
                        nbytes = n * pb * (2 if direction == "both" else 1)
                        records.append({"page_bytes": pb, "batch": n, "ids": pattern,
                                        "mode": mode_name, "direction": direction,
                                        "seconds": t, "gbs": nbytes / t / GB,
                                        "pages_per_s": nbytes / pb / t})
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
    del alloc, host
    torch.cuda.empty_cache()
    return records


def sweep_record(ctx):
    """A summary of the bandwidth sweep: page bytes {4 KiB, 64 KiB, 1 MiB} x
    batch {1, 32, 1024} x {sequential, random} ids x {D2H, H2D, both}, in
    zero-copy, STAGED and copy-engine mode."""
    kvb, link = ctx.kvb, ctx.link
    modes = (("zero_copy", kvb.KV_MODE_ZERO_COPY), ("staged", kvb.KV_MODE_STAGED),
             ("copy_engine", kvb.KV_MODE_COPY_ENGINE))
    near0 = bidir_nearby(ctx)
    with Window() as win:
        recs = sweep_points(ctx, SUMMARY_SIZES, SUMMARY_BATCHES, modes, reps=5, warmup=2,
                            pages=4096)
    near1 = bidir_nearby(ctx)
    ctx.set_config()
    peak = {"d2h": link["d2h"], "h2d": link["h2d"], "both": link["bidir"]}
    points = {"fields": ["page_bytes", "batch", "ids", "mode", "direction", "gbs",
                         "pct_of_peak", "us"],
              "rows": [[x["page_bytes"], x["batch"], x["ids"], x["mode"], x["direction"],
                        round(x["gbs"], 2), round(100 * x["gbs"] / peak[x["direction"]], 1),
                        round(1e6 * x["seconds"], 1)] for x in recs]}
    big = {d: next(x for x in recs if x["page_bytes"] == max(SUMMARY_SIZES) and
                   x["batch"] == max(SUMMARY_BATCHES) and x["ids"] == "random" and
                   x["mode"] == "zero_copy" and x["direction"] == d)
           for d in ("d2h", "h2d", "both")}
    a = big["both"]["gbs"]
    wins = {}
    for d in ("d2h", "h2d", "both"):
        for ids in ("seq", "random"):
            count = {m: 0 for m, _ in modes}
            for pb in SUMMARY_SIZES:
                for n in SUMMARY_BATCHES:
                    pt = {x["mode"]: x["gbs"] for x in recs if x["page_bytes"] == pb and
                          x["batch"] == n and x["ids"] == ids and x["direction"] == d}
                    count[max(pt, key=pt.get)] += 1
            wins[f"{d}_{ids}"] = count
    return {"workload": "one opaque run per page (L = C = T = H = 1, B = page bytes), 4,096-page "
                        "pool, random uint8 payload; ops of `batch` pages into slots 0..batch-1 "
                        "(backup) and from slots batch..2*batch-1 (restore)",
            "grid": {"page_bytes": SUMMARY_SIZES, "batch": SUMMARY_BATCHES,
                     "ids": ["seq", "random"], "direction": ["d2h", "h2d", "both"],
                     "mode": [m for m, _ in modes]},
            "value": round(a, 2), "unit": "GB/s",
            "roofline": {"bound": "host_link_bidirectional",
                         "kernel": "kv_move_kernel x 2 at once (1,024 random pages of 1 MiB each "
                                   "way)",
                         "achieved": round(a, 2), "peak": round(link["bidir"], 2),
                         "unit": "GB/s", "frac": round(a / link["bidir"], 4), "traffic": None,
                         "algorithmic_bytes_per_launch": 2 * max(SUMMARY_BATCHES) *
                         max(SUMMARY_SIZES),
                         "bidir_memcpy_nearby_gbs": [near0, near1],
                         "frac_of_nearby": round(a / max(near0, near1), 4),
                         "one_way": {d: {"gbs": round(big[d]["gbs"], 2),
                                         "frac": round(big[d]["gbs"] / peak[d], 4)}
                                     for d in ("d2h", "h2d")}},
            "winner_counts": wins,
            "points": points,
            "clocks": win,
            "cpu_baseline": cpu_record(wl.Geometry(L=1, C=1, P=4096, T=1, H=1, B=65536,
                                                   elem_bytes=1), 1024, 4096, 3.0, seed=1004)}


# ------------------------------------------------------- Llama-8B extras

def write_through(ctx, su):
    """The step's 512 pages written by 8 chunks of a stand-in forward (bf16
    GEMMs on a compute stream, sized near one chunk's backup time); each chunk's
    64 pages are backed up on the copy stream once that chunk's forward is done
    (a GPU-side event wait).  Exposed backup = pipelined - compute-only; the last
    chunk's backup can never overlap and is reported beside it."""
    torch, kvb, w = ctx.torch, ctx.kvb, su.w
    s_a = ctx.s_a
    comp = torch.cuda.Stream(device=ctx.dev)
    M, per_chunk, chunks = 3456, 16, 8
    A = torch.randn(M, M, dtype=torch.bfloat16, device=ctx.dev)
    Bm = torch.randn(M, M, dtype=torch.bfloat16, device=ctx.dev)
    Cm = torch.empty(M, M, dtype=torch.bfloat16, device=ctx.dev)
    cp = w.n // chunks

    def wt_timed(fn):
        def body(i):
            ev = torch.cuda.Event()
            ev.record(s_a)
            comp.wait_event(ev)
            fn(i)
            ev2 = torch.cuda.Event()
            ev2.record(comp)
            s_a.wait_event(ev2)
        return ctx.timed(body, s_a)

    def wt_compute(i):
        with torch.cuda.stream(comp):
            for _ in range(chunks * per_chunk):
                torch.matmul(A, Bm, out=Cm)

    def wt_backup(i, last_only=False):
        ids = su.ids(i)
        for c in range(chunks - 1 if last_only else 0, chunks):
            sl = slice(c * cp, (c + 1) * cp)
            kvb.kv_backup(su.pool, su.tier, ids.backup_src[sl], ids.backup_slots[sl],
                          s_a.cuda_stream)

    def wt_pipelined(i):
        ids = su.ids(i)
        for c in range(chunks):
            with torch.cuda.stream(comp):
                for _ in range(per_chunk):
                    torch.matmul(A, Bm, out=Cm)
            done = torch.cuda.Event()
            done.record(comp)
            s_a.wait_event(done)
            sl = slice(c * cp, (c + 1) * cp)
            kvb.kv_backup(su.pool, su.tier, ids.backup_src[sl], ids.backup_slots[sl],
                          s_a.cuda_stream)

    t_c = wt_timed(wt_compute)
    t_b = wt_timed(wt_backup)
    t_last = wt_timed(lambda i: wt_backup(i, True))
    t_p = wt_timed(wt_pipelined)
    # the SM budget of the backups: k CTAs of 1,024 threads (k whole SMs) each
    budget = []
    if not ctx.args.max_ctas and not ctx.args.cta_threads:
        for k in (4, 6, 8):
            ctx.set_config(max_ctas=k, cta_threads=1024)
            tb_k, tp_k = wt_timed(wt_backup), wt_timed(wt_pipelined)
            budget.append({"sms": k, "backup_only_ms": round(tb_k, 3),
                           "backup_gbs": round(w.n * su.g.page_bytes / (tb_k / 1e3) / GB, 1),
                           "pipelined_ms": round(tp_k, 3),
                           "exposed_backup_ms": round(tp_k - t_c, 3)})
        ctx.set_config()
    del A, Bm, Cm
    return {"forward_stand_in": f"bf16 GEMM {M}^3 x {per_chunk} per chunk on a compute stream",
            "chunks": chunks, "pages_per_chunk": cp,
            "compute_only_ms": round(t_c, 3), "backup_only_ms": round(t_b, 3),
            "pipelined_ms": round(t_p, 3), "exposed_backup_ms": round(t_p - t_c, 3),
            "last_chunk_backup_ms": round(t_last, 3),
            "exposed_beyond_last_chunk_ms": round(t_p - t_c - t_last, 3),
            "sm_budget": budget or None}


def l3_hop(ctx, su):
    """The step's 512 backed-up host slots (1 GiB) put into 512 records of a
    memfd and got back, on the host cores (host memory bandwidth bound)."""
    if not hasattr(os, "memfd_create"):
        return None
    kvb, w, g = ctx.kvb, su.w, su.g
    fd = os.memfd_create("kvb_bench_l3")
    threads = min(16, len(os.sched_getaffinity(0)))
    store = kvb.kv_l3_open(fd, 0, g.page_bytes, w.n, threads)
    ids = su.ids(0)
    recs = np.arange(w.n, dtype=np.int32)
    kvb.kv_l3_put(store, su.host.data_ptr(), w.host_slots, ids.backup_slots, recs)  # grows it
    tp, tg = [], []
    for _ in range(5):
        t0 = time.perf_counter()
        kvb.kv_l3_put(store, su.host.data_ptr(), w.host_slots, ids.backup_slots, recs)
        t1 = time.perf_counter()
        kvb.kv_l3_get(store, su.host.data_ptr(), w.host_slots, recs, ids.backup_slots)
        tp.append(t1 - t0)
        tg.append(time.perf_counter() - t1)
    kvb.kv_l3_close(store)
    os.close(fd)
    return {"store": f"memfd, {w.n} records of {g.page_bytes} bytes, host clock",
            "threads": threads,
            "put_gbs": round(w.n * g.page_bytes / statistics.median(tp) / GB, 2),
            "get_gbs": round(w.n * g.page_bytes / statistics.median(tg) / GB, 2)}


def ring_loop(ctx, kind, name, pools, tier, n_ops, idle_ns, body):
    """Runs body(sub) against a ring served by a host thread (kind "host") or by
    the GPU-resident server (kind "device"), then tears the ring down."""
    torch, kvb = ctx.torch, ctx.kvb
    sub = kvb.kv_ring_create(name, 64)
    srv = kvb.kv_ring_attach(name)
    rs = torch.cuda.Stream(device=ctx.dev)
    stop = threading.Event()
    served = [0]

    def serve_loop():
        while not stop.is_set() and served[0] < n_ops:
            served[0] += kvb.kv_ring_serve(srv, pools, tier, rs.cuda_stream, 64, 200_000_000)

    th, fence = None, None
    if kind == "host":
        th = threading.Thread(target=serve_loop, daemon=True)
        th.start()
    else:
        fence = kvb.kv_ring_serve_device(srv, pools, tier, rs.cuda_stream, n_ops, idle_ns)
    try:
        return body(sub)
    finally:
        if fence is not None:
            kvb.kv_fence_wait(fence, 30_000_000_000)
        stop.set()
        if th is not None:
            th.join(10)
        rs.synchronize()
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)


def small_ops(ctx, su):
    """The tiny workload (8 pages of 16 KiB) through the C ABI: call-to-fence
    latency, the descriptor ring's round trip and throughput."""
    torch, kvb = ctx.torch, ctx.kvb
    s_a = ctx.s_a
    w, g = su.w, su.g
    t = wl.TINY
    tg = t.geom
    tlay = kvb.make_layout(tg.L, tg.C, tg.P, tg.T, tg.H, tg.B, tg.order, tg.dev_heads,
                           tg.elem_bytes)
    talloc = torch.empty(tg.pool_bytes, dtype=torch.uint8, device=ctx.dev)
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
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=ctx.dev)
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
               "backup_us_p99": round(1e6 * sorted(lat_b)[int(0.99 * len(lat_b))], 1),
               "restore_us_p99": round(1e6 * sorted(lat_r)[int(0.99 * len(lat_r))], 1)}

    # descriptor ring round trip (submit -> ticket complete) for the same tiny
    # backups, served by a host thread and by the GPU-resident server
    ring_lat = {}
    iters = 400
    ops = [kvb.make_ring_op(0, srcs[i % 4], slot_sets[i % 2], operation_id=i)
           for i in range(iters)]
    for kind in ("host", "device"):
        def body(sub):
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
            rate = round((iters - half) / (time.perf_counter() - t0))
            return lat[20:], rate

        lat, rate = ring_loop(ctx, kind, f"/kvbbench_{os.getpid()}_{kind}", [tpool], ttier,
                              iters, 2_000_000_000, body)
        ring_lat[f"{kind}_served_descriptors_per_s"] = rate
        if kind == "host":
            # the same stream of descriptors with overlapped backups and restores
            old = kvb.kv_config_get()
            kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes,
                              old.flags | kvb.KV_CFG_OVERLAP_RESTORES |
                              kvb.KV_CFG_OVERLAP_BACKUPS, old.cta_threads)
            try:
                _, rate_ov = ring_loop(ctx, kind, f"/kvbbenchov_{os.getpid()}", [tpool], ttier,
                                       iters, 2_000_000_000, body)
            finally:
                kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags,
                                  old.cta_threads)
            ring_lat["host_served_overlapped_descriptors_per_s"] = rate_ov
        ring_lat[f"{kind}_served_us_median"] = round(1e6 * statistics.median(lat), 1)
        ring_lat[f"{kind}_served_us_p99"] = round(1e6 * sorted(lat)[int(0.99 * len(lat))], 1)
    ring_lat["workload"] = ("tiny: 8 pages x 16 KiB (128 KiB) backup per descriptor, submit "
                            "to ticket complete on the host clock, one descriptor in flight "
                            "(180 timed after 20), then 200 back to back with up to 32 in "
                            "flight (descriptors per second); 4 page sets in rotation, L2 warm")
    latency["ring_round_trip"] = ring_lat

    # descriptor ring throughput: each step is the Llama-8B step as 8 descriptors
    # (4 backups of 128 pages, then 4 restores of 128 pages), all submitted at
    # once, host clock from the first submit to the last ticket
    ring_tp = {}
    steps_r = 6
    per = w.n // 4
    for kind in ("host", "device"):
        def body(sub):
            times = []
            for i in range(steps_r):
                ids = su.ids(i)
                ops8 = [kvb.make_ring_op(0, ids.backup_src[c * per:(c + 1) * per],
                                         ids.backup_slots[c * per:(c + 1) * per])
                        for c in range(4)]
                ops8 += [kvb.make_ring_op(1, ids.restore_slots[c * per:(c + 1) * per],
                                          ids.restore_dst[c * per:(c + 1) * per])
                         for c in range(4)]
                t0 = time.perf_counter()
                tks = [kvb.kv_ring_submit(sub, op) for op in ops8]
                sts = [kvb.kv_ring_wait(sub, tk, 30_000_000_000) for tk in tks]
                times.append(time.perf_counter() - t0)
                if any(sts):
                    raise RuntimeError(f"ring {kind} step {i}: statuses {sts}")
            return times

        times = ring_loop(ctx, kind, f"/kvbbenchtp_{os.getpid()}_{kind}", [su.pool], su.tier,
                          8 * steps_r, 5_000_000_000, body)
        ring_tp[f"{kind}_served_gbs"] = round(2 * w.n * g.page_bytes /
                                              statistics.median(times[1:]) / GB, 2)

    # two rings, each with its own resident server: 4 x 64-page backups into slots
    # 0..255 through one, 4 x 64-page restores from slots 256..511 through the
    # other (disjoint pages and slots), both directions at once; with the default
    # 32 movers per server and with 64 (kv_config.max_ctas)
    def two_rings(movers):
        old_cfg = kvb.kv_config_get()
        kvb.kv_config_set(old_cfg.mode, movers, old_cfg.staging_bytes, old_cfg.flags,
                          old_cfg.cta_threads)
        names = [f"/kvbbenchbi_{os.getpid()}_{x}{movers}" for x in "ab"]
        subs = [kvb.kv_ring_create(nm, 16) for nm in names]
        srvs = [kvb.kv_ring_attach(nm) for nm in names]
        streams = [torch.cuda.Stream(device=ctx.dev) for _ in names]
        fences = [kvb.kv_ring_serve_device(sv, [su.pool], su.tier, st.cuda_stream, 4 * steps_r,
                                           5_000_000_000) for sv, st in zip(srvs, streams)]
        times = []
        q = w.n // 8
        try:
            for i in range(steps_r):
                ids = su.ids(i)
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
        finally:
            for f in fences:
                kvb.kv_fence_wait(f, 30_000_000_000)
            for h in srvs + subs:
                kvb.kv_ring_close(h)
            kvb.kv_config_set(old_cfg.mode, old_cfg.max_ctas, old_cfg.staging_bytes,
                              old_cfg.flags, old_cfg.cta_threads)
        return [round(w.n * g.page_bytes / x / GB, 2) for x in times[1:]]

    near = [bidir_nearby(ctx)]
    two32 = two_rings(0)
    near.append(bidir_nearby(ctx))
    two64 = two_rings(64)
    near.append(bidir_nearby(ctx))
    ring_tp["bidir_memcpy_nearby_gbs"] = near
    ring_tp["device_served_two_rings_gbs"] = statistics.median(two32)
    ring_tp["device_served_two_rings_gbs_steps"] = two32
    ring_tp["device_served_two_rings_64_movers_gbs"] = statistics.median(two64)
    ring_tp["device_served_two_rings_64_movers_gbs_steps"] = two64
    ring_tp["workload"] = ("Llama-8B step as 8 ring descriptors (4 x 128-page backups, then "
                           "4 x 128-page restores; 2 GiB), all submitted at once, host clock "
                           "from the first submit to the last ticket, median of 5 steps; "
                           "two_rings: 4 x 64-page backups and 4 x 64-page restores on two "
                           "rings with a resident server each (32 movers, or 64), at once "
                           "(1 GiB per step; median of 5 steps, each step listed)")
    latency["ring_throughput"] = ring_tp
    kvb.kv_pool_close(tpool)
    kvb.kv_host_close(ttier)
    del talloc, thost
    return latency


def records_summary(line):
    """The line's main figures in a few hundred bytes, last on the line (a
    reader that keeps only the line's tail still sees every record)."""
    out = {"headline": {"gbs": line["value"], "roofline_frac": line["roofline"]["frac"],
                        "e2e_gbs": line["e2e"]["value"]}}
    if line.get("roofline_hbm"):
        out["headline"]["hbm_gather_frac"] = line["roofline_hbm"]["frac"]
    m = line.get("mla_fp8")
    if m:
        out["mla_fp8"] = {
            "one_layer_calls_overlapped_gbs": m["value"], "frac": m["roofline"]["frac"],
            "e2e_gbs": m["e2e"]["value"],
            "plain_calls_gbs": m["plain_calls"]["gbs"],
            "plain_frac": m["plain_calls"]["roofline"]["frac"],
            "progressive_gbs": m["progressive_call"]["gbs"],
            "progressive_frac": m["progressive_call"]["roofline"]["frac"],
            "exposed_ms_beside_gemms": m["overlap_with_compute"]["exposed_transfer_ms"],
            "ring_host_served_gbs": m.get("ring_one_layer_descriptors", {}).get(
                "host_served_gbs"),
            "cpu_gbs": m.get("cpu_baseline", {}).get("value")}
    t = line.get("trtllm_ipc")
    if t:
        out["trtllm_ipc"] = {"gbs": t["value"], "frac_of_bidir": t["roofline"]["frac"],
                             "d2h_gbs": t["per_direction"]["d2h"]["gbs"],
                             "h2d_gbs": t["per_direction"]["h2d"]["gbs"],
                             "hbm_gather_frac": t["roofline_hbm"]["frac"],
                             "cpu_gbs": t.get("cpu_baseline", {}).get("value")}
    w = line.get("sweep")
    if w:
        out["sweep"] = {"both_1MiB_x1024_random_gbs": w["value"],
                        "frac_of_bidir": w["roofline"]["frac"],
                        "one_way_frac": {d: v["frac"] for d, v in w["roofline"]["one_way"].items()},
                        "cpu_gbs": w.get("cpu_baseline", {}).get("value")}
    if line.get("cpu_baseline"):
        out["cpu_baseline_gbs"] = line["cpu_baseline"]["value"]
    return out


def run_ours(args):
    ctx = Ctx(args)
    torch = ctx.torch
    ctx.clk = ClockSampler(ctx.local).start()   # before any warm-up: its start-up is not timed
    ctx.link = measure_link(ctx)
    line, su = headline(ctx)
    w = su.w
    if w is wl.LLAMA8B:
        line["write_through"] = write_through(ctx, su)
        line["l3_hop"] = l3_hop(ctx, su)
        line["latency_small_ops"] = small_ops(ctx, su)
    elif w is wl.MLA_FP8:
        line["mla_fp8"] = mla_layerwise(ctx, su, detail=True)
    su.close()
    del su
    torch.cuda.empty_cache()
    if ctx.ws == 1 and not args.no_subrecords and w is wl.LLAMA8B:
        line["mla_fp8"] = mla_record(ctx)
        torch.cuda.empty_cache()
        line["trtllm_ipc"] = trtllm_record(ctx)
        torch.cuda.empty_cache()
        line["sweep"] = sweep_record(ctx)
        torch.cuda.empty_cache()
    ctx.clk.stop()
    resolve_clocks(line, ctx.clk)
    if ctx.rank == 0 and ctx.ws == 1 and not args.no_cpu_baseline:
        g = w.geom
        gbs, used, sample, _ = oracle_sample(g, w.n, g.P, args.cpu_seconds, seed=w.seed + 2,
                                             layerwise=w is wl.MLA_FP8,
                                             max_steps=200 if w is wl.LLAMA8B else 50)
        line["cpu_baseline"] = {"value": round(gbs, 3), "unit": "GB/s", "cores": used,
                                "kind": "oracle", "sample": sample}
        if w is wl.LLAMA8B:
            gbs1, _, sample1, _ = oracle_sample(g, 64, 1024, max(1.0, args.cpu_seconds / 4),
                                                threads=1, seed=w.seed + 3)
            line["cpu_baseline_single_thread"] = {"value": round(gbs1, 3), "unit": "GB/s",
                                                  "cores": 1, "kind": "oracle",
                                                  "sample": sample1}
            gbs2, sample2 = numpy_statement_sample(max(1.0, args.cpu_seconds / 4))
            line["cpu_baseline_numpy_statement"] = {"value": round(gbs2, 3), "unit": "GB/s",
                                                    "cores": 1,
                                                    "kind": "oracle (numpy statement)",
                                                    "sample": sample2}
    else:
        line["cpu_baseline"] = None
    line["records_summary"] = records_summary(line)
    if ctx.rank == 0:
        print(json.dumps(line), flush=True)
    if ctx.dist is not None:
        ctx.dist.destroy_process_group()


# ------------------------------------------------------------ profile cases

def run_profile_case(args):
    """One kind of transfer repeated on a small case, for profiler captures:
    `warmup` untimed ops then `reps` ops, each one kernel launch
    (kv_move_kernel; kv_bulk_kernel / kv_tsp_kernel for gather and scatter)
    with its fence fused in, so ``ncu -k regex:kv_move -s W -c R`` captures
    exactly the R ops after W warm-up ops.  Cases: backup (zero-copy D2H),
    restore (zero-copy H2D), gather (device gather into a device buffer in
    host layout, HBM only), scatter (its inverse), restore_layer (one-layer
    restores, layer k % L; --overlap lets them overlap), restore_layers (every
    layer in one progressive call)."""
    import torch

    from hierarchical_kv_cache_backup_gb300 import build as kbuild

    kbuild.build_library()
    from hierarchical_kv_cache_backup_gb300 import kvb

    w = {"llama8b": wl.LLAMA8B, "trtllm": wl.TRTLLM, "mla": wl.MLA_FP8}[args.geometry]
    g = w.geom.with_(P=args.pool_pages)
    n = args.pages
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, args.max_ctas, 0,
                      kvb.KV_CFG_OVERLAP_RESTORES if args.overlap else 0, args.cta_threads)
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), w.pool_offset)
    host = torch.empty(n * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), n, g.host_heads, lay)
    buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device="cuda") \
        if args.profile_case in ("gather", "scatter") else None
    ids = [wl.op_ids(wl.Workload("p", 1, g, n=n, host_slots=n), seed=100 + k)
           for k in range(args.warmup + args.reps)]
    s = torch.cuda.Stream()
    f = None
    case = args.profile_case
    for k in range(args.warmup + args.reps):
        i = ids[k]
        if case == "backup":
            f = kvb.kv_backup(pool, tier, i.backup_src, i.backup_slots, s.cuda_stream)
        elif case == "restore":
            f = kvb.kv_restore(pool, tier, i.restore_slots, i.restore_dst, -1, s.cuda_stream)
        elif case == "restore_layer":
            f = kvb.kv_restore(pool, tier, i.restore_slots, i.restore_dst, k % g.L, s.cuda_stream)
        elif case == "restore_layers":
            f = kvb.kv_restore_layers(pool, tier, i.restore_slots, i.restore_dst, 0, g.L,
                                      s.cuda_stream)[-1]
        elif case == "gather":
            f = kvb.kv_device_gather(pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                     i.backup_src, s.cuda_stream)
        else:
            f = kvb.kv_device_scatter(pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                      i.restore_dst, -1, s.cuda_stream)
    kvb.kv_fence_wait(f, 120_000_000_000)
    kvb.kv_pool_close(pool)
    kvb.kv_host_close(tier)
    print(f"profile case {case} on {args.geometry}: {args.warmup} warm-up + {args.reps} ops of "
          f"{n} pages ({n * g.page_bytes / 2**20:.0f} MiB each)")


# --------------------------------------------------------------- full sweep

def run_sweep(args):
    """The full bandwidth sweep (workload 5): every page size in 4 KiB .. 1 MiB x
    batch 1 .. 4096 x sequential / random ids x D2H / H2D / both, in ZERO_COPY,
    STAGED and COPY_ENGINE mode.  Writes one JSON record per point to --out and
    prints a table of the zero-copy GB/s and the winning mode per point."""
    ctx = Ctx(args)
    kvb = ctx.kvb
    sizes = wl.SWEEP_PAGE_BYTES[::2] if args.quick else wl.SWEEP_PAGE_BYTES
    batches = wl.SWEEP_BATCHES[::2] if args.quick else wl.SWEEP_BATCHES
    if args.page_bytes:
        sizes = [x for x in sizes if x in args.page_bytes]
    if args.batches:
        batches = [x for x in batches if x in args.batches]
    modes = (("zero_copy", kvb.KV_MODE_ZERO_COPY), ("staged", kvb.KV_MODE_STAGED),
             ("copy_engine", kvb.KV_MODE_COPY_ENGINE))
    records = sweep_points(ctx, sizes, batches, modes, reps=args.reps, warmup=args.warmup,
                           pages=args.sweep_pages)
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0)
    with open(args.out, "w") as f:
        json.dump({"points": records}, f)
    for ids in ("random", "seq"):
        for direction in ("d2h", "h2d", "both"):
            print(f"\n{direction}, {ids} ids: zero-copy GB/s and the winner "
                  "(z zero-copy, s staged, c copy engine)")
            print("page \\ batch " + " ".join(f"{n:>7d}" for n in batches))
            for pb in sizes:
                cells = []
                for n in batches:
                    pt = {rr["mode"]: rr["gbs"] for rr in records if rr["page_bytes"] == pb and
                          rr["batch"] == n and rr["ids"] == ids and rr["direction"] == direction}
                    win = max(pt, key=pt.get)[0]
                    cells.append(f"{pt['zero_copy']:6.1f}{win}")
                print(f"{pb // 1024:>8d} KiB " + " ".join(cells))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.profile_case:
        run_profile_case(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
