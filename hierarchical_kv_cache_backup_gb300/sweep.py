"""Bandwidth sweep of the engine: page bytes x batch x id pattern x direction x mode.

    python -m hierarchical_kv_cache_backup_gb300.sweep --out sweep.json [--quick]

Pool: 8192 pages of one opaque run each (L = C = T = H = 1, B = page bytes),
random payload.  For every page size in 4 KiB .. 1 MiB and batch in 1 .. 4096,
with sequential (0..n-1) or seeded-random page ids, it times a backup (D2H),
a restore (H2D) and both at once on two streams (disjoint pages and slots), in
ZERO_COPY, STAGED and COPY_ENGINE mode, with CUDA events on the launching stream (median of
``--reps`` after warm-up; every rep uses another page set so small batches do
not run from L2).  Writes one JSON record per point and prints a table of the
zero-copy GB/s and which mode wins at each point.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


MODES = (("zero_copy", 0), ("staged", 1), ("copy_engine", 2))   # kv_mode values


def main(argv=None):
    import numpy as np
    import torch

    from hierarchical_kv_cache_backup_gb300 import kvb
    from hierarchical_kv_cache_backup_gb300 import workloads as wl

    p = argparse.ArgumentParser()
    p.add_argument("--out", default="sweep.json")
    p.add_argument("--reps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=2)
    p.add_argument("--quick", action="store_true", help="every other page size and batch")
    p.add_argument("--pages", type=int, default=8192)
    p.add_argument("--page-bytes", type=int, nargs="*", help="only these page sizes")
    p.add_argument("--batches", type=int, nargs="*", help="only these batch sizes")
    a = p.parse_args(argv)

    sizes = wl.SWEEP_PAGE_BYTES[::2] if a.quick else wl.SWEEP_PAGE_BYTES
    batches = wl.SWEEP_BATCHES[::2] if a.quick else wl.SWEEP_BATCHES
    if a.page_bytes:
        sizes = [x for x in sizes if x in a.page_bytes]
    if a.batches:
        batches = [x for x in batches if x in a.batches]
    P = a.pages
    max_pb, max_n = max(sizes), max(batches)
    dev_bytes = P * max_pb
    alloc = torch.empty(dev_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, 4004)
    host = torch.empty(2 * max_n * max_pb, dtype=torch.uint8, pin_memory=True)
    host.copy_(alloc[:host.numel()])
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    r = wl.rng(1004)
    records = []

    for pb in sizes:
        g = wl.Geometry(L=1, C=1, P=P, T=1, H=1, B=pb, elem_bytes=1)
        lay = kvb.make_layout(1, 1, P, 1, 1, pb, 0, 0, 1)
        pool = kvb.kv_pool_register(lay, alloc.data_ptr(), 0)
        slots_total = 2 * max_n
        tier = kvb.kv_host_register(host.data_ptr(), slots_total * pb, slots_total, 0, lay)
        for n in batches:
            for pattern in ("seq", "random"):
                sets = []
                for k in range(a.warmup + a.reps):
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
                for mode_name, mode in MODES:
                    kvb.kv_config_set(mode, 0, 0)
                    for direction in ("d2h", "h2d", "both"):
                        ts = []
                        for k, (src, dst) in enumerate(sets):
                            e0 = torch.cuda.Event(enable_timing=True)
                            e1 = torch.cuda.Event(enable_timing=True)
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
                            if k >= a.warmup:
                                ts.append(e0.elapsed_time(e1) / 1000)
                        t = statistics.median(ts)
                        nbytes = n * pb * (2 if direction == "both" else 1)
                        records.append({"page_bytes": pb, "batch": n, "ids": pattern,
                                        "mode": mode_name, "direction": direction,
                                        "seconds": t, "gbs": nbytes / t / 1e9,
                                        "pages_per_s": nbytes / pb / t})
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0)
    with open(a.out, "w") as f:
        json.dump({"points": records}, f)

    # summary: zero-copy GB/s and the winning mode per point
    # (winner: z = zero-copy, s = staged, c = copy engine)
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


if __name__ == "__main__":
    main()
