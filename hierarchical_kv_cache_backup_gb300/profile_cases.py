"""Run one kind of transfer repeatedly on a small case, for profiler captures.

    python -m hierarchical_kv_cache_backup_gb300.profile_cases --case backup \\
        --pool-pages 512 --pages 128 --warmup 2 --reps 3

Cases: ``backup`` (zero-copy D2H), ``restore`` (zero-copy H2D), ``gather``
(device-side gather into a device buffer in host layout, HBM only),
``scatter`` (its inverse), ``restore_layer`` (one-layer restores),
``restore_layers`` (every layer in one progressive call).  The
geometry is the Llama-8B page (32 x {K,V} x 8 heads x 16 tokens x 256 B) unless
``--geometry trtllm`` (page-first HND, 40 x 2 x 8 x 32 x 256 B) or ``mla``
(61 layers x 576 B latent x 256 tokens) is given.  Each op is one kernel launch
(kv_move_kernel; kv_bulk_kernel for ``gather`` / ``scatter``) with its fence
fused in, so ``ncu -k regex:kv_move -s W -c R`` captures exactly the R timed ops
after W warm-up ops.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    from hierarchical_kv_cache_backup_gb300 import kvb
    from hierarchical_kv_cache_backup_gb300 import workloads as wl

    p = argparse.ArgumentParser()
    p.add_argument("--case", choices=["backup", "restore", "gather", "scatter", "restore_layer",
                                      "restore_layers"], required=True)
    p.add_argument("--geometry", choices=["llama8b", "trtllm", "mla"], default="llama8b")
    p.add_argument("--pool-pages", type=int, default=512)
    p.add_argument("--pages", type=int, default=128)
    p.add_argument("--warmup", type=int, default=2)
    p.add_argument("--reps", type=int, default=3)
    p.add_argument("--max-ctas", type=int, default=0)
    a = p.parse_args(argv)

    w = {"llama8b": wl.LLAMA8B, "trtllm": wl.TRTLLM, "mla": wl.MLA_FP8}[a.geometry]
    g = w.geom.with_(P=a.pool_pages)
    n = a.pages
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, a.max_ctas, 0)
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), w.pool_offset)
    host = torch.empty(n * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), n, g.host_heads, lay)
    buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device="cuda") \
        if a.case in ("gather", "scatter") else None
    ids = [wl.op_ids(wl.Workload("p", 1, g, n=n, host_slots=n), seed=100 + k)
           for k in range(a.warmup + a.reps)]
    s = torch.cuda.Stream()
    f = None
    for k in range(a.warmup + a.reps):
        i = ids[k]
        if a.case == "backup":
            f = kvb.kv_backup(pool, tier, i.backup_src, i.backup_slots, s.cuda_stream)
        elif a.case == "restore":
            f = kvb.kv_restore(pool, tier, i.restore_slots, i.restore_dst, -1, s.cuda_stream)
        elif a.case == "restore_layer":
            f = kvb.kv_restore(pool, tier, i.restore_slots, i.restore_dst, k % g.L, s.cuda_stream)
        elif a.case == "restore_layers":
            f = kvb.kv_restore_layers(pool, tier, i.restore_slots, i.restore_dst, 0, g.L,
                                      s.cuda_stream)[-1]
        elif a.case == "gather":
            f = kvb.kv_device_gather(pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                     i.backup_src, s.cuda_stream)
        else:
            f = kvb.kv_device_scatter(pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                      i.restore_dst, -1, s.cuda_stream)
    kvb.kv_fence_wait(f, 120_000_000_000)
    kvb.kv_pool_close(pool)
    kvb.kv_host_close(tier)
    print(f"profile case {a.case} on {a.geometry}: {a.warmup} warm-up + {a.reps} ops of {n} pages "
          f"({n * g.page_bytes / 2**20:.0f} MiB each)")


if __name__ == "__main__":
    main()
