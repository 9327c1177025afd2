"""GPU test rig: a device pool (inside a larger allocation, at a byte offset),
a pinned host tier, both filled with seeded random bytes, registered through
the C ABI; and the oracle's expected result on byte-exact host copies."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from hierarchical_kv_cache_backup_gb300 import kvb
from hierarchical_kv_cache_backup_gb300 import workloads as wl

TAIL = 4096   # bytes after the pool inside its allocation (must stay untouched)


def oracle_geom(g: wl.Geometry):
    return oracle.geom(g.L, g.C, g.P, g.T, g.H, g.B, page_first=g.order == wl.PAGE_FIRST,
                       dev_hnd=g.dev_heads == wl.HND, host_hnd=g.host_heads == wl.HND)


def layout(g: wl.Geometry):
    return kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)


class Rig:
    def __init__(self, g: wl.Geometry, host_slots: int, pool_offset: int = 0, seed: int = 0,
                 device: str = "cuda:0", register: bool = True):
        self.g = g
        self.offset = pool_offset
        self.slots = host_slots
        self.alloc = torch.empty(pool_offset + g.pool_bytes + TAIL, dtype=torch.uint8, device=device)
        wl.fill_random_(self.alloc, seed)
        self.host = torch.empty(host_slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
        wl.fill_random_(self.host, seed + 1)
        self.layout = layout(g)
        self.pool = self.hostt = None
        if register:
            self.pool = kvb.kv_pool_register(self.layout, self.alloc.data_ptr(), pool_offset)
            self.hostt = kvb.kv_host_register(self.host.data_ptr(), self.host.numel(), host_slots,
                                              g.host_heads, self.layout)

    def close(self):
        if self.pool is not None:
            kvb.kv_pool_close(self.pool)
            self.pool = None
        if self.hostt is not None:
            kvb.kv_host_close(self.hostt)
            self.hostt = None

    def snapshot(self):
        torch.cuda.synchronize()
        return self.alloc.cpu().numpy(), self.host.numpy().copy()

    def expect_backup(self, snap, src, slots, threads=8):
        pool, host = snap[0], snap[1].copy()
        oracle.backup(oracle_geom(self.g), pool, host, src, slots, pool_offset=self.offset,
                      threads=threads)
        return pool, host

    def expect_restore(self, snap, slots, dst, layer=-1, threads=8):
        pool, host = snap[0].copy(), snap[1]
        oracle.restore(oracle_geom(self.g), pool, host, slots, dst, layer=layer,
                       pool_offset=self.offset, threads=threads)
        return pool, host

    def assert_equal(self, want):
        got = self.snapshot()
        for name, a, b in (("pool allocation", got[0], want[0]), ("host tier", got[1], want[1])):
            if not np.array_equal(a, b):
                bad = np.flatnonzero(a != b)
                raise AssertionError(f"{name}: {bad.size} bytes differ, first at {bad[0]} "
                                     f"(got {a[bad[0]]}, want {b[bad[0]]})")
