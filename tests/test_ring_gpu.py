"""Scheduler / data-plane split over the descriptor ring, on one GPU.

The scheduler process owns the pool (a raw allocation at a byte offset) and the
decisions; a second process -- the data plane -- imports the pool through CUDA
IPC, owns the pinned host tier and serves BACKUP / RESTORE descriptors from the
shared-memory ring -- from a host thread, or with the GPU-resident server --
and the GPU completes each ticket in shared memory.  The
scheduler checks its pool against the CPU oracle and sees the data plane's
errors come back through the ring."""
import multiprocessing as mp
import os
import uuid

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from gpu_rig import Rig, oracle_geom  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _data_plane(ring_name, desc_bytes, geom_kw, slots, expected_ops, q, server="host"):
    try:
        import sys
        sys.path[:0] = [ROOT]
        import torch as t
        from hierarchical_kv_cache_backup_gb300 import kvb as k
        from hierarchical_kv_cache_backup_gb300 import workloads as w

        g = w.Geometry(**geom_kw)
        pool = k.kv_pool_import(k.desc_from_bytes(desc_bytes))
        lay, _, _ = k.kv_pool_info(pool)
        host = t.zeros(slots * g.page_bytes, dtype=t.uint8, pin_memory=True)
        tier = k.kv_host_register(host.data_ptr(), host.numel(), slots, g.host_heads, lay)
        ring = k.kv_ring_attach(ring_name)
        stream = t.cuda.Stream()
        served = 0
        if server == "device":   # the resident kernel serves; its first op in this process
            f = k.kv_ring_serve_device(ring, [pool], tier, stream.cuda_stream, expected_ops,
                                       10_000_000_000)
            k.kv_fence_wait(f, 120_000_000_000)
            served, st = k.kv_ring_device_result(ring)
            if st != k.KV_OK:
                raise RuntimeError(f"resident server status {st}")
        while served < expected_ops:
            n = k.kv_ring_serve(ring, [pool], tier, stream.cuda_stream, 8, 30_000_000_000)
            if n == 0:
                break
            served += n
        stream.synchronize()
        k.kv_ring_close(ring)
        k.kv_host_close(tier)
        k.kv_pool_close(pool)
        q.put(("ok", served))
    except Exception as e:
        q.put(("error", repr(e)))


@pytest.mark.parametrize("wname,server", [("trtllm_ipc", "host"), ("llama8b", "host"),
                                          ("trtllm_ipc", "device"), ("llama8b", "device")])
def test_scheduler_and_data_plane_over_the_ring(wname, server):
    w = {x.name: x for x in wl.WORKLOADS}[wname]
    g = w.geom.with_(P=96)
    n = 24
    r = np.random.default_rng(w.seed + 77)
    rig = Rig(g, 1, pool_offset=w.pool_offset, seed=w.seed, register=False)
    pool = kvb.kv_pool_register(rig.layout, rig.alloc.data_ptr(), w.pool_offset, instance_id=5,
                                generation=1)
    name = f"/kvbring_{os.getpid()}_{uuid.uuid4().hex[:8]}"
    ring = kvb.kv_ring_create(name, 8)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    geom_kw = dict(L=g.L, C=g.C, P=g.P, T=g.T, H=g.H, B=g.B, order=g.order,
                   dev_heads=g.dev_heads, host_heads=g.host_heads)
    ops_total = 6
    # the scheduler's own GPU work happens before the data plane starts and after
    # it has ended: its context never competes with the resident server's
    snap = rig.snapshot()
    p = ctx.Process(target=_data_plane, args=(name, kvb.desc_to_bytes(kvb.kv_pool_export(pool)),
                                              geom_kw, n, ops_total, q, server))
    p.start()
    try:
        src = r.permutation(g.P)[:n]
        dst = np.setdiff1d(np.arange(g.P), src)[r.permutation(g.P - n)[:n]]
        slots = r.permutation(n)
        # BACKUP in two descriptors, then RESTORE of every layer, then one layer again
        t1 = kvb.kv_ring_submit(ring, kvb.make_ring_op(0, src[:10], slots[:10], operation_id=1))
        t2 = kvb.kv_ring_submit(ring, kvb.make_ring_op(0, src[10:], slots[10:], operation_id=2))
        assert kvb.kv_ring_wait(ring, t1, 60_000_000_000) == kvb.KV_OK
        assert kvb.kv_ring_wait(ring, t2, 60_000_000_000) == kvb.KV_OK
        t3 = kvb.kv_ring_submit(ring, kvb.make_ring_op(1, slots, dst, operation_id=3))
        assert kvb.kv_ring_wait(ring, t3, 60_000_000_000) == kvb.KV_OK
        # errors found by the data plane come back through the ring
        t4 = kvb.kv_ring_submit(ring, kvb.make_ring_op(1, slots[:2], [1, g.P], operation_id=4))
        t5 = kvb.kv_ring_submit(ring, kvb.make_ring_op(0, src[:1], slots[:1], pool_index=3))
        assert kvb.kv_ring_wait(ring, t4, 60_000_000_000) == kvb.KV_ERR_OUT_OF_RANGE
        assert kvb.kv_ring_wait(ring, t5, 60_000_000_000) == kvb.KV_ERR_INVALID_ARG
        t6 = kvb.kv_ring_submit(ring, kvb.make_ring_op(1, slots[:4], src[:4], layer=g.L - 1))
        assert kvb.kv_ring_wait(ring, t6, 60_000_000_000) == kvb.KV_OK
        status = q.get(timeout=300)
        p.join(120)
        assert status == ("ok", ops_total), status
        # the oracle: backup into a host tier of n slots, then the two restores
        og = oracle_geom(g)
        host = np.zeros(n * g.page_bytes, dtype=np.uint8)
        want = snap[0].copy()
        oracle.backup(og, want, host, src, slots, pool_offset=w.pool_offset, threads=8)
        oracle.restore(og, want, host, slots, dst, pool_offset=w.pool_offset, threads=8)
        oracle.restore(og, want, host, slots[:4], src[:4], layer=g.L - 1,
                       pool_offset=w.pool_offset, threads=8)
        got = rig.snapshot()[0]
        assert np.array_equal(got, want), "pool differs from the oracle"
    finally:
        if p.is_alive():
            p.join(60)
        kvb.kv_ring_close(ring)
        kvb.kv_pool_close(pool)
