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



def test_close_waits_for_a_store_queued_on_a_stream():
    """kv_ring_close unregisters and unmaps the shared segment, so a ready-word
    store still queued on a stream must run first: closing right after one that
    waits behind ~4 s of GPU work returns TIMEOUT and keeps the ring open (the
    segment stays mapped, so the store lands in it); once the stream is done,
    closing the same handle succeeds, and a descriptor gated on that word is
    served at once, its bytes equal to the oracle's BACKUP."""
    import time

    name = f"/kvbtest_close_{os.getpid()}_{uuid.uuid4().hex[:8]}"
    sub = kvb.kv_ring_create(name, 4)
    srv = kvb.kv_ring_attach(name)
    s = torch.cuda.Stream()
    rig = Rig(wl.TINY.geom, wl.TINY.host_slots, seed=3)
    try:
        kvb.kv_ring_ready_stream_set(srv, 3, 1, s.cuda_stream)   # loads the store's kernel
        s.synchronize()
        kvb.kv_ring_close(srv)                                    # nothing pending: closes
        srv = kvb.kv_ring_attach(name)
        with torch.cuda.stream(s):
            torch.cuda._sleep(8_000_000_000)                      # bounded GPU spin, ~4 s
        kvb.kv_ring_ready_stream_set(srv, 3, 7, s.cuda_stream)
        t0 = time.monotonic()
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_close(srv)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
        assert time.monotonic() - t0 >= 1.5
        assert "stays open" in kvb.kv_last_error()
        s.synchronize()                                           # the store has run
        kvb.kv_ring_close(srv)                                    # the same handle closes now
        srv = kvb.kv_ring_attach(name)
        want = rig.expect_backup(rig.snapshot(), [1, 2], [0, 1])
        tk = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1, 2], [0, 1], ready_index=3,
                                                      ready_value=7, ready_timeout_ms=3000))
        served = kvb.kv_ring_serve(srv, [rig.pool], rig.hostt, s.cuda_stream, 1, 1_000_000_000)
        assert served == 1
        assert kvb.kv_ring_wait(sub, tk, 10_000_000_000) == kvb.KV_OK   # not ABORTED
        s.synchronize()
        rig.assert_equal(want)
    finally:
        rig.close()
        if srv is not None:
            s.synchronize()
            kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
