"""The GPU-resident ring server (kv_ring_serve_device) against the oracle and
against the host server.

One process plays both sides here (the ring's creator submits, an attached
handle serves); the resident kernel takes each descriptor from the shared
segment, moves the pages and completes the ticket from the GPU.  Every case
checks the whole pool allocation and host tier against the oracle's replay of
the accepted descriptors, and the status of every ticket -- rejected ones
included -- against what the host server (kv_ring_serve) returns for the same
descriptors on an identical pool."""
import os
import time
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

WAIT = 60_000_000_000


def ring_pair(slots):
    name = f"/kvbdev_{os.getpid()}_{uuid.uuid4().hex[:8]}"
    sub = kvb.kv_ring_create(name, slots)
    return sub, kvb.kv_ring_attach(name)


def replay(g, rig_offset, snap, ops, statuses):
    """The oracle's pool and host tier after the accepted descriptors, in order."""
    og = oracle_geom(g)
    pool, host = snap[0].copy(), snap[1].copy()
    for (kind, a, b, layer, _), st in zip(ops, statuses):
        if st != kvb.KV_OK or len(a) == 0:
            continue
        if kind == kvb.KV_RING_OP_BACKUP:
            oracle.backup(og, pool, host, a, b, pool_offset=rig_offset, threads=8)
        else:
            oracle.restore(og, pool, host, a, b, layer=layer, pool_offset=rig_offset, threads=8)
    return pool, host


def random_ops(r, g, S, count, npools=1, n_range=(0, 12)):
    """Seeded descriptors: backups and whole / one-layer restores, some of them
    made invalid (ids out of range or negative, repeated write targets, a bad
    layer, a pool index past the table, a backup with a layer)."""
    ops = []
    for _ in range(count):
        kind = int(r.integers(2))
        hi = min(n_range[1], S, g.P)
        n = int(r.integers(min(n_range[0], hi), hi + 1))
        if kind == kvb.KV_RING_OP_BACKUP:
            a = r.integers(0, g.P, n)
            b = r.permutation(S)[:n]
            layer = -1
        else:
            a = r.integers(0, S, n)
            b = r.permutation(g.P)[:n]
            layer = -1 if r.random() < 0.5 else int(r.integers(0, g.L))
        pool_index = 0
        x = r.random()
        lim_a, lim_b = (g.P, S) if kind == 0 else (S, g.P)
        if x < 0.08 and n:
            a[r.integers(n)] = lim_a + int(r.integers(3))
        elif x < 0.16 and n:
            b[r.integers(n)] = lim_b + int(r.integers(3))
        elif x < 0.24 and n >= 2:
            i, j = sorted(r.choice(n, 2, replace=False))
            b[j] = b[i]                                  # a later repeat
        elif x < 0.28 and n:
            b[r.integers(n)] = -1 - int(r.integers(5))
        elif x < 0.32:
            layer = g.L if kind == 1 else 0             # out of range / backup with a layer
        elif x < 0.36:
            layer = -2
        elif x < 0.40:
            pool_index = npools + int(r.integers(2))
        ops.append((kind, a.astype(np.int64), b.astype(np.int64), layer, pool_index))
    return ops


def submit_all(sub, ops):
    return [kvb.kv_ring_submit(sub, kvb.make_ring_op(k, a, b, pool_index=pi, layer=ly,
                                                     operation_id=i), WAIT)
            for i, (k, a, b, ly, pi) in enumerate(ops)]


def run_device(g, w_offset, seed, S, ops, stream, max_ops=None, idle_ns=2_000_000_000):
    rig = Rig(g, S, pool_offset=w_offset, seed=seed)
    sub, srv = ring_pair(max(2, len(ops)))
    try:
        snap = rig.snapshot()
        fence = kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream,
                                         max_ops or len(ops), idle_ns)
        tickets = submit_all(sub, ops)
        statuses = [kvb.kv_ring_wait(sub, t, WAIT) for t in tickets]
        kvb.kv_fence_wait(fence, WAIT)
        served, st = kvb.kv_ring_device_result(srv)
        after = rig.snapshot()
        return snap, after, statuses, (served, st)
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()


def run_host(g, w_offset, seed, S, ops, stream):
    rig = Rig(g, S, pool_offset=w_offset, seed=seed)
    sub, srv = ring_pair(max(2, len(ops)))
    try:
        snap = rig.snapshot()
        tickets = submit_all(sub, ops)
        served = kvb.kv_ring_serve(srv, [rig.pool], rig.hostt, stream.cuda_stream, len(ops),
                                   1_000_000_000)
        statuses = [kvb.kv_ring_wait(sub, t, WAIT) for t in tickets]
        stream.synchronize()
        return snap, rig.snapshot(), statuses, served
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()


@pytest.mark.parametrize("wname", ["tiny", "llama8b", "mla_fp8", "trtllm_ipc"])
def test_device_server_matches_the_oracle(wname):
    """A fixed sequence -- two backups, a whole restore, a one-layer restore, an
    empty descriptor and five rejected ones -- through the resident server."""
    w = {x.name: x for x in wl.WORKLOADS}[wname]
    g = w.geom.with_(P=min(w.geom.P, 96))
    n = min(24, g.P // 3)
    S = n + 4
    r = np.random.default_rng(w.seed + 5)
    src = r.permutation(g.P)[:n]
    dst = np.setdiff1d(np.arange(g.P), src)[r.permutation(g.P - n)[:n]]
    slots = r.permutation(S)[:n]
    ops = [(0, src[:n // 2], slots[:n // 2], -1, 0),
           (0, src[n // 2:], slots[n // 2:], -1, 0),
           (1, slots, dst, -1, 0),
           (1, slots[:3], src[:3], g.L - 1, 0),
           (0, src[:0], slots[:0], -1, 0),
           (1, slots[:2], np.array([1, g.P]), -1, 0),          # OUT_OF_RANGE
           (1, slots[:3], np.array([4, 5, 4]), -1, 0),         # DUPLICATE
           (0, src[:1], slots[:1], -1, 3),                     # INVALID_ARG: pool index
           (0, src[:1], slots[:1], 0, 0),                      # INVALID_ARG: backup with a layer
           (1, slots[:1], src[:1], g.L, 0)]                    # OUT_OF_RANGE: layer
    stream = torch.cuda.Stream()
    snap, after, statuses, (served, st) = run_device(g, w.pool_offset, w.seed, S, ops, stream)
    assert statuses == [0, 0, 0, 0, 0, kvb.KV_ERR_OUT_OF_RANGE, kvb.KV_ERR_DUPLICATE,
                        kvb.KV_ERR_INVALID_ARG, kvb.KV_ERR_INVALID_ARG, kvb.KV_ERR_OUT_OF_RANGE]
    assert (served, st) == (len(ops), kvb.KV_OK)
    want = replay(g, w.pool_offset, snap, ops, statuses)
    assert np.array_equal(after[0], want[0]), "pool allocation differs from the oracle"
    assert np.array_equal(after[1], want[1]), "host tier differs from the oracle"


CASES = int(os.environ.get("KVB_RING_DEVICE_CASES", "24"))


@pytest.mark.parametrize("case", range(CASES))
def test_device_server_agrees_with_host_server_on_random_descriptors(case):
    """Seeded geometries and descriptor lists, run once through the host server
    and once through the resident server on identical pools: the same status
    for every ticket, and both results equal the oracle's replay."""
    r = np.random.default_rng(4000 + case)
    order, dev, host = (int(x) for x in r.integers(0, 2, 3))
    g = wl.Geometry(L=int(r.integers(1, 5)), C=int(r.integers(1, 3)), P=int(r.integers(8, 60)),
                    T=int(r.integers(1, 33)), H=int(r.integers(1, 9)), B=16 * int(r.integers(1, 17)),
                    order=order, dev_heads=dev, host_heads=host)
    S = int(r.integers(4, 24))
    offset = 16 * int(r.integers(0, 64))
    ops = random_ops(r, g, S, int(r.integers(4, 14)))
    stream = torch.cuda.Stream()
    h_snap, h_after, h_st, h_served = run_host(g, offset, 100 + case, S, ops, stream)
    d_snap, d_after, d_st, (served, st) = run_device(g, offset, 100 + case, S, ops, stream)
    assert d_st == h_st, (d_st, h_st)
    assert (served, st) == (len(ops), kvb.KV_OK) and h_served == len(ops)
    want = replay(g, offset, d_snap, ops, d_st)
    assert np.array_equal(d_after[0], want[0]) and np.array_equal(d_after[1], want[1])
    assert np.array_equal(h_after[0], want[0]) and np.array_equal(h_after[1], want[1])


@pytest.mark.parametrize("case", range(CASES // 3))
def test_device_server_agrees_with_host_server_on_large_descriptors(case):
    """As above with 33 to 1,024 ids per descriptor (the block-wide duplicate
    check rather than the one-warp one), on pools of many small pages."""
    r = np.random.default_rng(6000 + case)
    order, dev, host = (int(x) for x in r.integers(0, 2, 3))
    g = wl.Geometry(L=int(r.integers(1, 4)), C=int(r.integers(1, 3)),
                    P=int(r.integers(300, 1300)), T=int(r.integers(1, 9)),
                    H=int(r.integers(1, 5)), B=16 * int(r.integers(1, 5)),
                    order=order, dev_heads=dev, host_heads=host)
    S = int(r.integers(100, 1100))
    offset = 16 * int(r.integers(0, 64))
    ops = random_ops(r, g, S, int(r.integers(3, 9)), n_range=(33, 1024))
    stream = torch.cuda.Stream()
    h_snap, h_after, h_st, h_served = run_host(g, offset, 300 + case, S, ops, stream)
    d_snap, d_after, d_st, (served, st) = run_device(g, offset, 300 + case, S, ops, stream)
    assert d_st == h_st, (d_st, h_st)
    assert (served, st) == (len(ops), kvb.KV_OK) and h_served == len(ops)
    want = replay(g, offset, d_snap, ops, d_st)
    assert np.array_equal(d_after[0], want[0]) and np.array_equal(d_after[1], want[1])
    assert np.array_equal(h_after[0], want[0]) and np.array_equal(h_after[1], want[1])


def test_device_server_ends_when_idle_and_refuses_a_second_server():
    g = wl.TINY.geom
    rig = Rig(g, 16, seed=31)
    sub, srv = ring_pair(4)
    stream = torch.cuda.Stream()
    try:
        snap = rig.snapshot()
        t0 = time.perf_counter()
        fence = kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 100,
                                         300_000_000)
        with pytest.raises(kvb.KvError) as e:                 # one resident server per ring
            kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 1, 1000)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
        with pytest.raises(kvb.KvError) as e:                 # no result while it runs
            kvb.kv_ring_device_result(srv)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
        ops = [(0, [5, 9], [0, 3], -1, 0), (1, [0, 3], [20, 21], 0, 0)]
        tickets = submit_all(sub, ops)
        assert [kvb.kv_ring_wait(sub, t, WAIT) for t in tickets] == [0, 0]
        kvb.kv_fence_wait(fence, WAIT)
        assert time.perf_counter() - t0 >= 0.3                # ended by the idle bound
        assert kvb.kv_ring_device_result(srv) == (2, kvb.KV_OK)
        want = replay(g, 0, snap, ops, [0, 0])
        rig.assert_equal(want)
        # a second server on the same ring takes up at the next ticket
        fence = kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 1,
                                         WAIT // 100)
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [7], [9]))
        assert kvb.kv_ring_wait(sub, t, WAIT) == kvb.KV_OK
        kvb.kv_fence_wait(fence, WAIT)
        assert kvb.kv_ring_device_result(srv) == (1, kvb.KV_OK)
        want = replay(g, 0, want, [(0, [7], [9], -1, 0)], [0])
        rig.assert_equal(want)
        # limits checked before anything is enqueued
        for args, status in (((srv, [], rig.hostt), kvb.KV_ERR_INVALID_ARG),
                             ((srv, [rig.pool], 0), kvb.KV_ERR_INVALID_ARG)):
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_ring_serve_device(*args, stream.cuda_stream, 1, 1000)
            assert e.value.status == status
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 1,
                                     61_000_000_000)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()


def test_device_server_with_two_pools_and_a_split_pool():
    """A table of two pools (one contiguous page-first HND, one split layer-first
    NHD of the same slot geometry); descriptors pick their pool by index."""
    ga = wl.Geometry(L=3, C=2, P=40, T=16, H=4, B=64, order=wl.PAGE_FIRST, dev_heads=wl.HND)
    gb = ga.with_(order=wl.LAYER_FIRST, dev_heads=wl.NHD)
    S = 12
    rig = Rig(ga, S, pool_offset=32, seed=41)
    chunk = gb.P * gb.T * gb.H * gb.B
    bufs = [torch.empty(chunk, dtype=torch.uint8, device="cuda") for _ in range(gb.L * gb.C)]
    for k, b in enumerate(bufs):
        wl.fill_random_(b, 4200 + k)
    lay_b = kvb.make_layout(gb.L, gb.C, gb.P, gb.T, gb.H, gb.B, gb.order, gb.dev_heads)
    pool_b = kvb.kv_pool_register_split(lay_b, [b.data_ptr() for b in bufs])
    sub, srv = ring_pair(8)
    stream = torch.cuda.Stream()
    try:
        snap = rig.snapshot()
        flat = torch.cat(bufs).cpu().numpy()
        fence = kvb.kv_ring_serve_device(srv, [rig.pool, pool_b], rig.hostt, stream.cuda_stream,
                                         4, WAIT // 10)
        ops = [(0, [3, 17, 39], [0, 1, 2], -1, 0),     # pool 0 -> slots 0..2
               (1, [0, 1, 2], [5, 6, 7], -1, 1),       # slots -> split pool pages 5..7
               (0, [11, 12], [3, 4], -1, 1),           # split pool -> slots 3, 4
               (1, [3, 4], [30, 31], 1, 0)]            # layer 1 of slots 3, 4 -> pool 0
        tickets = submit_all(sub, ops)
        assert [kvb.kv_ring_wait(sub, t, WAIT) for t in tickets] == [0, 0, 0, 0]
        kvb.kv_fence_wait(fence, WAIT)
        assert kvb.kv_ring_device_result(srv) == (4, kvb.KV_OK)
        oa, ob = oracle_geom(ga), oracle_geom(gb)
        pool_a, host = snap[0].copy(), snap[1].copy()
        oracle.backup(oa, pool_a, host, [3, 17, 39], [0, 1, 2], pool_offset=32)
        oracle.restore(ob, flat, host, [0, 1, 2], [5, 6, 7])
        oracle.backup(ob, flat, host, [11, 12], [3, 4])
        oracle.restore(oa, pool_a, host, [3, 4], [30, 31], layer=1, pool_offset=32)
        rig.assert_equal((pool_a, host))
        assert np.array_equal(torch.cat(bufs).cpu().numpy(), flat), "split pool"
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        kvb.kv_pool_close(pool_b)
        rig.close()


def test_device_server_stops_on_request_and_on_close():
    """kv_ring_device_stop ends a resident server well before its idle limit,
    after the descriptor it is moving; closing the serving handle stops a
    running server before unmapping anything."""
    g = wl.TINY.geom
    rig = Rig(g, 16, seed=33)
    sub, srv = ring_pair(4)
    stream = torch.cuda.Stream()
    try:
        snap = rig.snapshot()
        with pytest.raises(kvb.KvError) as e:                 # nothing to stop yet
            kvb.kv_ring_device_stop(srv)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
        fence = kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 1000,
                                         30_000_000_000)
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [4, 8], [1, 2]))
        assert kvb.kv_ring_wait(sub, t, WAIT) == kvb.KV_OK
        t0 = time.perf_counter()
        kvb.kv_ring_device_stop(srv)
        kvb.kv_fence_wait(fence, WAIT)
        assert time.perf_counter() - t0 < 5.0                 # not the 30 s idle limit
        assert kvb.kv_ring_device_result(srv) == (1, kvb.KV_OK)
        rig.assert_equal(replay(g, 0, snap, [(0, [4, 8], [1, 2], -1, 0)], [0]))
        # a running server, then close of its handle: stopped first, then unmapped
        kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream, 1000,
                                 30_000_000_000)
        t0 = time.perf_counter()
        kvb.kv_ring_close(srv)
        srv = None
        assert time.perf_counter() - t0 < 5.0
        stream.synchronize()
    finally:
        if srv is not None:
            kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()


def test_two_resident_servers_at_once():
    """Two rings, each with its own resident server on its own stream (both
    grids resident together): backups through one ring and restores through
    the other, over disjoint pages and slots, submitted interleaved; the pool
    and host tier equal the oracle's."""
    g = wl.LLAMA8B.geom.with_(P=256)
    S = 96
    rig = Rig(g, S, seed=51)
    sub_a, srv_a = ring_pair(8)
    sub_b, srv_b = ring_pair(8)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    r = np.random.default_rng(52)
    pages = r.permutation(g.P)
    back_src, rest_dst = pages[:96], pages[96:192]
    back_slots, rest_slots = np.arange(0, 48), np.arange(48, 96)
    try:
        snap = rig.snapshot()
        fa = kvb.kv_ring_serve_device(srv_a, [rig.pool], rig.hostt, sa.cuda_stream, 4, WAIT // 10)
        fb = kvb.kv_ring_serve_device(srv_b, [rig.pool], rig.hostt, sb.cuda_stream, 4, WAIT // 10)
        ta, tb = [], []
        for c in range(4):
            q = slice(12 * c, 12 * c + 12)
            ta.append(kvb.kv_ring_submit(sub_a, kvb.make_ring_op(0, back_src[q], back_slots[q])))
            tb.append(kvb.kv_ring_submit(sub_b, kvb.make_ring_op(1, rest_slots[q], rest_dst[q])))
        assert [kvb.kv_ring_wait(sub_a, t, WAIT) for t in ta] == [0] * 4
        assert [kvb.kv_ring_wait(sub_b, t, WAIT) for t in tb] == [0] * 4
        kvb.kv_fence_wait(fa, WAIT)
        kvb.kv_fence_wait(fb, WAIT)
        assert kvb.kv_ring_device_result(srv_a) == (4, kvb.KV_OK)
        assert kvb.kv_ring_device_result(srv_b) == (4, kvb.KV_OK)
        og = oracle_geom(g)
        pool, host = snap[0].copy(), snap[1].copy()
        oracle.restore(og, pool, snap[1], rest_slots[:48], rest_dst[:48], threads=8)
        oracle.backup(og, snap[0], host, back_src[:48], back_slots, threads=8)
        rig.assert_equal((pool, host))
    finally:
        for h in (srv_a, srv_b, sub_a, sub_b):
            kvb.kv_ring_close(h)
        rig.close()


@pytest.mark.parametrize("movers", [1, 7, 64])
def test_device_server_with_other_mover_counts(movers):
    """kv_config.max_ctas sets the resident server's mover CTAs: one, an odd
    count and 64 give the same results and statuses as the oracle and the
    host server."""
    r = np.random.default_rng(7000 + movers)
    g = wl.Geometry(L=3, C=2, P=200, T=8, H=4, B=64, order=wl.PAGE_FIRST, dev_heads=wl.HND)
    S = 150
    ops = random_ops(r, g, S, 10, n_range=(1, 120))
    old = kvb.kv_config_get()
    stream = torch.cuda.Stream()
    try:
        h_snap, h_after, h_st, _ = run_host(g, 48, 90 + movers, S, ops, stream)
        kvb.kv_config_set(old.mode, movers, old.staging_bytes, old.flags, old.cta_threads)
        d_snap, d_after, d_st, (served, st) = run_device(g, 48, 90 + movers, S, ops, stream)
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
    assert d_st == h_st and (served, st) == (len(ops), kvb.KV_OK)
    want = replay(g, 48, d_snap, ops, d_st)
    assert np.array_equal(d_after[0], want[0]) and np.array_equal(d_after[1], want[1])


@pytest.mark.parametrize("case", range(4))
def test_device_server_keeps_ticket_order_on_one_layer_restores(case):
    """Streams of one-layer restores over a few layers -- consecutive ones at
    the same layer into overlapping pages (the later write must win), at other
    layers -- mixed with backups that read pages just restored and restores
    that read slots just backed up, a large descriptor followed by a small one
    so that a pair run out of order would show.  Bytes against the oracle's
    replay in ticket order, every ticket OK."""
    g = wl.Geometry(L=6, C=1, P=160, T=64, H=1, B=576, order=wl.LAYER_FIRST, dev_heads=wl.NHD,
                    host_heads=wl.NHD)
    S = 96
    r = np.random.default_rng(4100 + case)
    ops = []
    for i in range(72):
        x = r.random()
        n = int(r.choice([64, 3])) if i % 2 == 0 else int(r.integers(1, 64))
        if x < 0.12:                                     # backup of pages restored before
            pages = r.integers(0, g.P, n)
            ops.append((kvb.KV_RING_OP_BACKUP, pages, r.permutation(S)[:n], -1, 0))
        elif x < 0.18:                                   # whole restore
            ops.append((kvb.KV_RING_OP_RESTORE, r.integers(0, S, n), r.permutation(g.P)[:n],
                        -1, 0))
        else:                                            # one-layer restore, few layers
            layer = int(r.integers(0, 3)) if case % 2 == 0 else int(r.integers(0, g.L))
            dst = r.permutation(40)[:min(n, 40)]        # pages 0..39: consecutive ones overlap
            ops.append((kvb.KV_RING_OP_RESTORE, r.integers(0, S, dst.size), dst, layer, 0))
    stream = torch.cuda.Stream()
    snap, after, statuses, (served, st) = run_device(g, 4096, 4200 + case, S, ops, stream)
    assert statuses == [kvb.KV_OK] * len(ops)
    assert (served, st) == (len(ops), kvb.KV_OK)
    want = replay(g, 4096, snap, ops, statuses)
    assert np.array_equal(after[0], want[0]), "pool allocation differs from the oracle"
    assert np.array_equal(after[1], want[1]), "host tier differs from the oracle"


def test_device_server_one_layer_restores_of_a_prefix():
    """Every layer of a 64-page prefix as its own descriptor, layer after layer,
    twice from different slots into the same pages: the second pass's bytes
    win everywhere."""
    g = wl.MLA_FP8.geom.with_(P=96)
    S = 72
    r = np.random.default_rng(4300)
    dst = r.permutation(g.P)[:64]
    ops = [(kvb.KV_RING_OP_RESTORE, r.permutation(S)[:64], dst, l, 0) for l in range(g.L)]
    ops += [(kvb.KV_RING_OP_RESTORE, r.permutation(S)[:64], dst, l, 0) for l in range(g.L)]
    stream = torch.cuda.Stream()
    snap, after, statuses, (served, st) = run_device(g, 0, 4301, S, ops, stream)
    assert statuses == [kvb.KV_OK] * len(ops)
    assert (served, st) == (len(ops), kvb.KV_OK)
    want = replay(g, 0, snap, ops, statuses)
    assert np.array_equal(after[0], want[0]), "pool allocation differs from the oracle"
    assert np.array_equal(after[1], want[1]), "host tier differs from the oracle"


@pytest.mark.parametrize("server", ["host", "device"])
def test_gated_descriptors_wait_for_their_ready_words(server):
    """Descriptors with a ready fence, served by a host thread and by the
    resident server: a backup that waits until the submitter sets its ready word
    from the CPU (the restore behind it waits in ticket order), one whose word
    is never set (ABORTED after its 200 ms bound, nothing moved, the ring goes
    on), and a restore released from the submitter's GPU stream after other
    work on it.  Bytes against the oracle's replay of the moved descriptors."""
    import threading
    g = wl.TINY.geom.with_(P=48)
    S = 16
    r = np.random.default_rng(5100 + (server == "device"))
    pages = r.permutation(g.P)
    ops = [(0, pages[0:4], np.arange(0, 4), -1, 0, dict(ready_index=2, ready_value=5,
                                                        ready_timeout_ms=5000)),
           (1, np.arange(0, 4), pages[4:8], -1, 0, {}),
           (0, pages[8:12], np.arange(4, 8), -1, 0, dict(ready_index=7, ready_value=1,
                                                         ready_timeout_ms=200)),
           (0, pages[12:16], np.arange(8, 12), -1, 0, {}),
           (1, np.arange(8, 12), pages[16:20], 1, 0, dict(ready_index=9, ready_value=3,
                                                           ready_timeout_ms=5000))]
    rig = Rig(g, S, seed=5200)
    sub, srv = ring_pair(8)
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    # load the stand-in forward's kernel before any gate waits: with lazy module
    # loading a kernel's first launch waits for the device to go idle, which a
    # gate spinning for this very stream's word would hold off until its bound
    torch.cuda._sleep(1000)
    torch.cuda.synchronize()
    th, fence = None, None
    try:
        snap = rig.snapshot()
        if server == "device":
            fence = kvb.kv_ring_serve_device(srv, [rig.pool], rig.hostt, stream.cuda_stream,
                                             len(ops), 5_000_000_000)
        else:
            def serve():
                left = len(ops)
                for _ in range(10):   # bounded: each call waits at most 5 s for a descriptor
                    if left == 0:
                        break
                    left -= kvb.kv_ring_serve(srv, [rig.pool], rig.hostt, stream.cuda_stream,
                                              left, 5_000_000_000)
            th = threading.Thread(target=serve, daemon=True)
            th.start()
        tickets = [kvb.kv_ring_submit(sub, kvb.make_ring_op(k, a, b, pool_index=pi, layer=ly,
                                                            operation_id=i, **gate), WAIT)
                   for i, (k, a, b, ly, pi, gate) in enumerate(ops)]
        time.sleep(0.05)
        with pytest.raises(kvb.KvError) as e:            # its ready word is still 0
            kvb.kv_ring_wait(sub, tickets[0], 20_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
        kvb.kv_ring_ready_set(sub, 2, 5)
        assert kvb.kv_ring_wait(sub, tickets[0], WAIT) == kvb.KV_OK
        assert kvb.kv_ring_wait(sub, tickets[1], WAIT) == kvb.KV_OK
        assert kvb.kv_ring_wait(sub, tickets[2], WAIT) == kvb.KV_ERR_ABORTED
        assert kvb.kv_ring_wait(sub, tickets[3], WAIT) == kvb.KV_OK
        with torch.cuda.stream(side):                    # the submitter's "forward", then the word
            torch.cuda._sleep(2_000_000)
            kvb.kv_ring_ready_stream_set(sub, 9, 3, side.cuda_stream)
        assert kvb.kv_ring_wait(sub, tickets[4], WAIT) == kvb.KV_OK
        if fence is not None:
            kvb.kv_fence_wait(fence, WAIT)
            assert kvb.kv_ring_device_result(srv) == (len(ops), kvb.KV_OK)
        if th is not None:
            th.join(30)
        stream.synchronize()
        side.synchronize()
        after = rig.snapshot()
        statuses = [kvb.KV_OK, kvb.KV_OK, kvb.KV_ERR_ABORTED, kvb.KV_OK, kvb.KV_OK]
        want = replay(g, 0, snap, [op[:5] for op in ops], statuses)
        assert np.array_equal(after[0], want[0]), "pool allocation differs from the oracle"
        assert np.array_equal(after[1], want[1]), "host tier differs from the oracle"
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()
