"""Overlapped restores (KV_CFG_OVERLAP_RESTORES) against the CPU oracle, over
whole buffers: consecutive restores on one stream that the library may overlap
(other layers, or disjoint destination pages) and ones it must not (a page in
common, another op in between, another pool), each compared with the oracle
applied in call order.  Fences must still complete in call order.

The layer-by-layer restore is the PP prefetch PR's "Layer-wise H2D + forward"
(§PP Prefetch Ticket Path); the result of each restore is RESTORE's copy of
host-tier bytes into destination pages (RFC §Device IPC data path)."""
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

WAIT = 30_000_000_000


@pytest.fixture
def overlap():
    old = kvb.kv_config_get()

    def set_(max_ctas=0, cta_threads=0, flags=kvb.KV_CFG_OVERLAP_RESTORES):
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, max_ctas, 0, flags, cta_threads)

    set_()
    yield set_
    kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)


GEOMS = {
    # MLA latent pool (identity chunks, wide CTAs)
    "mla": wl.MLA_FP8.geom.with_(P=160, L=13),
    # Llama-8B page (identity, K and V)
    "llama8b": wl.LLAMA8B.geom.with_(P=96, L=9),
    # TRT-LLM page-first HND pool, NHD tier (head-order change, 256-thread CTAs)
    "trtllm": wl.TRTLLM.geom.with_(P=72, L=7),
}


def expect_layers(rig, want, slots, dst, layers):
    for layer in layers:
        oracle.restore(oracle_geom(rig.g), want[0], want[1], slots, dst, layer=layer,
                       pool_offset=rig.offset)
    return want


@pytest.mark.parametrize("shape", [(0, 0), (1, 1024), (2, 1024), (3, 256)],
                         ids=["default", "1x1024", "2x1024", "3x256"])
@pytest.mark.parametrize("gname", list(GEOMS))
def test_one_layer_restores_every_layer(gname, shape, overlap):
    """Every layer of n pages restored one layer per call, back to back on one
    stream (all but the first overlapped), in random layer order; whole pool and
    tier equal the oracle's; every fence completes, the last implies the others."""
    g = GEOMS[gname]
    overlap(*shape)
    n = 24
    r = np.random.default_rng(77)
    rig = Rig(g, n, pool_offset=(wl.TRTLLM.pool_offset if gname == "trtllm" else 0), seed=11)
    s = torch.cuda.Stream()
    try:
        slots = r.permutation(n).astype(np.int32)
        dst = wl.distinct_pages(r, g.P, n)
        layers = [int(x) for x in r.permutation(g.L)]
        want = rig.snapshot()
        want = (want[0].copy(), want[1])
        c0 = kvb.kv_overlap_count()
        fences = [kvb.kv_restore(rig.pool, rig.hostt, slots, dst, l, s.cuda_stream)
                  for l in layers]
        assert kvb.kv_overlap_count() - c0 == g.L - 1
        kvb.kv_fence_wait(fences[-1], WAIT)
        for f in fences:
            assert kvb.kv_fence_query(f) == kvb.KV_OK
        rig.assert_equal(expect_layers(rig, want, slots, dst, layers))
    finally:
        rig.close()


def test_same_layer_disjoint_pages_overlap_and_shared_pages_do_not(overlap):
    """Same layer: disjoint destination pages may overlap; a page in common must
    not (the later restore's bytes win, as in call order).  Repeated, since a
    wrong overlap would show only as a race."""
    g = GEOMS["mla"]
    n = 16
    r = np.random.default_rng(5)
    rig = Rig(g, 2 * n, seed=12)
    s = torch.cuda.Stream()
    try:
        for it in range(12):
            want = rig.snapshot()
            want = (want[0].copy(), want[1])
            pages = wl.distinct_pages(r, g.P, 3 * n)
            a, b = pages[:n], pages[n:2 * n]
            shared = np.concatenate([pages[2 * n:2 * n + n // 2], a[:n - n // 2]])  # meets a
            sl1 = r.permutation(2 * n)[:n].astype(np.int32)
            sl2 = r.permutation(2 * n)[:n].astype(np.int32)
            sl3 = r.permutation(2 * n)[:n].astype(np.int32)
            layer = int(r.integers(g.L))
            # (the first may overlap the previous iteration's last restore: other bytes)
            kvb.kv_restore(rig.pool, rig.hostt, sl1, a, layer, s.cuda_stream)
            c0 = kvb.kv_overlap_count()
            kvb.kv_restore(rig.pool, rig.hostt, sl2, b, layer, s.cuda_stream)   # disjoint: overlaps
            assert kvb.kv_overlap_count() - c0 == 1
            # the third shares pages with the first, not with the second: it may
            # overlap only once the first's fence is complete, and must land after it
            f = kvb.kv_restore(rig.pool, rig.hostt, sl3, shared, layer, s.cuda_stream)
            # the fourth writes the third's pages: it may overlap only once the third
            # is done (whether it did depends on timing); the bytes must be the oracle's
            f4 = kvb.kv_restore(rig.pool, rig.hostt, sl1, shared, layer, s.cuda_stream)
            kvb.kv_fence_wait(f4, WAIT)
            assert kvb.kv_fence_query(f) == kvb.KV_OK
            for sl, dd in ((sl1, a), (sl2, b), (sl3, shared), (sl1, shared)):
                expect_layers(rig, want, sl, dd, [layer])
            rig.assert_equal(want)
    finally:
        rig.close()


def test_whole_restores_with_disjoint_pages_overlap(overlap):
    g = GEOMS["llama8b"]
    n = 12
    r = np.random.default_rng(8)
    rig = Rig(g, n, seed=13)
    s = torch.cuda.Stream()
    try:
        want = rig.snapshot()
        want = (want[0].copy(), want[1])
        pages = wl.distinct_pages(r, g.P, 4 * n)
        c0 = kvb.kv_overlap_count()
        fs = []
        for k in range(4):
            sl = r.permutation(n).astype(np.int32)
            dd = pages[k * n:(k + 1) * n]
            fs.append(kvb.kv_restore(rig.pool, rig.hostt, sl, dd, -1, s.cuda_stream))
            oracle.restore(oracle_geom(g), want[0], want[1], sl, dd)
        assert kvb.kv_overlap_count() - c0 == 3
        kvb.kv_fence_wait(fs[-1], WAIT)
        assert all(kvb.kv_fence_query(f) == kvb.KV_OK for f in fs)
        rig.assert_equal(want)
    finally:
        rig.close()


def test_other_work_between_restores_ends_the_overlap(overlap):
    """A backup (reading what the restore wrote), a device gather or a progressive
    restore between two restores on the stream: the next restore does not overlap,
    and the backup and gather see the restored bytes."""
    g = GEOMS["mla"]
    n = 10
    r = np.random.default_rng(9)
    rig = Rig(g, 2 * n, seed=14)
    s = torch.cuda.Stream()
    buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device="cuda")
    og = oracle_geom(g)
    try:
        want = rig.snapshot()
        want = (want[0].copy(), want[1].copy())
        sl = np.arange(n, dtype=np.int32)
        dst = wl.distinct_pages(r, g.P, n)
        c0 = kvb.kv_overlap_count()
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 0, s.cuda_stream)
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 1, s.cuda_stream)           # overlaps
        kvb.kv_backup(rig.pool, rig.hostt, dst, np.arange(n, 2 * n, dtype=np.int32),
                      s.cuda_stream)                                              # reads both
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 2, s.cuda_stream)           # no overlap
        kvb.kv_device_gather(rig.pool, buf.data_ptr(), buf.numel(), g.host_heads, dst,
                             s.cuda_stream)
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 3, s.cuda_stream)           # no overlap
        kvb.kv_restore_layers(rig.pool, rig.hostt, sl, dst, 4, 2, s.cuda_stream)
        f = kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 6, s.cuda_stream)       # no overlap
        f = kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 7, s.cuda_stream)       # overlaps
        assert kvb.kv_overlap_count() - c0 == 2
        kvb.kv_fence_wait(f, WAIT)
        s.synchronize()
        expect_layers(rig, want, sl, dst, [0, 1])
        oracle.backup(og, want[0], want[1], dst, np.arange(n, 2 * n))
        expect_layers(rig, want, sl, dst, [2])
        gathered = np.zeros(n * g.page_bytes, dtype=np.uint8)
        oracle.backup(og, want[0], gathered, dst, np.arange(n))
        expect_layers(rig, want, sl, dst, [3, 4, 5, 6, 7])
        assert np.array_equal(buf.cpu().numpy(), gathered)
        rig.assert_equal(want)
    finally:
        rig.close()


def test_other_pool_or_stream_does_not_chain(overlap):
    """Restores of another pool handle, or on another stream, never overlap a
    restore; the flag off (or programmatic launch off) never overlaps."""
    g = GEOMS["mla"]
    n = 8
    r = np.random.default_rng(10)
    rig = Rig(g, n, seed=15)
    rig2 = Rig(g, n, seed=16)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        want1 = rig.snapshot()
        want1 = (want1[0].copy(), want1[1])
        want2 = rig2.snapshot()
        want2 = (want2[0].copy(), want2[1])
        sl = np.arange(n, dtype=np.int32)
        dst = wl.distinct_pages(r, g.P, n)
        c0 = kvb.kv_overlap_count()
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 0, s1.cuda_stream)
        kvb.kv_restore(rig2.pool, rig2.hostt, sl, dst, 1, s1.cuda_stream)   # other pool
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 2, s2.cuda_stream)     # other stream
        assert kvb.kv_overlap_count() == c0
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 5, None)               # legacy stream
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 6, None)
        assert kvb.kv_overlap_count() == c0
        overlap(flags=kvb.KV_CFG_OVERLAP_RESTORES | kvb.KV_CFG_NO_PDL)
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 3, s2.cuda_stream)
        overlap(flags=0)
        kvb.kv_restore(rig.pool, rig.hostt, sl, dst, 4, s2.cuda_stream)
        assert kvb.kv_overlap_count() == c0
        torch.cuda.synchronize()
        expect_layers(rig, want1, sl, dst, [0, 2, 5, 6, 3, 4])
        expect_layers(rig2, want2, sl, dst, [1])
        rig.assert_equal(want1)
        rig2.assert_equal(want2)
    finally:
        rig.close()
        rig2.close()


def test_compute_stream_waits_see_each_overlapped_layer(overlap):
    """A compute stream waiting on each overlapped layer's fence reads that layer
    already restored (what the oracle says), whatever the later layers do."""
    g = GEOMS["mla"]
    n = 32
    r = np.random.default_rng(12)
    rig = Rig(g, n, seed=17)
    copy_s, comp_s = torch.cuda.Stream(), torch.cuda.Stream()
    og = oracle_geom(g)
    try:
        sl = np.arange(n, dtype=np.int32)
        dst = wl.distinct_pages(r, g.P, n)
        want = rig.snapshot()
        want = (want[0].copy(), want[1])
        expect_layers(rig, want, sl, dst, range(g.L))
        fences = [kvb.kv_restore(rig.pool, rig.hostt, sl, dst, l, copy_s.cuda_stream)
                  for l in range(g.L)]
        lb = g.layer_page_bytes
        got = []
        for l, f in enumerate(fences):
            kvb.kv_fence_stream_wait(f, comp_s.cuda_stream)
            with torch.cuda.stream(comp_s):
                for p in dst[:4]:
                    off = oracle.dev_offset(og, int(p), l, 0, 0, 0)
                    got.append((off, rig.alloc[off:off + lb].clone()))
        comp_s.synchronize()
        for off, t in got:
            assert np.array_equal(t.cpu().numpy(), want[0][off:off + lb]), off
        kvb.kv_fence_wait(fences[-1], WAIT)
        rig.assert_equal(want)
    finally:
        rig.close()


def test_overlap_after_a_multi_launch_restore_and_a_gated_one(overlap):
    """A restore above one launch's 2,048 pages is never overlapped itself but
    starts a run the next restore may overlap; a gated restore in between ends
    the run.  Whole buffers against the oracle in call order."""
    g = wl.Geometry(L=3, C=2, P=5000, T=2, H=1, B=16, elem_bytes=1)
    rig = Rig(g, 4500, seed=21)
    r = np.random.default_rng(22)
    s = torch.cuda.Stream()
    ready = torch.zeros(1, dtype=torch.int64, device="cuda")
    try:
        want = rig.snapshot()
        want = (want[0].copy(), want[1])
        big_sl = r.permutation(4500)[:2100].astype(np.int32)
        big_dst = r.permutation(5000)[:2100].astype(np.int32)
        small_sl = r.permutation(4500)[:300].astype(np.int32)
        small_dst = np.setdiff1d(np.arange(5000), big_dst)[r.permutation(5000 - 2100)[:300]]
        small_dst = small_dst.astype(np.int32)
        c0 = kvb.kv_overlap_count()
        kvb.kv_restore(rig.pool, rig.hostt, big_sl, big_dst, 0, s.cuda_stream)     # 2 launches
        kvb.kv_restore(rig.pool, rig.hostt, small_sl, small_dst, 0, s.cuda_stream)  # disjoint
        assert kvb.kv_overlap_count() - c0 == 1
        kvb.kv_restore(rig.pool, rig.hostt, small_sl, small_dst, 1, s.cuda_stream)  # layer 1
        assert kvb.kv_overlap_count() - c0 == 2
        ready.fill_(5)
        torch.cuda.synchronize()
        kvb.kv_restore_when_ready(rig.pool, rig.hostt, small_sl, small_dst, ready.data_ptr(),
                                  5, 1_000_000_000, 2, s.cuda_stream)               # gated
        f = kvb.kv_restore(rig.pool, rig.hostt, big_sl[:100], big_dst[:100], 1, s.cuda_stream)
        assert kvb.kv_overlap_count() - c0 == 2                                     # after a gate
        kvb.kv_fence_wait(f, 30_000_000_000)
        og = oracle_geom(g)
        for sl, dd, layer in ((big_sl, big_dst, 0), (small_sl, small_dst, 0),
                              (small_sl, small_dst, 1), (small_sl, small_dst, 2),
                              (big_sl[:100], big_dst[:100], 1)):
            oracle.restore(og, want[0], want[1], sl, dd, layer=layer)
        rig.assert_equal(want)
    finally:
        rig.close()


def test_ring_host_server_with_overlapped_restores(overlap):
    """The host ring server issues each descriptor as kv_restore and a completion
    mark on its stream; with the flag on, one-layer restore descriptors of every
    layer still complete in ticket order, and the pool equals the oracle's."""
    import os
    import uuid

    g = GEOMS["mla"]
    n = 20
    r = np.random.default_rng(31)
    rig = Rig(g, n, seed=32)
    name = f"/kvbtest_ovl_{os.getpid()}_{uuid.uuid4().hex[:8]}"
    sub = kvb.kv_ring_create(name, 64)
    srv = kvb.kv_ring_attach(name)
    s = torch.cuda.Stream()
    try:
        want = rig.snapshot()
        want = (want[0].copy(), want[1])
        slots = r.permutation(n).astype(np.int32)
        dst = wl.distinct_pages(r, g.P, n)
        layers = [int(x) for x in r.permutation(g.L)]
        tks = [kvb.kv_ring_submit(sub, kvb.make_ring_op(1, slots, dst, layer=l)) for l in layers]
        served = 0
        while served < len(tks):
            served += kvb.kv_ring_serve(srv, [rig.pool], rig.hostt, s.cuda_stream, 64,
                                        1_000_000_000)
        for tk in tks:
            assert kvb.kv_ring_wait(sub, tk, 30_000_000_000) == kvb.KV_OK
        s.synchronize()
        rig.assert_equal(expect_layers(rig, want, slots, dst, layers))
    finally:
        s.synchronize()
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
        rig.close()


def test_overlapped_backups_and_their_hazards(overlap):
    """KV_CFG_OVERLAP_BACKUPS with KV_CFG_OVERLAP_RESTORES: backups into disjoint
    slots overlap; a backup into a slot an unfinished backup writes, a restore
    reading a slot an unfinished backup writes, and a backup of a page an
    unfinished restore writes all wait.  Whole buffers against the oracle in
    call order, repeated (a wrong overlap would show only as a race)."""
    overlap(flags=kvb.KV_CFG_OVERLAP_RESTORES | kvb.KV_CFG_OVERLAP_BACKUPS)
    g = GEOMS["llama8b"]
    n = 8
    r = np.random.default_rng(41)
    rig = Rig(g, 6 * n, seed=42)
    s = torch.cuda.Stream()
    og = oracle_geom(g)
    try:
        for it in range(10):
            want = rig.snapshot()
            want = (want[0].copy(), want[1].copy())
            pages = wl.distinct_pages(r, g.P, 4 * n)
            slots = r.permutation(6 * n).astype(np.int32)
            sa, sb, sc = slots[:n], slots[n:2 * n], slots[2 * n:3 * n]
            p1, p2, p3 = pages[:n], pages[n:2 * n], pages[2 * n:3 * n]
            ops = []
            kvb.kv_backup(rig.pool, rig.hostt, p1, sa, s.cuda_stream)
            ops.append(("b", p1, sa, -1))
            c0 = kvb.kv_overlap_count()
            kvb.kv_backup(rig.pool, rig.hostt, p2, sb, s.cuda_stream)      # disjoint slots
            ops.append(("b", p2, sb, -1))
            assert kvb.kv_overlap_count() - c0 == 1
            # the next three each conflict with their unfinished predecessor and wait
            # for it (or overlap once it is done: timing); the bytes must be the oracle's
            shared = np.concatenate([sb[:n // 2], sc[:n - n // 2]])        # meets the 2nd
            kvb.kv_backup(rig.pool, rig.hostt, p3, shared, s.cuda_stream)  # WAW on slots
            ops.append(("b", p3, shared, -1))
            kvb.kv_restore(rig.pool, rig.hostt, shared, p1, 2, s.cuda_stream)  # RAW on slots
            ops.append(("r", p1, shared, 2))
            kvb.kv_backup(rig.pool, rig.hostt, p1, sa, s.cuda_stream)      # reads pages the
            ops.append(("b", p1, sa, -1))                                   # restore writes
            f = kvb.kv_restore(rig.pool, rig.hostt, sc, p2, 5, s.cuda_stream)
            ops.append(("r", p2, sc, 5))
            kvb.kv_fence_wait(f, WAIT)
            for kind, pg, sl, layer in ops:
                if kind == "b":
                    oracle.backup(og, want[0], want[1], pg, sl)
                else:
                    oracle.restore(og, want[0], want[1], sl, pg, layer=layer)
            rig.assert_equal(want)
    finally:
        rig.close()


def test_many_small_overlapped_backups(overlap):
    """A stream of 400 small backups (8 pages each) into two alternating slot
    sets, and restores out of them: the tier and pool equal the oracle's and
    consecutive disjoint ops overlapped."""
    overlap(flags=kvb.KV_CFG_OVERLAP_RESTORES | kvb.KV_CFG_OVERLAP_BACKUPS)
    g = wl.TINY.geom.with_(P=64)
    r = np.random.default_rng(43)
    rig = Rig(g, 16, seed=44)
    s = torch.cuda.Stream()
    og = oracle_geom(g)
    try:
        want = rig.snapshot()
        want = (want[0].copy(), want[1].copy())
        c0 = kvb.kv_overlap_count()
        f = None
        for i in range(400):
            sl = np.arange(8 * (i % 2), 8 * (i % 2) + 8, dtype=np.int32)
            pg = r.permutation(g.P)[:8].astype(np.int32)
            if i % 5 == 4:
                f = kvb.kv_restore(rig.pool, rig.hostt, sl, pg, -1, s.cuda_stream)
                oracle.restore(og, want[0], want[1], sl, pg)
            else:
                f = kvb.kv_backup(rig.pool, rig.hostt, pg, sl, s.cuda_stream)
                oracle.backup(og, want[0], want[1], pg, sl)
        kvb.kv_fence_wait(f, WAIT)
        assert kvb.kv_overlap_count() - c0 > 100
        rig.assert_equal(want)
    finally:
        rig.close()
