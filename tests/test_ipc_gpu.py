"""CUDA IPC: a second process on the same GPU imports the pool through the C ABI
(allocation base + byte offset) and drives backup / restore on it; results are
checked byte for byte against the CPU oracle in the exporting process.  Also:
refcounted double import, and an exporter that exits while the importer still
holds the mapping (the mapping keeps the memory alive until it is closed)."""
import multiprocessing as mp
import os
import tempfile

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_rig import Rig, oracle_geom  # noqa: E402
import oracle  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child_drive(desc_bytes, geom_kw, ids, host_slots, host_seed, out_path, q):
    """Importer: maps the pool, owns its own pinned host tier, runs a backup on one
    stream while a restore runs on another, then saves its host tier."""
    try:
        import sys
        sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
        import torch as t
        from hierarchical_kv_cache_backup_gb300 import kvb as k
        from hierarchical_kv_cache_backup_gb300 import workloads as w

        g = w.Geometry(**geom_kw)
        desc = k.desc_from_bytes(desc_bytes)
        pool = k.kv_pool_import(desc)
        pool2 = k.kv_pool_import(desc)            # second import shares the mapping
        lay, ptr, nbytes = k.kv_pool_info(pool)
        host = t.empty(host_slots * g.page_bytes, dtype=t.uint8, pin_memory=True)
        w.fill_random_(host, host_seed)
        tier = k.kv_host_register(host.data_ptr(), host.numel(), host_slots, g.host_heads, lay)
        sa, sb = t.cuda.Stream(), t.cuda.Stream()
        fa = k.kv_backup(pool, tier, ids["backup_src"], ids["backup_slots"], sa.cuda_stream)
        fb = k.kv_restore(pool2, tier, ids["restore_slots"], ids["restore_dst"], -1, sb.cuda_stream)
        k.kv_fence_wait(fa, 30_000_000_000)
        k.kv_fence_wait(fb, 30_000_000_000)
        k.kv_pool_close(pool2)
        # the first handle still works after the second is closed
        f = k.kv_backup(pool, tier, [], [])
        k.kv_fence_wait(f, 30_000_000_000)
        k.kv_pool_close(pool)
        k.kv_host_close(tier)
        np.save(out_path, host.numpy())
        q.put(("ok", desc.alloc_offset, nbytes))
    except Exception as e:  # reported to the parent
        q.put(("error", repr(e), 0))


@pytest.mark.parametrize("P", [96, 2048], ids=["reduced", "full_2048_pages"])
def test_import_in_second_process_trtllm(P):
    w = wl.TRTLLM
    g = w.geom.with_(P=P)
    n = P // 4
    wk = wl.Workload("t", 3, g, n=n, host_slots=2 * n, pool_offset=w.pool_offset, concurrent=True)
    ids = wl.op_ids(wk)
    rig = Rig(g, 1, pool_offset=w.pool_offset, seed=w.seed, register=False)
    lay = rig.layout
    pool = kvb.kv_pool_register(lay, rig.alloc.data_ptr(), w.pool_offset, instance_id=11,
                                generation=1)
    try:
        desc = kvb.kv_pool_export(pool)
        assert desc.alloc_offset == w.pool_offset      # torch gave the allocation its own base
        assert desc.nbytes == g.pool_bytes and desc.generation == 1
        snap = rig.snapshot()
        host_seed = 4321
        # expected: the child's host tier starts as seeded random bytes
        host0 = torch.empty(2 * n * g.page_bytes, dtype=torch.uint8)
        wl.fill_random_(host0, host_seed)
        want_pool = snap[0].copy()
        want_host = host0.numpy().copy()
        og = oracle_geom(g)
        oracle.backup(og, want_pool, want_host, ids.backup_src, ids.backup_slots,
                      pool_offset=w.pool_offset, threads=8)
        oracle.restore(og, want_pool, want_host, ids.restore_slots, ids.restore_dst,
                       pool_offset=w.pool_offset, threads=8)
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        with tempfile.TemporaryDirectory() as td:
            out = os.path.join(td, "host.npy")
            geom_kw = dict(L=g.L, C=g.C, P=g.P, T=g.T, H=g.H, B=g.B, order=g.order,
                           dev_heads=g.dev_heads, host_heads=g.host_heads)
            ids_d = {k: np.asarray(v) for k, v in vars(ids).items()}
            p = ctx.Process(target=_child_drive,
                            args=(kvb.desc_to_bytes(desc), geom_kw, ids_d, 2 * n, host_seed, out, q))
            p.start()
            status = q.get(timeout=600)
            p.join(timeout=120)
            assert status[0] == "ok", status
            got_host = np.load(out)
        assert np.array_equal(got_host, want_host), "importer's host tier differs from the oracle"
        got = rig.snapshot()[0]
        assert np.array_equal(got, want_pool), "pool differs from the oracle"
    finally:
        kvb.kv_pool_close(pool)


def _child_export(q, done, P, seed):
    """Exporter that allocates, fills, exports, and exits when told to."""
    import sys
    sys.path[:0] = [ROOT]
    import torch as t
    from hierarchical_kv_cache_backup_gb300 import kvb as k
    from hierarchical_kv_cache_backup_gb300 import workloads as w

    g = w.TINY.geom.with_(P=P)
    alloc = t.empty(g.pool_bytes + 4096, dtype=t.uint8, device="cuda")
    w.fill_random_(alloc, seed)
    t.cuda.synchronize()
    lay = k.make_layout(g.L, g.C, g.P, g.T, g.H, g.B)
    pool = k.kv_pool_register(lay, alloc.data_ptr(), 4096 - 48 * 2, instance_id=99, generation=5)
    q.put(k.desc_to_bytes(k.kv_pool_export(pool)))
    done.wait(300)
    k.kv_pool_close(pool)


def test_exporter_exit_keeps_mapping_alive_and_generations():
    ctx = mp.get_context("spawn")
    q, done = ctx.Queue(), ctx.Event()
    P, seed = 64, 2024
    p = ctx.Process(target=_child_export, args=(q, done, P, seed))
    p.start()
    desc = kvb.desc_from_bytes(q.get(timeout=300))
    pool = kvb.kv_pool_import(desc)
    done.set()
    p.join(timeout=120)
    assert p.exitcode == 0
    try:
        # the exporter is gone; the mapping still holds its memory (seeded content)
        g = wl.TINY.geom.with_(P=P)
        expect = torch.empty(g.pool_bytes + 4096, dtype=torch.uint8, device="cuda")
        wl.fill_random_(expect, seed)
        host = torch.zeros(4 * g.page_bytes, dtype=torch.uint8, pin_memory=True)
        lay, _, _ = kvb.kv_pool_info(pool)
        tier = kvb.kv_host_register(host.data_ptr(), host.numel(), 4, 0, lay)
        f = kvb.kv_backup(pool, tier, [0, 17, 63, 5], [3, 2, 1, 0])
        kvb.kv_fence_wait(f, 30_000_000_000)
        want = np.zeros(host.numel(), dtype=np.uint8)
        oracle.backup(oracle_geom(g), expect.cpu().numpy(), want, [0, 17, 63, 5], [3, 2, 1, 0],
                      pool_offset=desc.alloc_offset)
        assert np.array_equal(host.numpy(), want)
        kvb.kv_host_close(tier)
        # a descriptor whose extent overruns the mapped allocation is refused, and
        # the mapping the live pool holds is unaffected
        far = kvb.desc_from_bytes(kvb.desc_to_bytes(desc))
        far.alloc_offset = 1 << 40
        big = kvb.desc_from_bytes(kvb.desc_to_bytes(desc))
        big.layout.num_pages = 1 << 20
        big.nbytes = (1 << 20) * g.page_bytes
        for bad in (far, big):
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_pool_import(bad)
            assert e.value.status == kvb.KV_ERR_OUT_OF_RANGE, kvb.kv_last_error()
        host.zero_()
        tier = kvb.kv_host_register(host.data_ptr(), host.numel(), 4, 0, lay)
        kvb.kv_fence_wait(kvb.kv_backup(pool, tier, [0, 17, 63, 5], [3, 2, 1, 0]), 30_000_000_000)
        assert np.array_equal(host.numpy(), want)
        kvb.kv_host_close(tier)
        # a newer generation of the same instance retires this one
        kvb.kv_pool_retire(99, 6)
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_import(desc)
        assert e.value.status == kvb.KV_ERR_STALE
    finally:
        kvb.kv_pool_close(pool)


def test_import_in_own_process_is_refused_cleanly():
    g = wl.TINY.geom
    t = torch.empty(g.pool_bytes, dtype=torch.uint8, device="cuda")
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B)
    pool = kvb.kv_pool_register(lay, t.data_ptr(), 0)
    try:
        desc = kvb.kv_pool_export(pool)
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_import(desc)
        assert e.value.status == kvb.KV_ERR_CUDA
        bad = kvb.desc_from_bytes(kvb.desc_to_bytes(desc))
        bad.device_uuid[0] ^= 0xFF
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_import(bad)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    finally:
        kvb.kv_pool_close(pool)


def _child_drive_split(desc_bytes, bufs_bytes, geom_kw, ids, host_slots, host_seed, out_path, q):
    """Importer of a split pool: maps every allocation once (imported twice to share
    the mappings), backs pages up on one stream while restoring others on another,
    then saves its host tier."""
    try:
        import sys
        sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]
        import torch as t
        from hierarchical_kv_cache_backup_gb300 import kvb as k
        from hierarchical_kv_cache_backup_gb300 import workloads as w

        g = w.Geometry(**geom_kw)
        desc = k.desc_from_bytes(desc_bytes)
        bufs = k.bufs_from_bytes(bufs_bytes)
        try:
            k.kv_pool_import(desc)
            raise AssertionError("a split descriptor was accepted by kv_pool_import")
        except k.KvError as e:
            assert e.status == k.KV_ERR_INVALID_ARG
        pool = k.kv_pool_import_split(desc, bufs)
        pool2 = k.kv_pool_import_split(desc, bufs)      # shares every mapping
        lay, _, nbytes = k.kv_pool_info(pool)
        host = t.empty(host_slots * g.page_bytes, dtype=t.uint8, pin_memory=True)
        w.fill_random_(host, host_seed)
        tier = k.kv_host_register(host.data_ptr(), host.numel(), host_slots, g.host_heads, lay)
        sa, sb = t.cuda.Stream(), t.cuda.Stream()
        fa = k.kv_backup(pool, tier, ids["backup_src"], ids["backup_slots"], sa.cuda_stream)
        fb = k.kv_restore(pool2, tier, ids["restore_slots"], ids["restore_dst"], -1,
                          sb.cuda_stream)
        k.kv_fence_wait(fa, 30_000_000_000)
        k.kv_fence_wait(fb, 30_000_000_000)
        k.kv_pool_close(pool2)
        # the first handle still maps every buffer after the second is closed: one layer
        f = k.kv_restore(pool, tier, ids["restore_slots"][:2], ids["backup_src"][:2], g.L - 1)
        k.kv_fence_wait(f, 30_000_000_000)
        # an entry whose offset overruns its allocation is refused, the live pool unharmed
        far = k.bufs_from_bytes(bufs_bytes)
        far[1].alloc_offset = 1 << 40
        try:
            k.kv_pool_import_split(desc, far)
            raise AssertionError("an overrunning buffer entry was accepted")
        except k.KvError as e:
            assert e.status == k.KV_ERR_OUT_OF_RANGE
        k.kv_pool_close(pool)
        k.kv_host_close(tier)
        np.save(out_path, host.numpy())
        q.put(("ok", nbytes, len(bufs)))
    except Exception as e:  # reported to the parent
        q.put(("error", repr(e), 0))


def test_split_pool_import_in_second_process():
    """A layer-first pool held as one buffer per (layer, K/V) -- four of them slices
    of one allocation at odd offsets, the rest tensors of their own -- exported
    with one handle per allocation and driven by a second process; the pool's
    buffers and the importer's host tier against the oracle, which sees the
    buffers as the contiguous pool they form."""
    g = wl.Geometry(L=4, C=2, P=48, T=16, H=8, B=256, order=wl.LAYER_FIRST, dev_heads=wl.NHD,
                    host_heads=wl.NHD)
    nb = g.L * g.C
    buf_bytes = g.P * g.T * g.H * g.B
    shared = torch.full((4 * buf_bytes + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    views = [shared[48 + k * (buf_bytes + 16):48 + k * (buf_bytes + 16) + buf_bytes]
             for k in range(4)]
    own = [torch.empty(buf_bytes, dtype=torch.uint8, device="cuda") for _ in range(nb - 4)]
    buffers = views + own
    for k, b in enumerate(buffers):
        wl.fill_random_(b, 6100 + k)
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    pool = kvb.kv_pool_register_split(lay, [b.data_ptr() for b in buffers], instance_id=12,
                                      generation=3)
    try:
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_export(pool)
        assert e.value.status == kvb.KV_ERR_LAYOUT
        desc, bufs = kvb.kv_pool_export_split(pool)
        assert desc.magic == kvb.KVB_IPC_MAGIC_SPLIT and desc.nbytes == nb * buf_bytes
        handles = [bytes(b.handle) for b in bufs]
        assert len(set(handles[:4])) == 1                # slices of one allocation share a handle
        assert [b.alloc_offset % 16 for b in bufs] == [0] * nb
        assert bufs[1].alloc_offset - bufs[0].alloc_offset == buf_bytes + 16
        n, S = 12, 24
        r = np.random.default_rng(6200)
        perm = r.permutation(g.P).astype(np.int32)
        ids = {"backup_src": perm[:n], "backup_slots": np.arange(n, dtype=np.int32),
               "restore_slots": np.arange(n, 2 * n, dtype=np.int32), "restore_dst": perm[n:2 * n]}
        torch.cuda.synchronize()
        contiguous = np.concatenate([b.cpu().numpy() for b in buffers])
        host_seed = 6300
        host0 = torch.empty(S * g.page_bytes, dtype=torch.uint8)
        wl.fill_random_(host0, host_seed)
        want_pool, want_host = contiguous.copy(), host0.numpy().copy()
        og = oracle_geom(g)
        oracle.backup(og, want_pool, want_host, ids["backup_src"], ids["backup_slots"])
        oracle.restore(og, want_pool, want_host, ids["restore_slots"], ids["restore_dst"])
        oracle.restore(og, want_pool, want_host, ids["restore_slots"][:2], ids["backup_src"][:2],
                       layer=g.L - 1)
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        with tempfile.TemporaryDirectory() as td:
            out = os.path.join(td, "host.npy")
            geom_kw = dict(L=g.L, C=g.C, P=g.P, T=g.T, H=g.H, B=g.B, order=g.order,
                           dev_heads=g.dev_heads, host_heads=g.host_heads)
            p = ctx.Process(target=_child_drive_split,
                            args=(kvb.desc_to_bytes(desc), kvb.bufs_to_bytes(bufs), geom_kw, ids,
                                  S, host_seed, out, q))
            p.start()
            status = q.get(timeout=600)
            p.join(timeout=120)
            assert status[0] == "ok", status
            assert status[1:] == (nb * buf_bytes, nb)
            got_host = np.load(out)
        assert np.array_equal(got_host, want_host), "importer's host tier differs from the oracle"
        torch.cuda.synchronize()
        for k, b in enumerate(buffers):
            assert np.array_equal(b.cpu().numpy(), want_pool[k * buf_bytes:(k + 1) * buf_bytes]), \
                f"layer buffer {k} differs from the oracle"
        # bytes of the shared allocation around the four slices are untouched
        outside = np.ones(shared.numel(), dtype=bool)
        for k in range(4):
            outside[48 + k * (buf_bytes + 16):48 + k * (buf_bytes + 16) + buf_bytes] = False
        assert (shared.cpu().numpy()[outside] == 0xA5).all()
    finally:
        kvb.kv_pool_close(pool)
