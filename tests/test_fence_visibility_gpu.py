"""Fence visibility: once a fence reports an op complete, every byte the op
wrote is visible to whoever observed the fence -- the host thread that waited
on (or polled) it, reading the pinned host tier with no CUDA call in between,
and a copy on another stream ordered after the op only by kv_fence_stream_wait.

The fused completion orders each CTA's stores at device scope and publishes
the fence with one system-scope release store; the copy-engine modes publish
it with a marker kernel after their copies; overlapped ops (the overlap flags)
publish in call order after waiting for their predecessor's fence.  Every
round below rewrites the source with a new value, so a byte left over from the
previous round, or one still in flight when the fence was seen, shows up as a
mismatch against the oracle (RFC "[HiCache] Out-of-process HiCache data
plane", §Device IPC data path: the completion handle says the copy has
landed)."""
import time

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

ROUNDS = 400
WAIT_NS = 30_000_000_000
MODES = {"zero_copy": kvb.KV_MODE_ZERO_COPY, "staged": kvb.KV_MODE_STAGED,
         "copy_engine": kvb.KV_MODE_COPY_ENGINE}
STAGING = 2 << 20      # the smallest: a 4 MiB STAGED op runs as 8 ping-pong chunks of 512 KiB
# 128 pages of 32 KiB (4 MiB): every CTA of the default grid takes segments
GEOMS = {
    "layer_first_nhd": wl.Geometry(L=2, C=2, P=128, T=16, H=4, B=128),
    "page_first_hnd": wl.Geometry(L=2, C=2, P=128, T=16, H=4, B=128, order=wl.PAGE_FIRST,
                                  dev_heads=wl.HND),
}


def _mismatch(name, got, want):
    bad = np.flatnonzero(got != want)
    return (f"{name}: {bad.size} bytes differ, first at {bad[0]} (got {got[bad[0]]}, "
            f"want {want[bad[0]]})")


@pytest.fixture
def mode_config():
    old = kvb.kv_config_get()
    yield
    kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)


@pytest.mark.parametrize("geom", sorted(GEOMS))
@pytest.mark.parametrize("mode", sorted(MODES))
def test_backup_bytes_are_on_the_host_when_its_fence_is(geom, mode, mode_config):
    g = GEOMS[geom]
    rig = Rig(g, g.P, pool_offset=4096 + 48, seed=301)
    try:
        kvb.kv_config_set(MODES[mode], 0, STAGING)
        alloc0, _ = rig.snapshot()
        off, nb = rig.offset, g.pool_bytes
        base = rig.alloc[off:off + nb].clone()
        base_np = alloc0[off:off + nb].copy()
        host_view = rig.host.numpy()          # the pinned tier itself, no copy
        r = np.random.default_rng(302)
        s = torch.cuda.Stream()
        og = oracle_geom(g)
        for k in range(ROUNDS):
            v = k % 255 + 1                    # a new, nonzero offset every round
            src = r.permutation(g.P).astype(np.int32)
            slots = r.permutation(g.P).astype(np.int32)
            with torch.cuda.stream(s):
                torch.add(base, v, out=rig.alloc[off:off + nb])   # wraps mod 256
            f = kvb.kv_backup(rig.pool, rig.hostt, src, slots, s.cuda_stream)
            if k % 2 == 0:
                kvb.kv_fence_wait(f, WAIT_NS)
            else:                              # poll instead of waiting
                deadline = time.monotonic() + WAIT_NS / 1e9
                while kvb.kv_fence_query(f) == kvb.KV_ERR_TIMEOUT:
                    assert time.monotonic() < deadline, f"round {k}: fence never completed"
                assert kvb.kv_fence_query(f) == kvb.KV_OK
            got = host_view.copy()             # read right after the fence, nothing synced
            pool_k = alloc0.copy()
            pool_k[off:off + nb] = base_np + np.uint8(v)
            want = np.zeros_like(got)
            oracle.backup(og, pool_k, want, src, slots, pool_offset=off, threads=4)
            assert np.array_equal(got, want), f"round {k}: " + _mismatch("host tier", got, want)
        torch.cuda.synchronize()
    finally:
        rig.close()


@pytest.mark.parametrize("geom", sorted(GEOMS))
@pytest.mark.parametrize("mode", sorted(MODES))
def test_restored_pages_are_seen_by_a_stream_that_waits_on_the_fence(geom, mode, mode_config):
    g = GEOMS[geom]
    rig = Rig(g, g.P, pool_offset=4096 + 48, seed=311)
    try:
        kvb.kv_config_set(MODES[mode], 0, STAGING)
        alloc_np, host0 = rig.snapshot()
        host_view = rig.host.numpy()
        out = torch.empty(rig.alloc.numel(), dtype=torch.uint8, pin_memory=True)
        r = np.random.default_rng(312)
        s, c = torch.cuda.Stream(), torch.cuda.Stream()
        og = oracle_geom(g)
        for k in range(ROUNDS):
            host_view[:] = host0 + np.uint8(k % 255 + 1)   # the host rewrites its tier
            slots = r.permutation(g.P).astype(np.int32)
            dst = r.permutation(g.P).astype(np.int32)
            f = kvb.kv_restore(rig.pool, rig.hostt, slots, dst, -1, s.cuda_stream)
            kvb.kv_fence_stream_wait(f, c.cuda_stream)
            with torch.cuda.stream(c):
                out.copy_(rig.alloc, non_blocking=True)   # ordered after the op by the fence only
            c.synchronize()
            oracle.restore(og, alloc_np, host_view, slots, dst, pool_offset=rig.offset, threads=4)
            got = out.numpy()
            assert np.array_equal(got, alloc_np), f"round {k}: " + _mismatch("pool", got,
                                                                             alloc_np)
            s.synchronize()                    # before the host rewrites what the op read
        torch.cuda.synchronize()
    finally:
        rig.close()


def test_overlapped_backups_are_on_the_host_in_fence_order(mode_config):
    """KV_CFG_OVERLAP_BACKUPS: four backups into disjoint slots run overlapped;
    once fence i completes, the slots of backups 0..i hold the oracle's bytes
    (fences complete in call order).  The pool is rewritten on another stream,
    synchronised before the round's calls, as the flag's contract asks."""
    g = GEOMS["layer_first_nhd"]
    rig = Rig(g, g.P, pool_offset=4096 + 48, seed=321)
    try:
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0, kvb.KV_CFG_OVERLAP_BACKUPS)
        alloc0, _ = rig.snapshot()
        off, nb, pb = rig.offset, g.pool_bytes, g.page_bytes
        base = rig.alloc[off:off + nb].clone()
        base_np = alloc0[off:off + nb].copy()
        host_view = rig.host.numpy()
        r = np.random.default_rng(322)
        s, w = torch.cuda.Stream(), torch.cuda.Stream()
        og = oracle_geom(g)
        groups = 4
        m = g.P // groups
        c0 = kvb.kv_overlap_count()
        for k in range(ROUNDS // 4):
            v = k % 255 + 1
            with torch.cuda.stream(w):
                torch.add(base, v, out=rig.alloc[off:off + nb])
            w.synchronize()
            pages = r.permutation(g.P).astype(np.int32)
            slots = r.permutation(g.P).astype(np.int32)
            fences = [kvb.kv_backup(rig.pool, rig.hostt, pages[i * m:(i + 1) * m],
                                    slots[i * m:(i + 1) * m], s.cuda_stream)
                      for i in range(groups)]
            pool_k = alloc0.copy()
            pool_k[off:off + nb] = base_np + np.uint8(v)
            want = np.zeros_like(host_view)
            oracle.backup(og, pool_k, want, pages, slots, pool_offset=off, threads=4)
            for i, f in enumerate(fences):
                kvb.kv_fence_wait(f, WAIT_NS)
                got = host_view.copy()
                for sl in slots[:(i + 1) * m]:
                    a, b = int(sl) * pb, (int(sl) + 1) * pb
                    assert np.array_equal(got[a:b], want[a:b]), (
                        f"round {k}, fence {i}: " + _mismatch(f"slot {sl}", got[a:b], want[a:b]))
        assert kvb.kv_overlap_count() - c0 >= (ROUNDS // 4) * (groups - 1)
        torch.cuda.synchronize()
    finally:
        rig.close()


def test_overlapped_one_layer_restores_are_seen_layer_by_layer(mode_config):
    """KV_CFG_OVERLAP_RESTORES: one-layer restores of every layer run overlapped;
    after layer l's fence -- waited on by a second stream on the GPU (even l) or
    by the host before it issues the copy (odd l) -- layers 0..l of the pool
    hold the oracle's bytes while later layers may still be moving."""
    g = wl.Geometry(L=8, C=2, P=64, T=16, H=2, B=128)
    rig = Rig(g, g.P, seed=331)
    try:
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0, kvb.KV_CFG_OVERLAP_RESTORES)
        alloc_np, host0 = rig.snapshot()
        host_view = rig.host.numpy()
        outs = [torch.empty(rig.alloc.numel(), dtype=torch.uint8, pin_memory=True)
                for _ in range(g.L)]
        r = np.random.default_rng(332)
        s, c = torch.cuda.Stream(), torch.cuda.Stream()
        og = oracle_geom(g)
        layer_block = g.P * g.layer_page_bytes     # one layer of every page (layer-first)
        c0 = kvb.kv_overlap_count()
        rounds = ROUNDS // 8
        for k in range(rounds):
            host_view[:] = host0 + np.uint8(k % 255 + 1)
            slots = r.permutation(g.P).astype(np.int32)
            dst = r.permutation(g.P).astype(np.int32)
            fences = [kvb.kv_restore(rig.pool, rig.hostt, slots, dst, l, s.cuda_stream)
                      for l in range(g.L)]
            for l, f in enumerate(fences):
                if l % 2 == 0:
                    kvb.kv_fence_stream_wait(f, c.cuda_stream)
                else:
                    kvb.kv_fence_wait(f, WAIT_NS)
                with torch.cuda.stream(c):
                    outs[l].copy_(rig.alloc, non_blocking=True)
            c.synchronize()
            for l in range(g.L):
                oracle.restore(og, alloc_np, host_view, slots, dst, layer=l, threads=4)
                got = outs[l].numpy()
                for lp in range(l + 1):                # layers whose fences precede l's
                    a, b = lp * layer_block, (lp + 1) * layer_block
                    assert np.array_equal(got[a:b], alloc_np[a:b]), (
                        f"round {k}, after layer {l}: " + _mismatch(f"layer {lp}", got[a:b],
                                                                    alloc_np[a:b]))
            s.synchronize()
        assert kvb.kv_overlap_count() - c0 >= rounds * (g.L - 1)
        torch.cuda.synchronize()
    finally:
        rig.close()
