"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (zero-copy mode, default grid shapes, one call per op through the C ABI).
Every check here compares the whole device allocation and the whole host tier
with the oracle, byte for byte (large buffers in 1 GiB slices with
np.array_equal, never a hash or a sum).

* Llama-8B: 8 GiB layer-first pool of 4,096 pages; 512 random pages backed up,
  then restored into 512 others.
* MLA fp8: 17.2 GiB pool of 2,048 pages; the 64-page prefix restored by 61
  one-layer calls, then by one progressive call into other pages (and once
  more with overlapped one-layer restores).
* Sweep extreme: 8,192 one-run pages of 1 MiB; 4,096 random pages backed up on
  one stream while 4,096 others are restored on another.
* HBM gather: the benchmark's 512 Llama-8B pages (identity chunks, the bulk
  kernel) and 512 TRT-LLM pages (HND pool -> NHD buffer, the transposing
  kernel) gathered into a device buffer in host layout, with and without a
  fence, compared with the oracle's backup into slots 0..511."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from gpu_rig import Rig, layout, oracle_geom  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

GIB = 1 << 30
WAIT_NS = 120_000_000_000


@pytest.fixture(autouse=True)
def default_config():
    old = kvb.kv_config_get()
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY)
    yield
    kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
    torch.cuda.empty_cache()


def to_host(t) -> np.ndarray:
    """A byte-exact host copy of a uint8 tensor, taken in 1 GiB slices."""
    torch.cuda.synchronize()
    out = np.empty(t.numel(), dtype=np.uint8)
    for lo in range(0, t.numel(), GIB):
        hi = min(t.numel(), lo + GIB)
        out[lo:hi] = t[lo:hi].cpu().numpy()
    return out


def assert_bytes_equal(t, want: np.ndarray, what: str):
    """Every byte of tensor t (device or pinned) equals `want`, compared in 1 GiB slices."""
    torch.cuda.synchronize()
    assert t.numel() == want.size, (what, t.numel(), want.size)
    for lo in range(0, t.numel(), GIB):
        hi = min(t.numel(), lo + GIB)
        got = t[lo:hi].cpu().numpy()
        ref = want[lo:hi]
        if not np.array_equal(got, ref):
            bad = np.flatnonzero(got != ref)
            raise AssertionError(f"{what}: {bad.size} bytes differ in [{lo}, {hi}), first at "
                                 f"{lo + bad[0]} (got {got[bad[0]]}, want {ref[bad[0]]})")


def test_llama8b_full_size_against_the_oracle():
    w = wl.LLAMA8B
    g = w.geom
    ids = wl.op_ids(w)
    rig = Rig(g, w.host_slots, seed=w.seed)
    s = torch.cuda.Stream()
    try:
        snap = rig.snapshot()
        want = rig.expect_backup(snap, ids.backup_src, ids.backup_slots, threads=16)
        kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.hostt, ids.backup_src, ids.backup_slots,
                                        s.cuda_stream), WAIT_NS)
        rig.assert_equal(want)
        want = rig.expect_restore(want, ids.restore_slots, ids.restore_dst, threads=16)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.hostt, ids.restore_slots,
                                         ids.restore_dst, -1, s.cuda_stream), WAIT_NS)
        rig.assert_equal(want)
    finally:
        rig.close()


def test_mla_full_size_layerwise_and_progressive():
    """The 17.2 GiB MLA pool: 61 one-layer restores of the 64-page prefix (the
    benchmark's step), then one progressive restore of every layer into 64 other
    pages, then 61 one-layer restores with overlap allowed into a third page set;
    after each, the whole allocation and the whole host tier equal the oracle's."""
    w = wl.MLA_FP8
    g = w.geom
    og = oracle_geom(g)
    ids = wl.op_ids(w)
    r = np.random.default_rng(w.seed + 9)
    alloc = torch.empty(g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    host = torch.empty(w.host_slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    wl.fill_random_(host, w.seed + 1)
    lay = layout(g)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), 0)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), w.host_slots, g.host_heads, lay)
    s = torch.cuda.Stream()
    old = kvb.kv_config_get()
    try:
        want = to_host(alloc)                 # the pool before any restore
        host_np = host.numpy().copy()         # restores never write the host tier
        dst2 = wl.distinct_pages(r, g.P, w.n, exclude=ids.restore_dst)
        dst3 = wl.distinct_pages(r, g.P, w.n, exclude=np.concatenate([ids.restore_dst, dst2]))

        f = None
        for layer in range(g.L):              # the benchmark's step: 61 one-layer calls
            f = kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, layer,
                               s.cuda_stream)
            oracle.restore(og, want, host_np, ids.restore_slots, ids.restore_dst, layer=layer)
        kvb.kv_fence_wait(f, WAIT_NS)
        assert_bytes_equal(alloc, want, "pool after 61 one-layer restores")
        assert_bytes_equal(host, host_np, "host tier after 61 one-layer restores")

        fences = kvb.kv_restore_layers(pool, tier, ids.restore_slots, dst2, 0, g.L,
                                       s.cuda_stream)
        for fc in fences:                     # raises unless every layer completed
            kvb.kv_fence_wait(fc, WAIT_NS)
        for layer in range(g.L):
            oracle.restore(og, want, host_np, ids.restore_slots, dst2, layer=layer)
        assert_bytes_equal(alloc, want, "pool after the progressive restore")
        assert_bytes_equal(host, host_np, "host tier after the progressive restore")

        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes,
                          old.flags | kvb.KV_CFG_OVERLAP_RESTORES, old.cta_threads)
        fences = [kvb.kv_restore(pool, tier, ids.restore_slots, dst3, layer, s.cuda_stream)
                  for layer in range(g.L)]
        kvb.kv_fence_wait(fences[-1], WAIT_NS)
        for fc in fences:                     # in call order: the last implies every other
            assert kvb.kv_fence_query(fc) == kvb.KV_OK
        for layer in range(g.L):
            oracle.restore(og, want, host_np, ids.restore_slots, dst3, layer=layer)
        assert_bytes_equal(alloc, want, "pool after 61 overlapped one-layer restores")
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
        del alloc


def test_sweep_extreme_full_size_concurrent():
    """8,192 pages of 1 MiB: 4,096 backed up on one stream while 4,096 others are
    restored on another; the whole pool and tier equal the oracle's (the two ops
    touch disjoint pages and slots, so either order gives the same result)."""
    pb, P, n = 1 << 20, 8192, 4096
    g = wl.Geometry(L=1, C=1, P=P, T=1, H=1, B=pb, elem_bytes=1)
    og = oracle_geom(g)
    r = np.random.default_rng(1004)
    alloc = torch.empty(P * pb, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, 4004)
    S = 2 * n
    host = torch.empty(S * pb, dtype=torch.uint8, pin_memory=True)
    wl.fill_random_(host, 4005)
    lay = layout(g)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), 0)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), S, 0, lay)
    src = wl.distinct_pages(r, P, n)
    dst = wl.distinct_pages(r, P, n, exclude=src)
    slots_b = np.arange(n, dtype=np.int32)
    slots_r = np.arange(n, S, dtype=np.int32)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        want_pool = to_host(alloc)
        torch.cuda.synchronize()
        want_host = host.numpy().copy()
        oracle.backup(og, want_pool, want_host, src, slots_b, threads=16)
        oracle.restore(og, want_pool, want_host, slots_r, dst, threads=16)
        torch.cuda.synchronize()
        ev = torch.cuda.Event()
        ev.record(sa)
        sb.wait_event(ev)
        fa = kvb.kv_backup(pool, tier, src, slots_b, sa.cuda_stream)
        fb = kvb.kv_restore(pool, tier, slots_r, dst, -1, sb.cuda_stream)
        kvb.kv_fence_wait(fa, WAIT_NS)
        kvb.kv_fence_wait(fb, WAIT_NS)
        assert_bytes_equal(alloc, want_pool, "pool after backup || restore")
        assert_bytes_equal(host, want_host, "host tier after backup || restore")
    finally:
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
        del alloc


@pytest.mark.parametrize("wname", ["llama8b", "trtllm_ipc"])
def test_hbm_gather_full_size_against_the_oracle(wname):
    """kv_device_gather of the benchmark's 512 pages (Llama-8B: 1 GiB through the
    bulk kernel; TRT-LLM: 2.5 GiB, HND pool -> NHD buffer, through the
    transposing kernel), with a fence and in stream order only, equals the
    oracle's backup of those pages into slots 0..511; the pool is unchanged."""
    w = {x.name: x for x in wl.WORKLOADS}[wname]
    g = w.geom
    og = oracle_geom(g)
    n = w.n
    alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    pool = kvb.kv_pool_register(layout(g), alloc.data_ptr(), w.pool_offset)
    buf = torch.empty(n * g.page_bytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    try:
        pool_np = to_host(alloc)
        for k, with_fence in enumerate((True, False)):
            src = wl.op_ids(w, seed=w.seed + 17 * k + 1).backup_src   # the bench's id sets
            want = np.zeros(n * g.page_bytes, dtype=np.uint8)
            oracle.backup(og, pool_np, want, src, np.arange(n, dtype=np.int32),
                          pool_offset=w.pool_offset, threads=16)
            buf.fill_(0x5A)
            torch.cuda.synchronize()
            f = kvb.kv_device_gather(pool, buf.data_ptr(), buf.numel(), g.host_heads, src,
                                     s.cuda_stream, fence=with_fence)
            if with_fence:
                kvb.kv_fence_wait(f, WAIT_NS)
            s.synchronize()
            assert_bytes_equal(buf, want, f"{wname} gather (fence={with_fence})")
        assert_bytes_equal(alloc, pool_np, f"{wname} pool after the gathers")
    finally:
        kvb.kv_pool_close(pool)
        del alloc, buf
