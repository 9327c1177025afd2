"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (zero-copy mode, default grid shapes, one call per op through the C ABI).

* Llama-8B: 8 GiB layer-first pool of 4,096 pages; 512 random pages backed up,
  then restored into 512 others.  The oracle runs on the whole pool and host
  tier; every byte of both is compared.
* MLA fp8: 17.2 GiB pool of 2,048 pages; the 64-page prefix restored by 61
  one-layer calls, then by one progressive call into other pages.  Every
  restored chunk (page, layer) is compared with the host slot the oracle's
  address functions name for it, and sampled chunks of other pages must be
  unchanged.
* Sweep extreme: 8,192 one-run pages of 1 MiB; 4,096 random pages backed up on
  one stream while 4,096 others are restored on another.  Every page is
  compared (page-copy property: for L = C = T = H = 1 a unit is a page), and a
  sample is checked at the byte offsets the oracle computes."""
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


@pytest.fixture(autouse=True)
def default_config():
    old = kvb.kv_config_get()
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY)
    yield
    kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
    torch.cuda.empty_cache()


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
                                        s.cuda_stream), 60_000_000_000)
        rig.assert_equal(want)
        want = rig.expect_restore(want, ids.restore_slots, ids.restore_dst, threads=16)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.hostt, ids.restore_slots,
                                         ids.restore_dst, -1, s.cuda_stream), 60_000_000_000)
        rig.assert_equal(want)
    finally:
        rig.close()


def _mla_check(alloc, host_np, og, g, slots, dst, before, r, untouched):
    """Every (page, layer) chunk restored into dst[i] equals slot slots[i]'s
    chunk at the oracle's offsets; sampled other chunks are unchanged."""
    cb = g.T * g.H * g.B
    for i in range(len(dst)):
        for l in range(g.L):
            off = oracle.dev_offset(og, int(dst[i]), l, 0, 0, 0)
            hoff = oracle.host_offset(og, int(slots[i]), l, 0, 0, 0)
            got = alloc[off:off + cb].cpu().numpy()
            assert np.array_equal(got, host_np[hoff:hoff + cb]), ("restored chunk", i, l)
    # spot-check single units at the oracle's unit offsets (t, h inside a chunk)
    for _ in range(64):
        i, l, t = int(r.integers(len(dst))), int(r.integers(g.L)), int(r.integers(g.T))
        off = oracle.dev_offset(og, int(dst[i]), l, 0, t, 0)
        hoff = oracle.host_offset(og, int(slots[i]), l, 0, t, 0)
        assert np.array_equal(alloc[off:off + g.B].cpu().numpy(), host_np[hoff:hoff + g.B])
    for (p, l), want in zip(untouched, before):
        off = oracle.dev_offset(og, p, l, 0, 0, 0)
        assert np.array_equal(alloc[off:off + cb].cpu().numpy(), want), ("untouched", p, l)


def test_mla_full_size_layerwise_and_progressive():
    w = wl.MLA_FP8
    g = w.geom
    og = oracle_geom(g)
    ids = wl.op_ids(w)
    r = np.random.default_rng(w.seed + 9)
    alloc = torch.empty(g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    host = torch.empty(w.host_slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    wl.fill_random_(host, w.seed + 1)
    host_np = host.numpy()
    lay = layout(g)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), 0)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), w.host_slots, g.host_heads, lay)
    s = torch.cuda.Stream()
    try:
        dst2 = wl.distinct_pages(r, g.P, w.n, exclude=ids.restore_dst)
        written = set(ids.restore_dst.tolist()) | set(dst2.tolist())
        others = np.array([p for p in range(g.P) if p not in written])
        untouched = [(int(r.choice(others)), int(r.integers(g.L))) for _ in range(48)]
        cb = g.T * g.H * g.B
        torch.cuda.synchronize()
        before = [alloc[oracle.dev_offset(og, p, l, 0, 0, 0):][:cb].cpu().numpy().copy()
                  for p, l in untouched]
        f = None
        for layer in range(g.L):                  # the bench's step: 61 one-layer calls
            f = kvb.kv_restore(pool, tier, ids.restore_slots, ids.restore_dst, layer,
                               s.cuda_stream)
        kvb.kv_fence_wait(f, 60_000_000_000)
        _mla_check(alloc, host_np, og, g, ids.restore_slots, ids.restore_dst, before, r,
                   untouched)
        fences = kvb.kv_restore_layers(pool, tier, ids.restore_slots, dst2, 0, g.L,
                                       s.cuda_stream)
        for fc in fences:                         # raises unless every layer completed
            kvb.kv_fence_wait(fc, 60_000_000_000)
        _mla_check(alloc, host_np, og, g, ids.restore_slots, dst2, before, r, untouched)
    finally:
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
        del alloc


def test_sweep_extreme_full_size_concurrent():
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
        torch.cuda.synchronize()
        # 4,096 sources + 4,096 destinations cover all 8,192 pages here; any page
        # left over must stay unchanged
        keep = np.setdiff1d(np.arange(P), np.concatenate([src, dst]))
        sample_keep = r.choice(keep, min(16, keep.size), replace=False)
        keep_before = alloc.view(P, pb)[torch.as_tensor(sample_keep, device="cuda")].cpu()
        restore_src = host.view(S, pb)[torch.as_tensor(slots_r)].clone()   # before the ops
        fa = kvb.kv_backup(pool, tier, src, slots_b, sa.cuda_stream)
        fb = kvb.kv_restore(pool, tier, slots_r, dst, -1, sb.cuda_stream)
        kvb.kv_fence_wait(fa, 60_000_000_000)
        kvb.kv_fence_wait(fb, 60_000_000_000)
        torch.cuda.synchronize()
        # every page: host slot i == source page src[i]; page dst[i] == slot n + i's old bytes
        pages = alloc.view(P, pb)
        got_host = host.view(S, pb)[:n].to("cuda")
        assert torch.equal(got_host, pages[torch.as_tensor(src, device="cuda")]), "backup"
        assert torch.equal(pages[torch.as_tensor(dst, device="cuda")], restore_src.to("cuda")), \
            "restore"
        assert torch.equal(pages[torch.as_tensor(sample_keep, device="cuda")].cpu(), keep_before)
        # a sample at the oracle's byte offsets
        host_np = host.numpy()
        for i in r.choice(n, 24, replace=False):
            off = oracle.dev_offset(og, int(src[i]), 0, 0, 0, 0)
            hoff = oracle.host_offset(og, int(slots_b[i]), 0, 0, 0, 0)
            assert np.array_equal(alloc[off:off + pb].cpu().numpy(), host_np[hoff:hoff + pb])
            off = oracle.dev_offset(og, int(dst[i]), 0, 0, 0, 0)
            hoff = oracle.host_offset(og, int(slots_r[i]), 0, 0, 0, 0)
            assert np.array_equal(alloc[off:off + pb].cpu().numpy(), host_np[hoff:hoff + pb])
    finally:
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
        del alloc
