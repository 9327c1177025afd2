"""Allocation-free staged backup: kv_backup_staged_noalloc against kv_backup and
against the CPU oracle.

Callers that cannot allocate GPU memory while backing pages up (an engine whose
allocator owns all of HBM, an out-of-memory or teardown path, a runtime that
forbids allocation calls while recording work) use kv_backup_staged_noalloc,
which stages through a fixed device array inside the library instead of a
cudaMalloc'd buffer.  Its host slots must hold exactly what kv_backup writes
for the same pages, call after call (the array is shared and reused), and the
whole host tier, untouched slots included, must equal the oracle's BACKUP
(RFC §Device IPC data path: BACKUP copies the named pages to the host tier).
This file sorts last so a stop-at-first-failure run has run every other test
first.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

LIMIT = 32 << 20   # KVB_NOALLOC_STAGING_BYTES


@pytest.mark.parametrize("wname", ["trtllm_ipc", "llama8b"])
def test_noalloc_backup_matches_kv_backup_and_the_oracle(wname):
    w = {x.name: x for x in wl.WORKLOADS}[wname]
    g = w.geom.with_(P=64)
    og = oracle.geom(g.L, g.C, g.P, g.T, g.H, g.B, page_first=g.order == wl.PAGE_FIRST,
                     dev_hnd=g.dev_heads == wl.HND, host_hnd=g.host_heads == wl.HND)
    max_n = LIMIT // g.page_bytes
    slots_total = 2 * max_n + 3            # three slots no call ever names
    alloc = torch.empty(w.pool_offset + g.pool_bytes, dtype=torch.uint8, device="cuda")
    wl.fill_random_(alloc, w.seed)
    host = torch.empty(slots_total * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    wl.fill_random_(host, w.seed + 1)
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    pool = kvb.kv_pool_register(lay, alloc.data_ptr(), w.pool_offset)
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), slots_total, g.host_heads, lay)
    stream = torch.cuda.Stream()
    r = np.random.default_rng(w.seed)
    try:
        torch.cuda.synchronize()
        pool_np = alloc.cpu().numpy()
        want = host.numpy().copy()
        for n in (max_n, max(1, max_n - 2)):          # two calls in a row, the first at the limit
            src = r.permutation(g.P)[:n].astype(np.int32)
            ref_slots = r.permutation(max_n)[:n].astype(np.int32)       # kv_backup -> [0, max_n)
            new_slots = (max_n + r.permutation(max_n)[:n]).astype(np.int32)  # no-alloc -> above
            kvb.kv_fence_wait(kvb.kv_backup(pool, tier, src, ref_slots), 30_000_000_000)
            kvb.kv_backup_staged_noalloc(pool, tier, src, new_slots, stream.cuda_stream)
            stream.synchronize()
            oracle.backup(og, pool_np, want, src, ref_slots, pool_offset=w.pool_offset)
            oracle.backup(og, pool_np, want, src, new_slots, pool_offset=w.pool_offset)
            view = host.view(slots_total, g.page_bytes)
            for a, b in zip(ref_slots, new_slots):    # the existing entry point's bytes
                assert torch.equal(view[a], view[b]), (wname, n, int(a), int(b))
            got = host.numpy()
            if not np.array_equal(got, want):         # the whole tier, untouched slots too
                bad = np.flatnonzero(got != want)
                raise AssertionError(f"{wname} n={n}: {bad.size} host bytes differ from the "
                                     f"oracle, first in slot {bad[0] // g.page_bytes}")
        assert np.array_equal(alloc.cpu().numpy(), pool_np)   # a backup never writes the pool
        # beyond the static array: refused with a clear error, nothing enqueued
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_backup_staged_noalloc(pool, tier, r.permutation(g.P)[:max_n + 1],
                                         np.arange(max_n + 1), stream.cuda_stream)
        assert e.value.status == kvb.KV_ERR_OUT_OF_RANGE
        assert "static staging area" in kvb.kv_last_error()
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_backup_staged_noalloc(pool, tier, [1, 2], [3, 3], stream.cuda_stream)
        assert e.value.status == kvb.KV_ERR_DUPLICATE
        stream.synchronize()
        assert np.array_equal(host.numpy(), want)   # the refused calls wrote nothing
    finally:
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
