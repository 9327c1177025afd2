"""Layer-first pools held in one device buffer per (layer, component), the way a
serving engine keeps per-layer K and V buffers: every path against the CPU
oracle run on the contiguous layer-first equivalent (the same bytes, cut at
every (layer, component))."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from gpu_rig import oracle_geom  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402


class SplitRig:
    def __init__(self, g, slots, seed):
        self.g = g
        per = g.P * g.layer_page_bytes // g.C          # one (layer, component) buffer
        self.per = per
        self.bufs = []
        for i in range(g.L * g.C):
            t = torch.empty(per + 64, dtype=torch.uint8, device="cuda")[32:32 + per]
            wl.fill_random_(t, seed + i)
            self.bufs.append(t)
        self.host = torch.empty(slots * g.page_bytes, dtype=torch.uint8, pin_memory=True)
        wl.fill_random_(self.host, seed + 999)
        self.layout = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, 0, g.dev_heads, g.elem_bytes)
        self.pool = kvb.kv_pool_register_split(self.layout, [b.data_ptr() for b in self.bufs])
        self.tier = kvb.kv_host_register(self.host.data_ptr(), self.host.numel(), slots,
                                         g.host_heads, self.layout)

    def contiguous(self):
        torch.cuda.synchronize()
        return np.concatenate([b.cpu().numpy() for b in self.bufs])   # [L][C][P][...] order

    def assert_pool(self, want):
        got = self.contiguous()
        assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"

    def close(self):
        kvb.kv_pool_close(self.pool)
        kvb.kv_host_close(self.tier)


@pytest.mark.parametrize("heads", [(wl.NHD, wl.NHD), (wl.HND, wl.NHD)], ids=["NHD", "HND-to-NHD"])
@pytest.mark.parametrize("mode", [kvb.KV_MODE_ZERO_COPY, kvb.KV_MODE_STAGED,
                                  kvb.KV_MODE_COPY_ENGINE], ids=["zc", "staged", "copy_engine"])
def test_split_pool_backup_restore(heads, mode):
    g = wl.LLAMA8B.geom.with_(P=40, L=6, dev_heads=heads[0], host_heads=heads[1])
    og = oracle_geom(g)
    r = np.random.default_rng(4)
    old = kvb.kv_config_get()
    kvb.kv_config_set(mode, 0, 4 << 20)
    rig = SplitRig(g, 12, seed=50)
    try:
        pool0, host0 = rig.contiguous(), rig.host.numpy().copy()
        src = r.permutation(g.P)[:9]
        slots = r.permutation(12)[:9]
        host_want = host0.copy()
        oracle.backup(og, pool0, host_want, src, slots)
        kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.tier, src, slots), 30_000_000_000)
        assert np.array_equal(rig.host.numpy(), host_want)
        dst = r.permutation(g.P)[:9]
        pool_want = pool0.copy()
        oracle.restore(og, pool_want, host_want, slots, dst)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.tier, slots, dst), 30_000_000_000)
        rig.assert_pool(pool_want)
        oracle.restore(og, pool_want, host_want, slots[:3], src[:3], layer=4)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.tier, slots[:3], src[:3], 4),
                          30_000_000_000)
        rig.assert_pool(pool_want)
        # progressive restore of layers 1..5 and the device-side gather
        for l in range(1, 6):
            oracle.restore(og, pool_want, host_want, slots[3:], dst[3:], layer=l)
        f = kvb.kv_restore_layers(rig.pool, rig.tier, slots[3:], dst[3:], 1, 5)
        kvb.kv_fence_wait(f[-1], 30_000_000_000)
        rig.assert_pool(pool_want)
        buf = torch.empty(9 * g.page_bytes, dtype=torch.uint8, device="cuda")
        want_buf = np.zeros(9 * g.page_bytes, dtype=np.uint8)
        oracle.backup(og, pool_want, want_buf, dst, np.arange(9))
        kvb.kv_fence_wait(kvb.kv_device_gather(rig.pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                               dst), 30_000_000_000)
        assert np.array_equal(buf.cpu().numpy(), want_buf)
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_export(rig.pool)
        assert e.value.status == kvb.KV_ERR_LAYOUT
    finally:
        rig.close()
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)


def test_split_pool_checks_on_device():
    g = wl.TINY.geom
    per = g.P * g.layer_page_bytes // g.C
    bufs = [torch.empty(per, dtype=torch.uint8, device="cuda") for _ in range(g.L * g.C)]
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B)
    host = torch.empty(per, dtype=torch.uint8, pin_memory=True)
    ptrs = [b.data_ptr() for b in bufs]
    with pytest.raises(kvb.KvError) as e:                      # host memory is not a layer buffer
        kvb.kv_pool_register_split(lay, ptrs[:-1] + [host.data_ptr()])
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    p = kvb.kv_pool_register_split(lay, ptrs)
    lay2, ptr, nbytes = kvb.kv_pool_info(p)
    assert ptr == ptrs[0] and nbytes == g.pool_bytes
    kvb.kv_pool_close(p)


@pytest.mark.parametrize("heads", [(wl.NHD, wl.NHD), (wl.HND, wl.NHD)], ids=["NHD", "HND-to-NHD"])
def test_split_pool_overlapped_one_layer_restores(heads):
    """Every layer restored one per call with KV_CFG_OVERLAP_RESTORES on a split
    pool (each layer in its own buffers): all but the first overlapped, the
    layer buffers equal the oracle's pool."""
    g = wl.LLAMA8B.geom.with_(P=48, L=7, dev_heads=heads[0], host_heads=heads[1])
    og = oracle_geom(g)
    r = np.random.default_rng(6)
    old = kvb.kv_config_get()
    kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0, kvb.KV_CFG_OVERLAP_RESTORES)
    rig = SplitRig(g, 16, seed=60)
    s = torch.cuda.Stream()
    try:
        want = rig.contiguous()
        host_np = rig.host.numpy().copy()
        slots = r.permutation(16).astype(np.int32)
        dst = r.permutation(g.P)[:16].astype(np.int32)
        c0 = kvb.kv_overlap_count()
        fences = [kvb.kv_restore(rig.pool, rig.tier, slots, dst, l, s.cuda_stream)
                  for l in range(g.L)]
        assert kvb.kv_overlap_count() - c0 == g.L - 1
        kvb.kv_fence_wait(fences[-1], 30_000_000_000)
        for l in range(g.L):
            oracle.restore(og, want, host_np, slots, dst, layer=l)
        rig.assert_pool(want)
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        rig.close()
