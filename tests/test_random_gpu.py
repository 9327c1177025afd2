"""Seeded random parity: 200 cases (KVB_RANDOM_CASES; a run of 2,000 passed)
drawing a geometry (layers, components, tokens, heads, head bytes), a pool
layout and host head order, a byte offset,
an operation (backup, whole or one-layer restore, progressive restore, device
gather or scatter), ids and a transfer configuration (mode, staging size,
bulk copies off, CTA size).  Each case runs through the C ABI and is compared
byte for byte with the oracle over the whole pool allocation and host tier
(or the device buffer) -- corners the fixed cases do not reach: bulk segments
that end mid-chunk, transposed chunks of odd heads x tokens, staging buffers
that hold one layer, the register fallback."""
import os

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

CASES = int(os.environ.get("KVB_RANDOM_CASES", "200"))   # seeds 7000 .. 7000 + CASES


def draw(seed):
    r = np.random.default_rng(seed)
    L, C = int(r.integers(1, 6)), int(r.integers(1, 3))
    T, H = int(r.integers(1, 41)), int(r.integers(1, 13))
    B = 16 * int(r.integers(1, 21))
    P = int(r.integers(4, 70))
    order, dev, host = int(r.integers(2)), int(r.integers(2)), int(r.integers(2))
    g = wl.Geometry(L=L, C=C, P=P, T=T, H=H, B=B, order=order, dev_heads=dev, host_heads=host)
    offset = 16 * int(r.integers(0, 300))
    op = str(r.choice(["backup", "restore", "restore_layer", "restore_layers", "gather",
                       "scatter"]))
    mode = int(r.choice([kvb.KV_MODE_ZERO_COPY, kvb.KV_MODE_STAGED, kvb.KV_MODE_COPY_ENGINE]))
    flags = int(r.choice([0, kvb.KV_CFG_NO_BULK, kvb.KV_CFG_NO_PDL]))
    threads = int(r.choice([0, 256, 1024]))
    staging = (2 + int(r.integers(0, 7))) << 20
    return r, g, offset, op, mode, flags, threads, staging


@pytest.mark.parametrize("case", range(CASES))
def test_random_case_matches_the_oracle(case):
    r, g, offset, op, mode, flags, threads, staging = draw(7000 + case)
    if mode == kvb.KV_MODE_STAGED and g.L * g.C * g.T * g.H * g.B // g.L > staging // 4:
        mode = kvb.KV_MODE_ZERO_COPY                  # a layer must fit one staging buffer
    S = int(r.integers(1, g.P + 3))
    n = int(r.integers(0, min(g.P, S) + 1))
    src = r.integers(0, g.P, n).astype(np.int32)                 # sources may repeat
    slots = r.permutation(S)[:n].astype(np.int32)
    dst = r.permutation(g.P)[:n].astype(np.int32)
    layer = int(r.integers(0, g.L))
    old = kvb.kv_config_get()
    rig = Rig(g, S, pool_offset=offset, seed=8000 + case)
    og = oracle_geom(g)
    try:
        kvb.kv_config_set(mode, 0, staging, flags, threads)
        snap = rig.snapshot()
        if op == "backup":
            want = rig.expect_backup(snap, src, slots)
            kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.hostt, src, slots), 20_000_000_000)
            rig.assert_equal(want)
        elif op in ("restore", "restore_layer"):
            lay = layer if op == "restore_layer" else -1
            want = rig.expect_restore(snap, slots, dst, layer=lay)
            kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.hostt, slots, dst, lay),
                              20_000_000_000)
            rig.assert_equal(want)
        elif op == "restore_layers":
            first = int(r.integers(0, g.L))
            count = int(r.integers(1, g.L - first + 1))
            want = (snap[0].copy(), snap[1])
            for l in range(first, first + count):
                oracle.restore(og, want[0], snap[1], slots, dst, layer=l, pool_offset=offset)
            for f in kvb.kv_restore_layers(rig.pool, rig.hostt, slots, dst, first, count):
                kvb.kv_fence_wait(f, 20_000_000_000)
            rig.assert_equal(want)
        else:
            pb = g.page_bytes
            buf = torch.zeros(max(1, n) * pb + 64, dtype=torch.uint8, device="cuda")
            if op == "gather":
                want_buf = np.zeros(max(1, n) * pb, dtype=np.uint8)
                oracle.backup(og, snap[0], want_buf, src, np.arange(n), pool_offset=offset)
                with_fence = case % 2 == 0             # odd cases: stream order only
                f = kvb.kv_device_gather(rig.pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                         src, fence=with_fence)
                if with_fence:
                    kvb.kv_fence_wait(f, 20_000_000_000)
                torch.cuda.synchronize()
                assert np.array_equal(buf[:n * pb].cpu().numpy(), want_buf[:n * pb])
                rig.assert_equal(snap)
            else:
                data = r.integers(0, 256, max(1, n) * pb, dtype=np.uint8)
                buf[:data.size].copy_(torch.from_numpy(data))
                want = (snap[0].copy(), snap[1])
                oracle.restore(og, want[0], data, np.arange(n), dst, pool_offset=offset)
                with_fence = case % 2 == 0
                f = kvb.kv_device_scatter(rig.pool, buf.data_ptr(), buf.numel(), g.host_heads,
                                          dst, fence=with_fence)
                if with_fence:
                    kvb.kv_fence_wait(f, 20_000_000_000)
                rig.assert_equal(want)                 # (synchronizes the device)
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        rig.close()


@pytest.mark.parametrize("case", range(CASES // 2))
def test_random_split_pool_case_matches_the_oracle(case):
    """The same draws on a layer-first pool held as one device buffer per
    (layer, component): compared through the contiguous pool those buffers
    form ([L][C][P][T][H][B] cut at every (l, c))."""
    r, g, _, op, mode, flags, threads, staging = draw(9000 + case)
    g = wl.Geometry(L=g.L, C=g.C, P=g.P, T=g.T, H=g.H, B=g.B, order=wl.LAYER_FIRST,
                    dev_heads=g.dev_heads, host_heads=g.host_heads)
    if mode == kvb.KV_MODE_STAGED and g.C * g.T * g.H * g.B > staging // 4:
        mode = kvb.KV_MODE_ZERO_COPY
    S = int(r.integers(1, g.P + 3))
    n = int(r.integers(0, min(g.P, S) + 1))
    src = r.integers(0, g.P, n).astype(np.int32)
    slots = r.permutation(S)[:n].astype(np.int32)
    dst = r.permutation(g.P)[:n].astype(np.int32)
    layer = int(r.integers(0, g.L))
    chunk_bytes = g.P * g.T * g.H * g.B
    bufs = [torch.empty(chunk_bytes, dtype=torch.uint8, device="cuda") for _ in range(g.L * g.C)]
    for k, b in enumerate(bufs):
        wl.fill_random_(b, 9500 + 10 * case + k)
    host = torch.empty(S * g.page_bytes, dtype=torch.uint8, pin_memory=True)
    wl.fill_random_(host, 9400 + case)
    lay = kvb.make_layout(g.L, g.C, g.P, g.T, g.H, g.B, g.order, g.dev_heads, g.elem_bytes)
    old = kvb.kv_config_get()
    pool = kvb.kv_pool_register_split(lay, [b.data_ptr() for b in bufs])
    tier = kvb.kv_host_register(host.data_ptr(), host.numel(), S, g.host_heads, lay)
    og = oracle_geom(g)
    try:
        kvb.kv_config_set(mode, 0, staging, flags, threads)
        torch.cuda.synchronize()
        flat, hst = torch.cat(bufs).cpu().numpy(), host.numpy().copy()
        if op in ("backup", "gather"):
            if op == "backup":
                oracle.backup(og, flat, hst, src, slots)
                kvb.kv_fence_wait(kvb.kv_backup(pool, tier, src, slots), 20_000_000_000)
            else:
                buf = torch.zeros(max(1, n) * g.page_bytes, dtype=torch.uint8, device="cuda")
                want_buf = np.zeros(buf.numel(), dtype=np.uint8)
                oracle.backup(og, flat, want_buf, src, np.arange(n))
                kvb.kv_fence_wait(kvb.kv_device_gather(pool, buf.data_ptr(), buf.numel(),
                                                       g.host_heads, src), 20_000_000_000)
                torch.cuda.synchronize()
                assert np.array_equal(buf.cpu().numpy(), want_buf)
        elif op == "restore_layers":
            for l in range(g.L):
                oracle.restore(og, flat, hst, slots, dst, layer=l)
            for f in kvb.kv_restore_layers(pool, tier, slots, dst, 0, g.L):
                kvb.kv_fence_wait(f, 20_000_000_000)
        else:   # restore, restore_layer, scatter (as a one-layer restore from the tier)
            lay_ = layer if op != "restore" else -1
            oracle.restore(og, flat, hst, slots, dst, layer=lay_)
            kvb.kv_fence_wait(kvb.kv_restore(pool, tier, slots, dst, lay_), 20_000_000_000)
        torch.cuda.synchronize()
        assert np.array_equal(torch.cat(bufs).cpu().numpy(), flat), "split pool"
        assert np.array_equal(host.numpy(), hst), "host tier"
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        kvb.kv_pool_close(pool)
        kvb.kv_host_close(tier)
