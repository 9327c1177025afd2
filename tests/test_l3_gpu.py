"""GPU pool -> host tier -> L3 record store -> host tier -> GPU pool, against
the same chain in the oracle.

Backup n pages into host slots, put those slots into records of a memfd,
scribble over the slots, get the records back into other slots, then restore
those slots into other pool pages (whole prefix, then one layer).  Every
intermediate state -- host tier, file image, pool allocation -- is compared
with the oracle's byte for byte."""
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


def file_bytes(fd, size):
    out = bytearray()
    while len(out) < size:
        chunk = os.pread(fd, size - len(out), len(out))
        if not chunk:
            break
        out += chunk
    return np.frombuffer(bytes(out), dtype=np.uint8)


@pytest.mark.parametrize("wname", ["llama8b", "trtllm_ipc", "mla_fp8"])
def test_backup_put_get_restore_chain(wname):
    w = {x.name: x for x in wl.WORKLOADS}[wname]
    g = w.geom.with_(P=48)
    S, R, n = 24, 40, 10
    pb = g.page_bytes
    r = np.random.default_rng(w.seed + 5)
    rig = Rig(g, S, pool_offset=w.pool_offset, seed=w.seed)
    fd = os.memfd_create("kvb_l3_chain")
    base = 4096
    image = r.integers(0, 256, base + R * pb, dtype=np.uint8)
    os.pwrite(fd, image.tobytes(), 0)
    store = kvb.kv_l3_open(fd, base, pb, R, 4)
    try:
        src = r.permutation(g.P)[:n].astype(np.int32)
        slots = r.permutation(S)[:n].astype(np.int32)
        snap = rig.snapshot()
        want = rig.expect_backup(snap, src, slots)
        kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.hostt, src, slots), 20_000_000_000)
        rig.assert_equal(want)

        records = r.permutation(R)[:n].astype(np.int32)
        kvb.kv_l3_put(store, rig.host.data_ptr(), S, slots, records)
        oracle.l3_put(want[1], pb, slots, records, image, base)
        assert np.array_equal(file_bytes(fd, image.size), image), "file after put"

        # the slots are reused meanwhile; the records come back into other slots
        rig.host.fill_(0xA5)
        host_want = np.full_like(want[1], 0xA5)
        back = np.setdiff1d(np.arange(S), slots)[:n].astype(np.int32)
        kvb.kv_l3_get(store, rig.host.data_ptr(), S, records, back)
        oracle.l3_get(image, pb, records, back, host_want, base)
        assert np.array_equal(rig.host.numpy(), host_want), "host tier after get"

        dst = np.setdiff1d(np.arange(g.P), src)[r.permutation(g.P - n)[:n]].astype(np.int32)
        snap = rig.snapshot()
        want = rig.expect_restore(snap, back, dst)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.hostt, back, dst), 20_000_000_000)
        rig.assert_equal(want)
        # end to end: the restored pages hold what the backed-up pages held
        og = oracle_geom(g)
        h1 = np.zeros(n * pb, dtype=np.uint8)
        h2 = np.zeros(n * pb, dtype=np.uint8)
        oracle.backup(og, snap[0], h1, src, np.arange(n), pool_offset=w.pool_offset)
        oracle.backup(og, rig.snapshot()[0], h2, dst, np.arange(n), pool_offset=w.pool_offset)
        assert np.array_equal(h1, h2), "restored pages differ from the backed-up pages"
    finally:
        kvb.kv_l3_close(store)
        os.close(fd)
        rig.close()


def test_prefetch_from_l3_then_gated_restore():
    """The storage-prefetch flow: a RESTORE is enqueued first and waits on the
    GPU for a ready word; a host thread gets the records from the L3 store into
    the host slots and then sets the word; the restore then runs.  The pool
    equals the oracle's restore of the records' pages."""
    import threading
    g = wl.LLAMA8B.geom.with_(P=40, L=4)
    S, R, n = 16, 24, 6
    pb = g.page_bytes
    r = np.random.default_rng(9)
    rig = Rig(g, S, seed=9)
    fd = os.memfd_create("kvb_l3_prefetch")
    records = np.random.default_rng(10).integers(0, 256, R * pb, dtype=np.uint8)
    os.pwrite(fd, records.tobytes(), 0)
    store = kvb.kv_l3_open(fd, 0, pb, R, 4)
    word = torch.zeros(1, dtype=torch.int64, pin_memory=True)
    try:
        recs = r.permutation(R)[:n].astype(np.int32)
        slots = r.permutation(S)[:n].astype(np.int32)
        dst = r.permutation(g.P)[:n].astype(np.int32)
        snap = rig.snapshot()
        # expected: the slots hold the records, then the restore moves them
        host_want = snap[1].copy()
        oracle.l3_get(records, pb, recs, slots, host_want)
        pool_want = snap[0].copy()
        oracle.restore(oracle_geom(g), pool_want, host_want, slots, dst)
        s = torch.cuda.Stream()
        f = kvb.kv_restore_when_ready(rig.pool, rig.hostt, slots, dst, word.data_ptr(), 1,
                                      30_000_000_000, -1, s.cuda_stream)

        def prefetch():
            kvb.kv_l3_get(store, rig.host.data_ptr(), S, recs, slots)
            word[0] = 1                                  # host data landed: release the gate

        th = threading.Thread(target=prefetch)
        th.start()
        th.join(60)
        kvb.kv_fence_wait(f, 30_000_000_000)
        rig.assert_equal((pool_want, host_want))
    finally:
        kvb.kv_l3_close(store)
        os.close(fd)
        rig.close()
