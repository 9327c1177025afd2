"""Mixed concurrency stress: four host threads, each on its own stream and its
own disjoint range of pages and slots, issue a seeded random mix of backups,
whole-prefix and one-layer restores and progressive restores (one of them above
2,048 pages, through the device id buffer) while the process-wide transfer mode
switches between zero-copy, STAGED and COPY_ENGINE.  The shared resources --
fence ring, staging ping-pong buffers and their side streams, the device id
buffer -- must keep every op exact: the oracle replays each thread's ops in
order and the whole pool allocation and host tier must match."""
import threading

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

THREADS, PAGES, SLOTS = 4, 3000, 2600
MODES = [kvb.KV_MODE_ZERO_COPY, kvb.KV_MODE_STAGED, kvb.KV_MODE_COPY_ENGINE]


def plan_ops(t, g, r):
    """A seeded list of ops for thread t inside its page and slot ranges."""
    p0, s0 = t * PAGES, t * SLOTS
    ops = []
    for k in range(10):
        kind = str(r.choice(["backup", "restore", "restore_layer", "restore_layers"]))
        n = int(r.integers(1, 300))
        if t == 0 and k == 3:                          # above one launch's id capacity
            kind, n = "restore_layers", 2200
        pages = (p0 + r.permutation(PAGES)[:n]).astype(np.int32)
        slots = (s0 + r.permutation(SLOTS)[:n]).astype(np.int32)
        layer = int(r.integers(0, g.L))
        ops.append((kind, pages, slots, layer, MODES[int(r.integers(len(MODES)))]))
    return ops


def test_mixed_ops_from_four_threads_match_the_oracle():
    g = wl.Geometry(L=4, C=2, P=THREADS * PAGES, T=16, H=4, B=64)
    rig = Rig(g, THREADS * SLOTS, seed=91)
    old = kvb.kv_config_get()
    r = np.random.default_rng(91)
    plans = [plan_ops(t, g, r) for t in range(THREADS)]
    errors = []
    try:
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 8 << 20)
        snap = rig.snapshot()

        def run(t):
            try:
                s = torch.cuda.Stream()
                fences = []
                for kind, pages, slots, layer, mode in plans[t]:
                    kvb.kv_config_set(mode, 0, 8 << 20)   # process-wide: affects every thread
                    if kind == "backup":
                        fences.append(kvb.kv_backup(rig.pool, rig.hostt, pages, slots,
                                                    s.cuda_stream))
                    elif kind == "restore":
                        fences.append(kvb.kv_restore(rig.pool, rig.hostt, slots, pages, -1,
                                                     s.cuda_stream))
                    elif kind == "restore_layer":
                        fences.append(kvb.kv_restore(rig.pool, rig.hostt, slots, pages, layer,
                                                     s.cuda_stream))
                    else:
                        fences += kvb.kv_restore_layers(rig.pool, rig.hostt, slots, pages, 0,
                                                        g.L, s.cuda_stream)
                for f in fences:
                    kvb.kv_fence_wait(f, 120_000_000_000)
            except Exception as e:  # noqa: BLE001 - reported below
                errors.append((t, repr(e)))

        ts = [threading.Thread(target=run, args=(t,)) for t in range(THREADS)]
        for th in ts:
            th.start()
        for th in ts:
            th.join()
        assert not errors, errors
        # the oracle: each thread's ops in order (threads touch disjoint bytes)
        og = oracle_geom(g)
        pool, host = snap[0].copy(), snap[1].copy()
        for t in range(THREADS):
            for kind, pages, slots, layer, _ in plans[t]:
                if kind == "backup":
                    oracle.backup(og, pool, host, pages, slots, threads=8)
                else:
                    oracle.restore(og, pool, host, slots, pages,
                                   layer=layer if kind == "restore_layer" else -1, threads=8)
        rig.assert_equal((pool, host))
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        rig.close()


def test_overlapped_restores_from_four_threads_match_the_oracle():
    """Four threads, each on its own stream, issue mostly one-layer restores
    drawn from a small page range (so consecutive restores often share a page
    and layer, and must not overlap, and often do not, and may), mixed with
    whole-prefix restores, backups of pages just restored and progressive
    restores, while the process-wide config flips KV_CFG_OVERLAP_RESTORES and
    KV_CFG_OVERLAP_BACKUPS on and off and the mode between zero-copy, STAGED and
    COPY_ENGINE.  The oracle
    replays each thread's ops in order; the whole allocation and tier match."""
    P_T, S_T = 400, 400
    g = wl.Geometry(L=4, C=2, P=THREADS * P_T, T=16, H=4, B=64)
    rig = Rig(g, THREADS * S_T, seed=93)
    old = kvb.kv_config_get()
    r = np.random.default_rng(93)
    OV = kvb.KV_CFG_OVERLAP_RESTORES
    OB = kvb.KV_CFG_OVERLAP_BACKUPS

    def plan(t):
        ops = []
        for _ in range(40):
            kind = str(r.choice(["restore_layer"] * 6 + ["restore", "backup", "backup",
                                                          "restore_layers"]))
            n = int(r.integers(1, 120))
            pages = (t * P_T + r.permutation(P_T)[:n]).astype(np.int32)
            slots = (t * S_T + r.permutation(S_T)[:n]).astype(np.int32)
            mode = [kvb.KV_MODE_ZERO_COPY] * 4 + [kvb.KV_MODE_STAGED, kvb.KV_MODE_COPY_ENGINE]
            ops.append((kind, pages, slots, int(r.integers(g.L)), int(r.choice(mode)),
                        int(r.choice([OV | OB, OV | OB, OV, OB, 0]))))
        return ops

    plans = [plan(t) for t in range(THREADS)]
    errors = []
    c0 = kvb.kv_overlap_count()
    try:
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 8 << 20)
        snap = rig.snapshot()

        def run(t):
            try:
                s = torch.cuda.Stream()
                fences = []
                for kind, pages, slots, layer, mode, flags in plans[t]:
                    kvb.kv_config_set(mode, 0, 8 << 20, flags)   # process-wide
                    if kind == "backup":
                        fences.append(kvb.kv_backup(rig.pool, rig.hostt, pages, slots,
                                                    s.cuda_stream))
                    elif kind == "restore":
                        fences.append(kvb.kv_restore(rig.pool, rig.hostt, slots, pages, -1,
                                                     s.cuda_stream))
                    elif kind == "restore_layer":
                        fences.append(kvb.kv_restore(rig.pool, rig.hostt, slots, pages, layer,
                                                     s.cuda_stream))
                    else:
                        fences += kvb.kv_restore_layers(rig.pool, rig.hostt, slots, pages, 0,
                                                        g.L, s.cuda_stream)
                kvb.kv_fence_wait(fences[-1], 120_000_000_000)
                for f in fences:   # the last complete implies every earlier one on the stream
                    assert kvb.kv_fence_query(f) == kvb.KV_OK
            except Exception as e:  # noqa: BLE001 - reported below
                errors.append((t, repr(e)))

        ts = [threading.Thread(target=run, args=(t,)) for t in range(THREADS)]
        for th in ts:
            th.start()
        for th in ts:
            th.join()
        assert not errors, errors
        assert kvb.kv_overlap_count() > c0    # the flag took effect on some of them
        og = oracle_geom(g)
        pool, host = snap[0].copy(), snap[1].copy()
        for t in range(THREADS):
            for kind, pages, slots, layer, _, _ in plans[t]:
                if kind == "backup":
                    oracle.backup(og, pool, host, pages, slots, threads=8)
                else:
                    oracle.restore(og, pool, host, slots, pages,
                                   layer=layer if kind == "restore_layer" else -1, threads=8)
        rig.assert_equal((pool, host))
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        rig.close()
