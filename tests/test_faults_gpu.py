"""Host-side failure drills on the GPU path: an injected failure at each point
returns its code, enqueues nothing, leaves every byte of the pool and the host
tier unchanged, and the next operation succeeds (the engine keeps serving).
No GPU fault, trap or hang is involved: the failures are made on the host."""
import multiprocessing as mp
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_rig import Rig  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402
from hierarchical_kv_cache_backup_gb300 import workloads as wl  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture
def rig():
    r = Rig(wl.LLAMA8B.geom.with_(P=48, L=4), 16, seed=61)
    yield r
    for p in ("staging_alloc", "fence_reserve", "launch", "ipc_open", "host_register",
              "launch_nth"):
        kvb.kv_fault_inject(p, 0)
    r.close()


def _ops(rig):
    return {
        "backup": lambda: kvb.kv_backup(rig.pool, rig.hostt, [3, 9, 11], [0, 5, 7]),
        "restore": lambda: kvb.kv_restore(rig.pool, rig.hostt, [0, 5], [20, 21]),
        "restore_layer": lambda: kvb.kv_restore(rig.pool, rig.hostt, [0, 5], [20, 21], 2),
        "restore_layers": lambda: kvb.kv_restore_layers(rig.pool, rig.hostt, [0, 5], [20, 21],
                                                         0, 4)[-1],
    }


@pytest.mark.parametrize("point,status,mode", [
    ("fence_reserve", kvb.KV_ERR_NO_MEMORY, kvb.KV_MODE_ZERO_COPY),
    ("launch", kvb.KV_ERR_CUDA, kvb.KV_MODE_ZERO_COPY),
    ("launch", kvb.KV_ERR_CUDA, kvb.KV_MODE_STAGED),
    ("staging_alloc", kvb.KV_ERR_NO_MEMORY, kvb.KV_MODE_STAGED),
])
def test_injected_failure_has_no_side_effect_and_engine_recovers(rig, point, status, mode):
    old = kvb.kv_config_get()
    try:
        ops = _ops(rig)
        names = ["backup", "restore", "restore_layer"] + (["restore_layers"]
                                                          if mode == kvb.KV_MODE_ZERO_COPY else [])
        for i, name in enumerate(names):
            # a new staging size forces the staged path to allocate again
            kvb.kv_config_set(mode, 0, (6 + i) << 20)
            snap = rig.snapshot()
            launches = kvb.kv_launch_count()
            kvb.kv_fault_inject(point, 1)
            with pytest.raises(kvb.KvError) as e:
                ops[name]()
            assert e.value.status == status, (name, kvb.kv_last_error())
            assert "injected" in kvb.kv_last_error()
            assert kvb.kv_launch_count() == launches
            rig.assert_equal(snap)
            # and the next one lands, bit-exact
            if name == "backup":
                want = rig.expect_backup(snap, [3, 9, 11], [0, 5, 7])
            elif name == "restore":
                want = rig.expect_restore(snap, [0, 5], [20, 21])
            elif name == "restore_layer":
                want = rig.expect_restore(snap, [0, 5], [20, 21], 2)
            else:
                want = rig.expect_restore(snap, [0, 5], [20, 21])
            kvb.kv_fence_wait(ops[name](), 30_000_000_000)
            rig.assert_equal(want)
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)


def test_fault_points_armed_from_the_environment():
    code = f"""
import sys
sys.path[:0] = [{ROOT!r}, {os.path.join(ROOT, 'tests')!r}]
import torch
from gpu_rig import Rig
from hierarchical_kv_cache_backup_gb300 import kvb, workloads as wl
rig = Rig(wl.TINY.geom, 16, seed=3)
codes = []
for _ in range(3):
    try:
        kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.hostt, [1], [2]), 10_000_000_000)
        codes.append(0)
    except kvb.KvError as e:
        codes.append(e.status)
print("CODES", codes)
"""
    env = dict(os.environ, KVB_FAULT="fence_reserve:1,launch:1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert f"CODES [{kvb.KV_ERR_NO_MEMORY}, {kvb.KV_ERR_CUDA}, 0]" in r.stdout


def _export(q, done):
    sys.path.insert(0, ROOT)
    import torch as t
    from hierarchical_kv_cache_backup_gb300 import kvb as k
    from hierarchical_kv_cache_backup_gb300 import workloads as w

    g = w.TINY.geom
    a = t.zeros(g.pool_bytes, dtype=t.uint8, device="cuda")
    lay = k.make_layout(g.L, g.C, g.P, g.T, g.H, g.B)
    p = k.kv_pool_register(lay, a.data_ptr(), 0)
    q.put(k.desc_to_bytes(k.kv_pool_export(p)))
    done.wait(300)
    k.kv_pool_close(p)


def test_injected_ipc_open_failure_then_import():
    ctx = mp.get_context("spawn")
    q, done = ctx.Queue(), ctx.Event()
    p = ctx.Process(target=_export, args=(q, done))
    p.start()
    try:
        desc = kvb.desc_from_bytes(q.get(timeout=300))
        kvb.kv_fault_inject("ipc_open", 1)
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_import(desc)
        assert e.value.status == kvb.KV_ERR_CUDA and "injected" in kvb.kv_last_error()
        pool = kvb.kv_pool_import(desc)          # the retry maps it
        kvb.kv_pool_close(pool)
    finally:
        done.set()
        p.join(120)


@pytest.mark.parametrize("mode,kind,n,nth", [
    (kvb.KV_MODE_STAGED, "backup", 200, 3),      # 7 chunks of 32 pages: the 3rd launch fails
    (kvb.KV_MODE_STAGED, "restore", 200, 4),
    (kvb.KV_MODE_ZERO_COPY, "backup", 2100, 2),  # two launches: the second fails
    (kvb.KV_MODE_ZERO_COPY, "restore", 2100, 2),
])
def test_failure_in_the_middle_of_an_op_then_the_engine_recovers(mode, kind, n, nth):
    """A launch that fails after part of an op was enqueued: the op reports
    CUDA, what it enqueued before still completes, nothing else is touched,
    and the following ops (which may reuse the staging buffers) are exact."""
    g = wl.Geometry(L=2, C=2, P=3 * n + 100, T=16, H=2, B=128)   # three disjoint page sets
    rig = Rig(g, 2 * n, seed=77)
    old = kvb.kv_config_get()
    try:
        kvb.kv_config_set(mode, 0, 2 << 20)       # 512 KiB ping-pong buffers: many chunks
        r = np.random.default_rng(5)
        pages = r.permutation(g.P).astype(np.int32)
        a_src, b_src, dst = pages[:n], pages[n:2 * n], pages[2 * n:3 * n]
        slots_a = np.arange(n, dtype=np.int32)
        slots_b = np.arange(n, 2 * n, dtype=np.int32)
        snap = rig.snapshot()
        kvb.kv_fault_inject("launch_nth", nth)
        with pytest.raises(kvb.KvError) as e:
            if kind == "backup":
                kvb.kv_backup(rig.pool, rig.hostt, a_src, slots_a)
            else:
                kvb.kv_restore(rig.pool, rig.hostt, slots_a, dst)
        assert e.value.status == kvb.KV_ERR_CUDA
        torch.cuda.synchronize()
        after = rig.snapshot()
        # the failed op wrote only where it was allowed to (backup: slots_a; restore: dst)
        if kind == "backup":
            assert np.array_equal(after[0], snap[0])
            keep = np.ones(after[1].size, bool)
            keep[:n * g.page_bytes] = False
            assert np.array_equal(after[1][keep], snap[1][keep])
        else:
            assert np.array_equal(after[1], snap[1])
            from gpu_rig import oracle_geom
            import oracle
            moved = snap[0].copy()
            oracle.restore(oracle_geom(g), moved, snap[1], slots_a, dst, threads=8)
            untouched = np.flatnonzero(moved == snap[0])
            assert np.array_equal(after[0][untouched], snap[0][untouched])
        # the engine keeps serving, exactly: a backup and a restore through the same path
        want = rig.expect_backup(after, b_src, slots_b)
        kvb.kv_fence_wait(kvb.kv_backup(rig.pool, rig.hostt, b_src, slots_b), 60_000_000_000)
        rig.assert_equal(want)
        want = rig.expect_restore(want, slots_b, dst)
        kvb.kv_fence_wait(kvb.kv_restore(rig.pool, rig.hostt, slots_b, dst), 60_000_000_000)
        rig.assert_equal(want)
    finally:
        kvb.kv_fault_inject("launch_nth", 0)
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)
        rig.close()


def test_gated_op_failing_after_its_gate_does_not_poison_the_next_op(rig):
    """A gated backup whose move launch fails after its gate was enqueued: the
    gate still runs and, its ready word never arriving, records a give-up
    under the op's sequence number.  That number must not pass to the next op:
    the following gated backup, its ready word set, moves its pages exactly
    and its fence reports success, not ABORTED."""
    word = torch.zeros(1, dtype=torch.int64, pin_memory=True)
    snap = rig.snapshot()
    kvb.kv_fault_inject("launch", 1)
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_backup_when_ready(rig.pool, rig.hostt, [3, 9], [0, 5], word.data_ptr(), 1,
                                 50_000_000)                   # 50 ms, never satisfied
    assert e.value.status == kvb.KV_ERR_CUDA
    torch.cuda.synchronize()                                   # the stale gate has given up
    rig.assert_equal(snap)
    word[0] = 1
    want = rig.expect_backup(snap, [11, 4], [2, 6])
    f = kvb.kv_backup_when_ready(rig.pool, rig.hostt, [11, 4], [2, 6], word.data_ptr(), 1,
                                 1_000_000_000)
    kvb.kv_fence_wait(f, 20_000_000_000)
    assert kvb.kv_fence_query(f) == kvb.KV_OK
    rig.assert_equal(want)


_CHAIN_STALL_CHILD = r'''
import sys, numpy as np, torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import oracle
from gpu_rig import Rig, oracle_geom
from hierarchical_kv_cache_backup_gb300 import kvb
from hierarchical_kv_cache_backup_gb300 import workloads as wl
g = wl.MLA_FP8.geom.with_(P=64, L=4)
rig = Rig(g, 8, seed=71)
want = rig.snapshot()
want = (want[0].copy(), want[1])
s = torch.cuda.Stream()
kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 0, 0, kvb.KV_CFG_OVERLAP_RESTORES)
slots, dst = np.arange(8, dtype=np.int32), np.arange(10, 18, dtype=np.int32)
f0 = kvb.kv_restore(rig.pool, rig.hostt, slots, dst, 0, s.cuda_stream)
kvb.kv_fault_inject("chain_stall", 1)
f1 = kvb.kv_restore(rig.pool, rig.hostt, slots, dst, 1, s.cuda_stream)   # overlapped, stalls
assert kvb.kv_overlap_count() == 1
s.synchronize()                                     # the wait ran out and the kernel ended
try:
    kvb.kv_fence_wait(f1, 30_000_000_000)
    print("NO-ERROR")
except kvb.KvError as e:
    print("STATUS", e.status == kvb.KV_ERR_TIMEOUT, "out of call order" in kvb.kv_last_error())
for layer in (0, 1):
    oracle.restore(oracle_geom(g), want[0], want[1], slots, dst, layer=layer)
rig.assert_equal(want)                              # the bytes landed all the same
print("BYTES-OK")
'''


def test_chained_fence_wait_runs_out_and_reports_timeout():
    """An overlapped restore whose chained fence wait cannot be satisfied (the
    "chain_stall" drill: a sequence number its predecessor never stores) gives
    up after its 2 s bound, publishes its fence, and every fence query then
    reports KV_ERR_TIMEOUT; its bytes are the oracle's.  Run in a child process:
    the kernel error word it sets is sticky for the process."""
    import subprocess
    import sys
    root = __import__("os").path.dirname(__import__("os").path.dirname(
        __import__("os").path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHAIN_STALL_CHILD, root], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "STATUS True True" in r.stdout, r.stdout + r.stderr
    assert "BYTES-OK" in r.stdout
