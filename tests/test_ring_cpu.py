"""The descriptor ring without a GPU: submit / pop / complete / wait between two
handles and between two processes, ring-full and wait time-outs, a server that
dies with a descriptor taken (the submitter's wait times out: fail closed),
and argument errors."""
import multiprocessing as mp
import os
import time
import uuid

import pytest

from hierarchical_kv_cache_backup_gb300 import build as kbuild

kbuild.build_library()
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ring_name():
    return f"/kvbtest_{os.getpid()}_{uuid.uuid4().hex[:8]}"


def test_round_trip_in_one_process():
    name = ring_name()
    sub = kvb.kv_ring_create(name, 4)
    srv = kvb.kv_ring_attach(name)
    try:
        op = kvb.make_ring_op(kvb.KV_RING_OP_RESTORE, [3, 1, 4], [10, 20, 30], pool_index=2,
                              layer=5, operation_id=77)
        t = kvb.kv_ring_submit(sub, op)
        assert t == 1
        t2, got = kvb.kv_ring_pop(srv)
        assert t2 == 1 and got.kind == 1 and got.pool_index == 2 and got.layer == 5
        assert got.operation_id == 77 and got.n == 3
        assert list(got.a[:3]) == [3, 1, 4] and list(got.b[:3]) == [10, 20, 30]
        with pytest.raises(kvb.KvError) as e:                     # not complete yet
            kvb.kv_ring_wait(sub, 1, 20_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
        kvb.kv_ring_complete(srv, 1, kvb.KV_OK)
        assert kvb.kv_ring_wait(sub, 1) == kvb.KV_OK
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1], [2], operation_id=78))
        t3, _ = kvb.kv_ring_pop(srv)
        kvb.kv_ring_complete(srv, t3, kvb.KV_ERR_OUT_OF_RANGE)   # the server's error comes back
        assert kvb.kv_ring_wait(sub, t) == kvb.KV_ERR_OUT_OF_RANGE
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_wait(sub, 99)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)


def test_ring_full_and_slot_reuse():
    name = ring_name()
    sub = kvb.kv_ring_create(name, 2)
    srv = kvb.kv_ring_attach(name)
    try:
        op = kvb.make_ring_op(0, [0], [0])
        assert [kvb.kv_ring_submit(sub, op) for _ in range(2)] == [1, 2]
        t0 = time.perf_counter()
        with pytest.raises(kvb.KvError) as e:                     # nothing taken: full
            kvb.kv_ring_submit(sub, op, 50_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT and time.perf_counter() - t0 >= 0.04
        kvb.kv_ring_pop(srv)
        with pytest.raises(kvb.KvError) as e:                     # taken but not complete
            kvb.kv_ring_submit(sub, op, 20_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
        kvb.kv_ring_complete(srv, 1)
        assert kvb.kv_ring_submit(sub, op) == 3
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_pop(srv, 0) and kvb.kv_ring_pop(srv, 0) and kvb.kv_ring_pop(srv, 10_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
    finally:
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)


def _server(name, count, die_after):
    import sys
    sys.path.insert(0, ROOT)
    from hierarchical_kv_cache_backup_gb300 import kvb as k

    r = k.kv_ring_attach(name)
    for i in range(count):
        t, op = k.kv_ring_pop(r, 20_000_000_000)
        if die_after is not None and i == die_after:
            os._exit(0)                                          # dies holding the descriptor
        ok = op.n == 5 and all(op.a[j] == op.operation_id + j and op.b[j] == -j for j in range(5))
        status = k.KV_ERR_LAYOUT if not ok else (
            k.KV_OK if op.operation_id % 2 == 0 else k.KV_ERR_OUT_OF_RANGE)
        k.kv_ring_complete(r, t, status)
    k.kv_ring_close(r)


def test_two_processes_wrap_around():
    name = ring_name()
    sub = kvb.kv_ring_create(name, 8)
    ctx = mp.get_context("spawn")
    n = 300
    p = ctx.Process(target=_server, args=(name, n, None))
    p.start()
    try:
        tickets = []
        for i in range(n):
            op = kvb.make_ring_op(0, [i + j for j in range(5)], [-j for j in range(5)],
                                  operation_id=i)
            tickets.append(kvb.kv_ring_submit(sub, op, 30_000_000_000))
        statuses = [kvb.kv_ring_wait(sub, t, 30_000_000_000) for t in tickets[-8:]]
        assert tickets == list(range(1, n + 1))
        want = [kvb.KV_OK if i % 2 == 0 else kvb.KV_ERR_OUT_OF_RANGE for i in range(n - 8, n)]
        assert statuses == want
    finally:
        p.join(60)
        kvb.kv_ring_close(sub)
    assert p.exitcode == 0


def test_server_death_fails_closed():
    name = ring_name()
    sub = kvb.kv_ring_create(name, 4)
    ctx = mp.get_context("spawn")
    p = ctx.Process(target=_server, args=(name, 2, 1))
    p.start()
    try:
        op = [kvb.make_ring_op(0, [i + j for j in range(5)], [-j for j in range(5)],
                               operation_id=i) for i in range(2)]
        t1 = kvb.kv_ring_submit(sub, op[0])
        t2 = kvb.kv_ring_submit(sub, op[1])
        assert kvb.kv_ring_wait(sub, t1, 30_000_000_000) == kvb.KV_OK
        p.join(60)
        with pytest.raises(kvb.KvError) as e:                     # taken, never completed
            kvb.kv_ring_wait(sub, t2, 200_000_000)
        assert e.value.status == kvb.KV_ERR_TIMEOUT
    finally:
        kvb.kv_ring_close(sub)


def test_argument_errors():
    for bad in ["noslash", "/", "/a/b", "/" + "x" * 300]:
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_create(bad, 4)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    name = ring_name()
    for slots in (0, 1, 5000):
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_create(name, slots)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    r = kvb.kv_ring_create(name, 4)
    with pytest.raises(kvb.KvError) as e:                         # name taken
        kvb.kv_ring_create(name, 4)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    op = kvb.make_ring_op(0, [1], [1])
    op.kind = 7
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_ring_submit(r, op)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    kvb.kv_ring_close(r)
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_ring_close(r)
    assert e.value.status == kvb.KV_ERR_CLOSED
    with pytest.raises(kvb.KvError) as e:                         # unlinked by its creator
        kvb.kv_ring_attach(name)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG


def _shm_view(name):
    import mmap
    fd = os.open("/dev/shm" + name, os.O_RDWR)
    try:
        return mmap.mmap(fd, os.fstat(fd).st_size)
    finally:
        os.close(fd)


def test_malformed_descriptor_in_shared_memory_is_failed_not_served():
    """An entry kv_ring_submit would refuse (written into the segment directly)
    is taken, completed with INVALID_ARG for the submitter, and reported to
    the server with its ticket; the ring keeps working."""
    import struct
    name = ring_name()
    sub = kvb.kv_ring_create(name, 4)
    srv = kvb.kv_ring_attach(name)
    m = _shm_view(name)
    try:
        slots, entry_bytes, _, entry_off = struct.unpack_from("<IIQQ", m, 8)
        assert slots == 4
        for field, value in ((8, kvb.KV_RING_MAX_IDS + 1), (0, 7)):   # n, then kind
            t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1], [2]))
            struct.pack_into("<I", m, entry_off + ((t - 1) % slots) * entry_bytes + field, value)
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_ring_pop(srv)
            assert e.value.status == kvb.KV_ERR_INVALID_ARG
            assert kvb.kv_ring_wait(sub, t) == kvb.KV_ERR_INVALID_ARG
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(1, [5, 6], [7, 8], layer=-1))
        t2, got = kvb.kv_ring_pop(srv)
        assert t2 == t and got.n == 2 and list(got.a[:2]) == [5, 6]
        kvb.kv_ring_complete(srv, t2, kvb.KV_OK)
        assert kvb.kv_ring_wait(sub, t) == kvb.KV_OK
    finally:
        m.close()
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)


def test_attach_refuses_a_header_whose_regions_overrun_the_segment():
    import struct
    name = ring_name()
    sub = kvb.kv_ring_create(name, 4)
    m = _shm_view(name)
    try:
        comp_off, entry_off, total = struct.unpack_from("<QQQ", m, 16)
        for off, bad in ((16, total + 4096), (24, total), (24, comp_off)):
            orig = struct.unpack_from("<Q", m, off)[0]
            struct.pack_into("<Q", m, off, bad)
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_ring_attach(name)
            assert e.value.status == kvb.KV_ERR_INVALID_ARG
            struct.pack_into("<Q", m, off, orig)
        kvb.kv_ring_close(kvb.kv_ring_attach(name))               # intact again: attaches
    finally:
        m.close()
        kvb.kv_ring_close(sub)


def test_gated_descriptors_and_ready_words_without_gpu():
    """Gated descriptors: the gate fields travel with the descriptor; a gate that
    names no ready word or waits above 60 s is refused by submit and, written
    into the segment directly, taken and failed by pop; ready words set through
    one handle are seen through the other (shared memory)."""
    import ctypes
    import struct
    name = ring_name()
    sub = kvb.kv_ring_create(name, 4)
    srv = kvb.kv_ring_attach(name)
    m = _shm_view(name)
    try:
        assert ctypes.sizeof(kvb.kv_ring_op) == 24 + 16 + 8 * kvb.KV_RING_MAX_IDS
        op = kvb.make_ring_op(0, [1, 2], [3, 4], ready_index=5, ready_value=9,
                              ready_timeout_ms=250)
        t = kvb.kv_ring_submit(sub, op)
        t2, got = kvb.kv_ring_pop(srv)
        assert (t2, got.ready_index, got.ready_value, got.ready_timeout_ms) == (t, 5, 9, 250)
        kvb.kv_ring_complete(srv, t2, kvb.KV_OK)
        for bad in (dict(ready_index=kvb.KV_RING_READY_WORDS, ready_value=1),
                    dict(ready_index=0, ready_value=1, ready_timeout_ms=60001)):
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1], [2], **bad))
            assert e.value.status == kvb.KV_ERR_INVALID_ARG
        # not gated (ready_value 0): any index is ignored
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1], [2], ready_index=999))
        t2, got = kvb.kv_ring_pop(srv)
        kvb.kv_ring_complete(srv, t2, kvb.KV_OK)
        # a bad gate written into the shared segment directly: taken, failed
        slots, entry_bytes, _, entry_off = struct.unpack_from("<IIQQ", m, 8)
        t = kvb.kv_ring_submit(sub, kvb.make_ring_op(0, [1], [2], ready_index=1, ready_value=1))
        struct.pack_into("<I", m, entry_off + ((t - 1) % slots) * entry_bytes + 24, 4096)
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_pop(srv)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
        assert kvb.kv_ring_wait(sub, t) == kvb.KV_ERR_INVALID_ARG
        # ready words: set through one handle, read in the shared header
        kvb.kv_ring_ready_set(sub, 3, 41)
        kvb.kv_ring_ready_set(srv, 63, 7)
        ready_off = 256   # after the fixed fields, tail, head and server_pid (64 B each)
        assert struct.unpack_from("<Q", m, ready_off + 8 * 3)[0] == 41
        assert struct.unpack_from("<Q", m, ready_off + 8 * 63)[0] == 7
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_ring_ready_set(sub, kvb.KV_RING_READY_WORDS, 1)
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    finally:
        m.close()
        kvb.kv_ring_close(srv)
        kvb.kv_ring_close(sub)
