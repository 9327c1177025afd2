"""The L3 record store (kv_l3_*) against the oracle, without a GPU.

The store moves whole host-tier pages between slots of a host buffer and
page-sized records of a file descriptor.  Every case starts the file and the
host buffer from seeded random bytes, runs the library and the oracle
(kvo_l3_put / kvo_l3_get on the file's byte image) on the same ids, and
compares the whole file and the whole host buffer byte for byte, so untouched
records, slots and the bytes around the store are checked too."""
import os
import threading

import numpy as np
import pytest

import oracle
from hierarchical_kv_cache_backup_gb300 import build as kbuild

kbuild.build_library()
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402

if not hasattr(os, "memfd_create"):
    pytest.skip("memfd_create is Linux-only", allow_module_level=True)


def file_bytes(fd, size):
    out = bytearray()
    while len(out) < size:
        chunk = os.pread(fd, size - len(out), len(out))
        if not chunk:
            break
        out += chunk
    return np.frombuffer(bytes(out), dtype=np.uint8)


def make_fd(kind, tmp_path, size, seed):
    if kind == "memfd":
        fd = os.memfd_create("kvb_l3_test")
    else:
        fd = os.open(str(tmp_path / f"store_{seed}.bin"), os.O_RDWR | os.O_CREAT | os.O_TRUNC,
                     0o600)
    init = np.random.default_rng(seed).integers(0, 256, size, dtype=np.uint8)
    os.pwrite(fd, init.tobytes(), 0)
    return fd, init


CASES = [  # (record bytes, host slots, records, base offset, n, id pattern, threads)
    (4096, 64, 200, 0, 40, "random", 0),
    (4096, 3100, 3200, 4096 + 48, 3000, "consecutive", 4),     # several runs of 1,024
    (65536, 40, 64, 16, 33, "random", 16),
    (1 << 20, 80, 80, 4096, 70, "consecutive", 1),             # runs capped at 64 MiB
    (48, 9, 12, 32, 9, "random", 3),
    (8192, 16, 16, 0, 16, "reversed", 2),
]


@pytest.mark.parametrize("kind", ["memfd", "file", "file_syscalls"])
@pytest.mark.parametrize("rb,S,R,base,n,pattern,threads", CASES)
def test_put_then_get_matches_oracle(kind, tmp_path, rb, S, R, base, n, pattern, threads):
    """memfd and read-write files go through a shared mapping; a write-only
    descriptor (put) and a read-only one (get) take the pwritev / preadv path."""
    r = np.random.default_rng(rb + S + R + n)
    size = base + R * rb + 100
    fd, image = make_fd("memfd" if kind == "memfd" else "file", tmp_path, size, seed=n)
    fd_get = fd
    if kind == "file_syscalls":
        path = str(tmp_path / f"store_{n}.bin")
        os.close(fd)
        fd = os.open(path, os.O_WRONLY)
        fd_get = os.open(path, os.O_RDONLY)
    host = r.integers(0, 256, S * rb, dtype=np.uint8)
    slots = r.permutation(S)[:n].astype(np.int32)
    if pattern == "consecutive":
        first = int(r.integers(0, R - n + 1))
        records = np.arange(first, first + n, dtype=np.int32)
    elif pattern == "reversed":
        records = np.arange(n - 1, -1, -1, dtype=np.int32)
    else:
        records = r.permutation(R)[:n].astype(np.int32)
    st = kvb.kv_l3_open(fd, base, rb, R, threads)
    st_get = kvb.kv_l3_open(fd_get, base, rb, R, threads) if fd_get != fd else st
    try:
        kvb.kv_l3_put(st, host.ctypes.data, S, slots, records)
        want = image.copy()
        oracle.l3_put(host, rb, slots, records, want, base)
        assert np.array_equal(file_bytes(fd_get, size), want), "file after put"
        # get the records back into a shuffled set of slots of another buffer
        back = r.integers(0, 256, S * rb, dtype=np.uint8)
        want_back = back.copy()
        gslots = r.permutation(S)[:n].astype(np.int32)
        kvb.kv_l3_get(st_get, back.ctypes.data, S, records, gslots)
        oracle.l3_get(want, rb, records, gslots, want_back, base)
        assert np.array_equal(back, want_back), "host after get"
    finally:
        kvb.kv_l3_close(st)
        os.close(fd)
        if fd_get != fd:
            kvb.kv_l3_close(st_get)
            os.close(fd_get)


def test_errors_leave_everything_untouched(tmp_path):
    rb, S, R = 4096, 8, 8
    fd, image = make_fd("memfd", tmp_path, R * rb, seed=1)
    host = np.arange(S * rb, dtype=np.uint8)
    st = kvb.kv_l3_open(fd, 0, rb, R)
    try:
        for slots, records, code in [([0, 8], [1, 2], kvb.KV_ERR_OUT_OF_RANGE),
                                     ([0, 1], [1, 8], kvb.KV_ERR_OUT_OF_RANGE),
                                     ([0, -1], [1, 2], kvb.KV_ERR_OUT_OF_RANGE),
                                     ([0, 1], [3, 3], kvb.KV_ERR_DUPLICATE)]:
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_l3_put(st, host.ctypes.data, S, slots, records)
            assert e.value.status == code
        with pytest.raises(kvb.KvError) as e:                   # a get writes a slot twice
            kvb.kv_l3_get(st, host.ctypes.data, S, [1, 2], [4, 4])
        assert e.value.status == kvb.KV_ERR_DUPLICATE
        assert np.array_equal(file_bytes(fd, R * rb), image)
        assert np.array_equal(host, np.arange(S * rb, dtype=np.uint8))
        kvb.kv_l3_put(st, host.ctypes.data, S, [], [])          # empty call is a no-op
        kvb.kv_l3_put(st, host.ctypes.data, S, [2, 2], [0, 1])  # a put may read a slot twice
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_l3_put(st, 0, S, [0], [0])
        assert e.value.status == kvb.KV_ERR_INVALID_ARG
    finally:
        kvb.kv_l3_close(st)
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_l3_close(st)
    assert e.value.status == kvb.KV_ERR_CLOSED
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_l3_put(st, host.ctypes.data, S, [0], [0])
    assert e.value.status == kvb.KV_ERR_CLOSED
    os.close(fd)


@pytest.mark.parametrize("syscalls", [False, True])
def test_get_past_the_end_of_the_file_is_an_io_error(tmp_path, syscalls):
    rb = 4096
    path = str(tmp_path / "short.bin")
    fd = os.open(path, os.O_RDWR | os.O_CREAT, 0o600)
    os.ftruncate(fd, 2 * rb)                                    # two records exist
    fd_get = os.open(path, os.O_RDONLY) if syscalls else fd
    st = kvb.kv_l3_open(fd, 0, rb, 10)
    st_get = kvb.kv_l3_open(fd_get, 0, rb, 10) if syscalls else st
    host = np.zeros(4 * rb, dtype=np.uint8)
    try:
        kvb.kv_l3_get(st_get, host.ctypes.data, 4, [0, 1], [0, 1])
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_l3_get(st_get, host.ctypes.data, 4, [5], [2])
        assert e.value.status == kvb.KV_ERR_IO and "end" in str(e.value)
        kvb.kv_l3_put(st, host.ctypes.data, 4, [3], [9])        # a put grows the file
        assert os.fstat(fd).st_size == 10 * rb
    finally:
        kvb.kv_l3_close(st)
        os.close(fd)
        if syscalls:
            kvb.kv_l3_close(st_get)
            os.close(fd_get)


def test_open_checks():
    fd = os.memfd_create("kvb_l3_open")
    rd, wr = os.pipe()
    try:
        for args in [(-1, 0, 4096, 4, 0), (rd, 0, 4096, 4, 0), (fd, 0, 0, 4, 0),
                     (fd, 0, 4096, 0, 0), (fd, 0, 4096, 4, 65)]:
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_l3_open(*args)
            assert e.value.status == kvb.KV_ERR_INVALID_ARG, args
        for args in [(fd, 0, 4096, (1 << 31) + 1, 0), (fd, (1 << 63) - 4096, 4096, 2, 0)]:
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_l3_open(*args)
            assert e.value.status == kvb.KV_ERR_OUT_OF_RANGE, args
    finally:
        os.close(fd)
        os.close(rd)
        os.close(wr)


def test_calls_from_several_threads_on_one_store():
    rb, R, S = 16384, 256, 256
    fd = os.memfd_create("kvb_l3_threads")
    st = kvb.kv_l3_open(fd, 0, rb, R, 4)
    host = np.random.default_rng(3).integers(0, 256, S * rb, dtype=np.uint8)
    errors = []

    def job(k):
        try:
            recs = np.arange(k * 32, (k + 1) * 32, dtype=np.int32)
            for _ in range(20):
                kvb.kv_l3_put(st, host.ctypes.data, S, recs, recs)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    try:
        ts = [threading.Thread(target=job, args=(k,)) for k in range(8)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errors, errors
        assert np.array_equal(file_bytes(fd, R * rb), host)    # record r <- slot r
    finally:
        kvb.kv_l3_close(st)
        os.close(fd)
