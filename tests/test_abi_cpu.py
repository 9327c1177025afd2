"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and its host-side checks return the documented codes."""
import ctypes
import os
import re

import numpy as np
import pytest

from hierarchical_kv_cache_backup_gb300 import build as kbuild

kbuild.build_library()
from hierarchical_kv_cache_backup_gb300 import kvb  # noqa: E402

HEADER = os.path.join(kbuild.INCLUDE, "kvb.h")


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^KVB_API\s+[\w\s\*]*?\b(kv_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported():
    declared = header_functions()
    assert len(declared) >= 19
    lib = ctypes.CDLL(kvb.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(kvb.EXPORTS) == declared


def test_struct_sizes_match_header():
    assert ctypes.sizeof(kvb.kv_layout) == 40
    assert ctypes.sizeof(kvb.kv_ipc_desc) == 168
    assert ctypes.sizeof(kvb.kv_config) == 24   # mode, max_ctas, staging, flags, cta_threads
    assert kvb.kv_abi_version() == 2


def lay(**kw):
    d = dict(L=2, C=2, P=64, T=16, H=2, B=128)
    d.update(kw)
    return kvb.make_layout(d["L"], d["C"], d["P"], d["T"], d["H"], d["B"],
                           kw.get("order", 0), kw.get("heads", 0))


def test_page_bytes():
    assert kvb.kv_layout_page_bytes(lay()) == 2 * 2 * 16 * 2 * 128
    assert kvb.kv_layout_page_bytes(lay(L=61, C=1, T=256, H=1, B=576)) == 8994816


@pytest.mark.parametrize("kw,status", [
    (dict(L=0), kvb.KV_ERR_LAYOUT), (dict(H=0), kvb.KV_ERR_LAYOUT), (dict(B=0), kvb.KV_ERR_LAYOUT),
    (dict(B=120), kvb.KV_ERR_ALIGNMENT), (dict(B=8), kvb.KV_ERR_ALIGNMENT),
    (dict(order=2), kvb.KV_ERR_LAYOUT), (dict(heads=7), kvb.KV_ERR_LAYOUT),
    (dict(L=1 << 20, P=1 << 30, T=1 << 20), kvb.KV_ERR_LAYOUT),
])
def test_bad_layouts(kw, status):
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_layout_page_bytes(lay(**kw))
    assert e.value.status == status
    assert kvb.kv_last_error()


def test_reserved_must_be_zero():
    l = lay()
    l.reserved = 1
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_layout_page_bytes(l)
    assert e.value.status == kvb.KV_ERR_LAYOUT


BACKUP, RESTORE = 0, 1


@pytest.mark.parametrize("kind,a,b,layer,status", [
    (BACKUP, [1, 2, 3], [0, 1, 2], -1, kvb.KV_OK),
    (BACKUP, [1, 1, 3], [0, 1, 2], -1, kvb.KV_OK),              # repeated source page is fine
    (BACKUP, [1, 2, 3], [0, 1, 1], -1, kvb.KV_ERR_DUPLICATE),   # slot written twice
    (BACKUP, [1, 64, 3], [0, 1, 2], -1, kvb.KV_ERR_OUT_OF_RANGE),
    (BACKUP, [-1, 2, 3], [0, 1, 2], -1, kvb.KV_ERR_OUT_OF_RANGE),
    (BACKUP, [1, 2, 3], [0, 1, 16], -1, kvb.KV_ERR_OUT_OF_RANGE),
    (BACKUP, [1, 2, 3], [0, 1, 2], 0, kvb.KV_ERR_INVALID_ARG),  # backup has no layer argument
    (RESTORE, [0, 1, 2], [5, 6, 7], -1, kvb.KV_OK),
    (RESTORE, [0, 0, 2], [5, 6, 7], 1, kvb.KV_OK),              # repeated source slot is fine
    (RESTORE, [0, 1, 2], [5, 6, 5], -1, kvb.KV_ERR_DUPLICATE),  # page written twice
    (RESTORE, [0, 1, 2], [5, 6, 64], -1, kvb.KV_ERR_OUT_OF_RANGE),
    (RESTORE, [0, 17, 2], [5, 6, 7], -1, kvb.KV_ERR_OUT_OF_RANGE),
    (RESTORE, [0, 1, 2], [5, 6, 7], 2, kvb.KV_ERR_OUT_OF_RANGE),  # layer >= L
    (RESTORE, [0, 1, 2], [5, 6, 7], -2, kvb.KV_ERR_OUT_OF_RANGE),
    (2, [0], [0], -1, kvb.KV_ERR_INVALID_ARG),
    (BACKUP, [], [], -1, kvb.KV_OK),
])
def test_op_validation(kind, a, b, layer, status):
    assert kvb.kv_op_validate(lay(), 16, kind, a, b, layer) == status


def test_op_validation_null_arrays():
    lib = kvb.library()
    st = lib.kv_op_validate(ctypes.byref(lay()), 16, 0, None, None, 3, -1)
    assert st == kvb.KV_ERR_INVALID_ARG


def test_duplicate_detection_large_random():
    r = np.random.default_rng(3)
    L = lay(P=4096)
    src = r.permutation(4096)[:512]
    slots = r.permutation(600)[:512]
    assert kvb.kv_op_validate(L, 600, BACKUP, src, slots) == kvb.KV_OK
    slots2 = slots.copy()
    slots2[400] = slots2[17]
    assert kvb.kv_op_validate(L, 600, BACKUP, src, slots2) == kvb.KV_ERR_DUPLICATE
    # many calls in a row reuse the duplicate stamps correctly
    for _ in range(50):
        assert kvb.kv_op_validate(L, 600, BACKUP, src, slots) == kvb.KV_OK


def test_config_roundtrip_and_checks():
    old = kvb.kv_config_get()
    try:
        kvb.kv_config_set(kvb.KV_MODE_STAGED, 64, 64 << 20)
        c = kvb.kv_config_get()
        assert (c.mode, c.max_ctas, c.staging_bytes) == (1, 64, 64 << 20)
        kvb.kv_config_set(kvb.KV_MODE_COPY_ENGINE)
        assert kvb.kv_config_get().mode == 2
        for bad in [dict(mode=3), dict(mode=5), dict(max_ctas=1 << 20), dict(staging_bytes=1000),
                    dict(flags=16), dict(flags=kvb.KV_CFG_OVERLAP_RESTORES | 32),
                    dict(cta_threads=512)]:
            with pytest.raises(kvb.KvError) as e:
                kvb.kv_config_set(**bad)
            assert e.value.status == kvb.KV_ERR_INVALID_ARG
        every = (kvb.KV_CFG_NO_BULK | kvb.KV_CFG_NO_PDL | kvb.KV_CFG_OVERLAP_RESTORES |
                 kvb.KV_CFG_OVERLAP_BACKUPS)
        kvb.kv_config_set(kvb.KV_MODE_ZERO_COPY, 6, 0, every, 1024)
        c = kvb.kv_config_get()
        assert (c.mode, c.max_ctas, c.flags, c.cta_threads) == (0, 6, every, 1024)
    finally:
        kvb.kv_config_set(old.mode, old.max_ctas, old.staging_bytes, old.flags, old.cta_threads)


def test_handles_and_fences_without_gpu():
    # unknown handles are reported, never dereferenced
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_pool_close(12345)
    assert e.value.status == kvb.KV_ERR_CLOSED
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_host_close(777)
    assert e.value.status == kvb.KV_ERR_CLOSED
    assert kvb.kv_fence_query(0) == kvb.KV_ERR_INVALID_ARG
    assert kvb.kv_fence_query((1 << 56) | 999999) == kvb.KV_ERR_INVALID_ARG
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_backup(12345, 777, [0], [0])
    assert e.value.status == kvb.KV_ERR_CLOSED


def test_register_rejects_before_touching_cuda():
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_pool_register(lay(), 0)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_pool_register(lay(), 0x1000, 8)              # pool start not 16-B aligned
    assert e.value.status == kvb.KV_ERR_ALIGNMENT
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_host_register(0x1008, 1 << 20, 4, 0, lay())  # host tier not 16-B aligned
    assert e.value.status == kvb.KV_ERR_ALIGNMENT
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_host_register(0x1000, 1000, 4, 0, lay())     # too small for 4 slots
    assert e.value.status == kvb.KV_ERR_OUT_OF_RANGE


def test_descriptor_bytes_roundtrip():
    d = kvb.kv_ipc_desc()
    d.magic, d.version, d.alloc_offset, d.generation = kvb.KVB_IPC_MAGIC, kvb.kv_abi_version(), \
        2 * 1024 * 1024 + 48, 7
    d.layout = lay(P=2048, L=40, T=32, H=8, B=256, order=1, heads=1)
    b = kvb.desc_to_bytes(d)
    assert len(b) == 168
    e = kvb.desc_from_bytes(b)
    assert e.alloc_offset == d.alloc_offset and e.layout.num_pages == 2048 and e.generation == 7
    bad = bytearray(b)
    bad[0] ^= 0xFF
    with pytest.raises(kvb.KvError) as err:
        kvb.kv_pool_import(kvb.desc_from_bytes(bytes(bad)))
    assert err.value.status == kvb.KV_ERR_INVALID_ARG


def test_split_pool_checks_before_cuda():
    lay_pf = lay(order=1)
    with pytest.raises(kvb.KvError) as e:                      # split pools are layer-first
        kvb.kv_pool_register_split(lay_pf, [0x1000] * 4)
    assert e.value.status == kvb.KV_ERR_LAYOUT
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_pool_register_split(lay(), [0x1000, 0, 0x2000, 0x3000])
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_pool_register_split(lay(), [0x1000, 0x1008, 0x2000, 0x3000])
    assert e.value.status == kvb.KV_ERR_ALIGNMENT
    lib = kvb.library()
    out = ctypes.c_void_p()
    assert lib.kv_pool_register_split(ctypes.byref(lay()), None, 0, 0, ctypes.byref(out)) == \
        kvb.KV_ERR_INVALID_ARG


def test_split_descriptor_checks_before_cuda():
    """kv_pool_import_split refuses malformed split descriptors before any CUDA
    call, kv_pool_import refuses a split descriptor, and the buffer entries
    survive a bytes round trip."""
    assert ctypes.sizeof(kvb.kv_ipc_buffer) == 72
    L, C, P, T, H, B = 2, 2, 64, 16, 2, 128
    d = kvb.kv_ipc_desc()
    d.magic, d.version = kvb.KVB_IPC_MAGIC_SPLIT, kvb.kv_abi_version()
    d.layout = lay(L=L, C=C, P=P, T=T, H=H, B=B)
    d.nbytes = L * C * P * T * H * B
    bufs = (kvb.kv_ipc_buffer * (L * C))()
    for i, b in enumerate(bufs):
        b.handle[0], b.alloc_offset = i, 4096 * i
    again = kvb.bufs_from_bytes(kvb.bufs_to_bytes(bufs))
    assert [b.alloc_offset for b in again] == [4096 * i for i in range(L * C)]
    assert [b.handle[0] for b in again] == list(range(L * C))

    def status(desc, entries):
        with pytest.raises(kvb.KvError) as e:
            kvb.kv_pool_import_split(desc, entries)
        return e.value.status

    def copy(desc, **kw):
        c = kvb.desc_from_bytes(kvb.desc_to_bytes(desc))
        for k, v in kw.items():
            setattr(c, k, v)
        return c

    assert status(copy(d, magic=kvb.KVB_IPC_MAGIC), bufs) == kvb.KV_ERR_INVALID_ARG
    assert status(copy(d, layout=lay(L=L, C=C, P=P, T=T, H=H, B=B, order=1)), bufs) == \
        kvb.KV_ERR_LAYOUT                                       # split pools are layer-first
    assert status(d, list(bufs)[:3]) == kvb.KV_ERR_INVALID_ARG  # L x C entries
    assert status(copy(d, nbytes=d.nbytes - 16), bufs) == kvb.KV_ERR_LAYOUT
    odd = kvb.bufs_from_bytes(kvb.bufs_to_bytes(bufs))
    odd[2].alloc_offset = 4100
    assert status(d, odd) == kvb.KV_ERR_ALIGNMENT
    with pytest.raises(kvb.KvError) as e:                       # the single-allocation import
        kvb.kv_pool_import(d)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG and "split" in kvb.kv_last_error()
    lib = kvb.library()
    out = ctypes.c_void_p()
    assert lib.kv_pool_import_split(ctypes.byref(d), None, L * C, ctypes.byref(out)) == \
        kvb.KV_ERR_INVALID_ARG


def test_fault_injection_points_without_gpu():
    with pytest.raises(kvb.KvError) as e:
        kvb.kv_fault_inject("no_such_point", 1)
    assert e.value.status == kvb.KV_ERR_INVALID_ARG
    kvb.kv_fault_inject("host_register", 1)
    with pytest.raises(kvb.KvError) as e:        # checks pass, then the injected failure
        kvb.kv_host_register(0x10000, 1 << 20, 4, 0, lay())
    assert e.value.status == kvb.KV_ERR_CUDA and "injected" in kvb.kv_last_error()
    kvb.kv_fault_inject("host_register", 0)
    for p in ("staging_alloc", "fence_reserve", "launch", "ipc_open", "launch_nth"):
        kvb.kv_fault_inject(p, 0)


def test_id_lists_are_refused_rather_than_wrapped():
    """The binding passes int32 ids; a wider id or a non-integer is refused,
    never wrapped or truncated into another page's id."""
    a, p = kvb._ids(np.array([3, 1, 2], dtype=np.int32))
    assert p is not None and a.dtype == np.int32
    b, _ = kvb._ids([5, 2**31 - 1, -1])                     # converted, in range
    assert b.dtype == np.int32 and b.tolist() == [5, 2**31 - 1, -1]
    c, pc = kvb._ids([])
    assert c.size == 0 and pc is None
    for bad, exc in (([2**31], ValueError), (np.array([2**32 + 5], np.int64), ValueError),
                     ([-2**31 - 1], ValueError), ([1.0, 2.0], TypeError),
                     (np.array([True]), TypeError), ([[1, 2]], ValueError)):
        with pytest.raises(exc):
            kvb._ids(bad)
    lay = kvb.make_layout(2, 2, 64, 16, 2, 128)
    with pytest.raises(ValueError):                         # before the C call
        kvb.kv_op_validate(lay, 16, 0, [2**32 + 3], [0], -1)


def test_binding_fails_loudly_without_the_library(tmp_path):
    """The binding has no fallback: a copy of it next to no built library
    refuses to import, naming the missing file."""
    import shutil
    import subprocess
    import sys

    pkg = tmp_path / "unbuilt_pkg"
    pkg.mkdir()
    shutil.copy(kvb.__file__, pkg / "kvb.py")
    (pkg / "__init__.py").write_text("")
    r = subprocess.run([sys.executable, "-c", "import unbuilt_pkg.kvb"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libkvb.so is missing" in r.stderr
