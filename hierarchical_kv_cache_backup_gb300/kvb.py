"""Thin ctypes binding of the C ABI in include/kvb.h (argument marshalling only).

Every function has the C name.  Pointers are Python ints (``tensor.data_ptr()``),
streams are ``torch.cuda.Stream.cuda_stream`` ints (or None for the legacy
default stream), id lists are anything ``numpy.asarray(..., int32)`` accepts.
A non-OK status raises :class:`KvError` carrying the status and the library's
message; ``kv_fence_query`` returns its status instead (TIMEOUT = not yet).

The library must have been built (``python -m hierarchical_kv_cache_backup_gb300.build``
or ``__graft_entry__.build()``); importing this module without it fails loudly.
There is no fallback path of any kind.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libkvb.so")

KV_OK = 0
KV_ERR_INVALID_ARG = 1
KV_ERR_OUT_OF_RANGE = 2
KV_ERR_DUPLICATE = 3
KV_ERR_ALIGNMENT = 4
KV_ERR_LAYOUT = 5
KV_ERR_STALE = 6
KV_ERR_TIMEOUT = 7
KV_ERR_CUDA = 8
KV_ERR_NO_MEMORY = 9
KV_ERR_CLOSED = 10
KV_ERR_ABORTED = 11
KV_ERR_IO = 12
STATUS_NAMES = {v: k for k, v in dict(globals()).items() if k.startswith("KV_OK") or k.startswith("KV_ERR_")}

KV_LAYER_FIRST, KV_PAGE_FIRST = 0, 1
KV_NHD, KV_HND = 0, 1
KV_MODE_ZERO_COPY, KV_MODE_STAGED, KV_MODE_COPY_ENGINE = 0, 1, 2
KV_CFG_NO_BULK = 1
KV_CFG_NO_PDL = 2
KV_CFG_OVERLAP_RESTORES = 4
KV_CFG_OVERLAP_BACKUPS = 8
KVB_IPC_MAGIC = 0x4B564231
KVB_IPC_MAGIC_SPLIT = 0x4B564253

# the symbols include/kvb.h declares
EXPORTS = ("kv_pool_register", "kv_pool_register_split", "kv_pool_export", "kv_pool_import",
           "kv_pool_export_split", "kv_pool_import_split", "kv_pool_close",
           "kv_pool_retire", "kv_pool_info", "kv_host_register", "kv_host_close", "kv_backup",
           "kv_restore", "kv_restore_layers", "kv_backup_when_ready", "kv_restore_when_ready", "kv_device_gather", "kv_device_scatter", "kv_backup_staged_noalloc",
           "kv_op_validate", "kv_fence_query", "kv_fence_wait",
           "kv_fence_stream_wait", "kv_config_get", "kv_config_set", "kv_layout_page_bytes",
           "kv_launch_count", "kv_overlap_count", "kv_last_error", "kv_abi_version", "kv_ring_create",
           "kv_ring_attach", "kv_ring_close", "kv_ring_submit", "kv_ring_wait", "kv_ring_serve",
           "kv_ring_pop", "kv_ring_complete", "kv_ring_serve_device", "kv_ring_device_result",
           "kv_ring_device_stop", "kv_ring_ready_set", "kv_ring_ready_stream_set",
           "kv_fault_inject", "kv_l3_open", "kv_l3_close",
           "kv_l3_put", "kv_l3_get")


class KvError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


class kv_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in ("num_layers", "num_comps", "num_pages",
                                               "page_tokens", "num_heads", "head_bytes", "order",
                                               "heads", "elem_bytes", "reserved")]


class kv_ipc_desc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("handle", ctypes.c_uint8 * 64), ("alloc_offset", ctypes.c_uint64),
                ("nbytes", ctypes.c_uint64), ("instance_id", ctypes.c_uint64),
                ("generation", ctypes.c_uint64), ("exporter_pid", ctypes.c_int64),
                ("device_uuid", ctypes.c_uint8 * 16), ("layout", kv_layout)]


class kv_ipc_buffer(ctypes.Structure):
    _fields_ = [("handle", ctypes.c_uint8 * 64), ("alloc_offset", ctypes.c_uint64)]


KV_RING_MAX_IDS = 1024
KV_RING_OP_BACKUP, KV_RING_OP_RESTORE = 0, 1
KV_RING_READY_WORDS = 64


class kv_ring_op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_uint32), ("pool_index", ctypes.c_uint32),
                ("n", ctypes.c_uint32), ("layer", ctypes.c_int32),
                ("operation_id", ctypes.c_uint64),
                ("ready_index", ctypes.c_uint32), ("ready_timeout_ms", ctypes.c_uint32),
                ("ready_value", ctypes.c_uint64),
                ("a", ctypes.c_int32 * KV_RING_MAX_IDS), ("b", ctypes.c_int32 * KV_RING_MAX_IDS)]


class kv_config(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_uint32), ("max_ctas", ctypes.c_uint32),
                ("staging_bytes", ctypes.c_uint64), ("flags", ctypes.c_uint32),
                ("cta_threads", ctypes.c_uint32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -m hierarchical_kv_cache_backup_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    u32, u64, i32, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p
    st = ctypes.c_int
    P = ctypes.POINTER
    sig = {
        "kv_pool_register": (st, [P(kv_layout), vp, u64, u64, u64, P(vp)]),
        "kv_pool_register_split": (st, [P(kv_layout), P(vp), u64, u64, P(vp)]),
        "kv_pool_export": (st, [vp, P(kv_ipc_desc)]),
        "kv_pool_import": (st, [P(kv_ipc_desc), P(vp)]),
        "kv_pool_export_split": (st, [vp, P(kv_ipc_desc), P(kv_ipc_buffer), u32]),
        "kv_pool_import_split": (st, [P(kv_ipc_desc), P(kv_ipc_buffer), u32, P(vp)]),
        "kv_pool_close": (st, [vp]),
        "kv_pool_retire": (st, [u64, u64]),
        "kv_pool_info": (st, [vp, P(kv_layout), P(vp), P(u64)]),
        "kv_host_register": (st, [vp, u64, u32, u32, P(kv_layout), P(vp)]),
        "kv_host_close": (st, [vp]),
        "kv_backup": (st, [vp, vp, vp, vp, u32, vp, P(u64)]),
        "kv_restore": (st, [vp, vp, vp, vp, u32, i32, vp, P(u64)]),
        "kv_restore_layers": (st, [vp, vp, vp, vp, u32, u32, u32, vp, P(u64)]),
        "kv_restore_when_ready": (st, [vp, vp, vp, vp, u32, i32, vp, u64, u64, vp, P(u64)]),
        "kv_backup_when_ready": (st, [vp, vp, vp, vp, u32, vp, u64, u64, vp, P(u64)]),
        "kv_device_gather": (st, [vp, vp, u64, u32, vp, u32, vp, P(u64)]),
        "kv_device_scatter": (st, [vp, vp, u64, u32, vp, u32, i32, vp, P(u64)]),
        "kv_backup_staged_noalloc": (st, [vp, vp, vp, vp, u32, vp]),
        "kv_op_validate": (st, [P(kv_layout), u32, ctypes.c_int, vp, vp, u32, i32]),
        "kv_fence_query": (st, [u64]),
        "kv_fence_wait": (st, [u64, u64]),
        "kv_fence_stream_wait": (st, [u64, vp]),
        "kv_config_get": (st, [P(kv_config)]),
        "kv_config_set": (st, [P(kv_config)]),
        "kv_layout_page_bytes": (st, [P(kv_layout), P(u64)]),
        "kv_launch_count": (u64, []),
        "kv_overlap_count": (u64, []),
        "kv_last_error": (ctypes.c_char_p, []),
        "kv_abi_version": (u32, []),
        "kv_ring_create": (st, [ctypes.c_char_p, u32, P(vp)]),
        "kv_ring_attach": (st, [ctypes.c_char_p, P(vp)]),
        "kv_ring_close": (st, [vp]),
        "kv_ring_submit": (st, [vp, P(kv_ring_op), u64, P(u64)]),
        "kv_ring_wait": (st, [vp, u64, u64, P(ctypes.c_int)]),
        "kv_ring_serve": (st, [vp, P(vp), u32, vp, vp, u32, u64, P(u32)]),
        "kv_ring_pop": (st, [vp, u64, P(kv_ring_op), P(u64)]),
        "kv_ring_complete": (st, [vp, u64, ctypes.c_int]),
        "kv_ring_serve_device": (st, [vp, P(vp), u32, vp, vp, u32, u64, P(u64)]),
        "kv_ring_device_result": (st, [vp, P(u32), P(ctypes.c_int)]),
        "kv_ring_device_stop": (st, [vp]),
        "kv_ring_ready_set": (st, [vp, u32, u64]),
        "kv_ring_ready_stream_set": (st, [vp, u32, u64, vp]),
        "kv_fault_inject": (st, [ctypes.c_char_p, u32]),
        "kv_l3_open": (st, [ctypes.c_int, u64, u64, u64, u32, P(vp)]),
        "kv_l3_close": (st, [vp]),
        "kv_l3_put": (st, [vp, vp, u64, vp, vp, u32]),
        "kv_l3_get": (st, [vp, vp, u64, vp, vp, u32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def _check(status: int):
    if status != KV_OK:
        raise KvError(status, _lib.kv_last_error().decode(errors="replace"))


_I32 = np.dtype(np.int32)


def _ids(x):
    """An int32 C-contiguous view or copy of `x` and its address (None if empty).
    Arrays that already qualify pass through; the address comes from the buffer
    protocol (cheaper than ndarray.ctypes on every call).  Anything else is
    converted only if it is a one-dimensional list of integers inside the int32
    range: a wider id is refused, never wrapped into another page's id."""
    if type(x) is not np.ndarray or x.dtype != _I32 or not x.flags.c_contiguous:
        a = np.asarray(x)
        if a.ndim > 1:
            raise ValueError(f"ids must be one-dimensional, got shape {a.shape}")
        if a.size:
            if a.dtype.kind not in "iu":
                raise TypeError(f"ids must be integers, got dtype {a.dtype}")
            if a.dtype != _I32 and (int(a.min()) < -2**31 or int(a.max()) >= 2**31):
                raise ValueError("ids outside the int32 range")
        x = np.ascontiguousarray(a, dtype=np.int32).reshape(-1)
    if x.size == 0:
        return x, None
    try:
        return x, ctypes.addressof(ctypes.c_char.from_buffer(x))
    except TypeError:                       # read-only buffer
        return x, x.ctypes.data


def make_layout(L, C, P, T, H, B, order=KV_LAYER_FIRST, heads=KV_NHD, elem_bytes=2) -> kv_layout:
    """A kv_layout: L layers, C components, P pages, T tokens per page, H heads, B bytes per
    head vector; order / heads of the device pool."""
    return kv_layout(L, C, P, T, H, B, order, heads, elem_bytes, 0)


# ------------------------------------------------------------------- pools

def kv_pool_register(layout: kv_layout, base: int, offset: int = 0, instance_id: int = 0,
                     generation: int = 0) -> int:
    """Registers a pool that starts `offset` bytes after device pointer `base`; returns its
    handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_pool_register(ctypes.byref(layout), base, offset, instance_id, generation,
                                 ctypes.byref(out)))
    return out.value


def kv_pool_register_split(layout: kv_layout, bases, instance_id: int = 0,
                           generation: int = 0) -> int:
    """bases: L x C device pointers, entry l * C + c."""
    arr = (ctypes.c_void_p * max(1, len(bases)))(*bases)
    out = ctypes.c_void_p()
    _check(_lib.kv_pool_register_split(ctypes.byref(layout), arr, instance_id, generation,
                                       ctypes.byref(out)))
    return out.value


def kv_pool_export(pool: int) -> kv_ipc_desc:
    """The pool as a kv_ipc_desc (IPC handle of its allocation, offset, size, identity) for
    another process."""
    d = kv_ipc_desc()
    _check(_lib.kv_pool_export(pool, ctypes.byref(d)))
    return d


def kv_pool_import(desc: kv_ipc_desc) -> int:
    """Maps a pool exported by another process (one mapping per allocation, refcounted);
    returns its handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_pool_import(ctypes.byref(desc), ctypes.byref(out)))
    return out.value


def kv_pool_export_split(pool: int):
    """A split pool as (kv_ipc_desc, array of L x C kv_ipc_buffer): the allocation handle and
    offset of every layer buffer, for another process."""
    lay, _, _ = kv_pool_info(pool)
    nb = lay.num_layers * lay.num_comps
    d, bufs = kv_ipc_desc(), (kv_ipc_buffer * nb)()
    _check(_lib.kv_pool_export_split(pool, ctypes.byref(d), bufs, nb))
    return d, bufs


def kv_pool_import_split(desc: kv_ipc_desc, bufs) -> int:
    """Maps a split pool exported by another process (each distinct allocation once,
    refcounted); returns its handle."""
    arr = (kv_ipc_buffer * len(bufs))(*bufs)
    out = ctypes.c_void_p()
    _check(_lib.kv_pool_import_split(ctypes.byref(desc), arr, len(bufs), ctypes.byref(out)))
    return out.value


def bufs_to_bytes(bufs) -> bytes:
    """An array of kv_ipc_buffer as bytes (to send to another process)."""
    return b"".join(ctypes.string_at(ctypes.addressof(b), ctypes.sizeof(b)) for b in bufs)


def bufs_from_bytes(b: bytes):
    """The kv_ipc_buffer entries bufs_to_bytes produced."""
    n = ctypes.sizeof(kv_ipc_buffer)
    if len(b) % n != 0:
        raise ValueError(f"buffer entries are {n} bytes each, got {len(b)} bytes")
    return [kv_ipc_buffer.from_buffer_copy(b[i:i + n]) for i in range(0, len(b), n)]


def kv_pool_close(pool: int) -> None:
    """Closes a pool handle (the last close of an imported allocation unmaps it)."""
    _check(_lib.kv_pool_close(pool))


def kv_pool_retire(instance_id: int, min_generation: int) -> None:
    """Refuses, from now on, pools of `instance_id` older than `min_generation` (KV_ERR_STALE)."""
    _check(_lib.kv_pool_retire(instance_id, min_generation))


def kv_pool_info(pool: int):
    """Returns (layout, device address of the pool, bytes) of a pool handle."""
    lay, ptr, nb = kv_layout(), ctypes.c_void_p(), ctypes.c_uint64()
    _check(_lib.kv_pool_info(pool, ctypes.byref(lay), ctypes.byref(ptr), ctypes.byref(nb)))
    return lay, ptr.value, nb.value


def desc_to_bytes(d: kv_ipc_desc) -> bytes:
    """The kv_ipc_desc as bytes (to send to another process)."""
    return ctypes.string_at(ctypes.addressof(d), ctypes.sizeof(d))


def desc_from_bytes(b: bytes) -> kv_ipc_desc:
    """A kv_ipc_desc from the bytes desc_to_bytes produced."""
    if len(b) != ctypes.sizeof(kv_ipc_desc):
        raise ValueError(f"descriptor must be {ctypes.sizeof(kv_ipc_desc)} bytes, got {len(b)}")
    return kv_ipc_desc.from_buffer_copy(b)


# --------------------------------------------------------------- host tier

def kv_host_register(host: int, nbytes: int, num_slots: int, host_heads: int,
                     pool_layout: kv_layout) -> int:
    """Registers a pinned, device-mapped host tier of `num_slots` page slots; returns its
    handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_host_register(host, nbytes, num_slots, host_heads, ctypes.byref(pool_layout),
                                 ctypes.byref(out)))
    return out.value


def kv_host_close(host: int) -> None:
    """Closes a host tier handle."""
    _check(_lib.kv_host_close(host))


# -------------------------------------------------------------- operations

def kv_backup(pool: int, host: int, src_pages, host_slots, stream=None) -> int:
    """BACKUP: host slot host_slots[i] <- page src_pages[i], every layer; enqueued on
    `stream`; returns the fence."""
    a, pa = _ids(src_pages)
    b, pb = _ids(host_slots)
    if a.size != b.size:
        raise ValueError("src_pages and host_slots differ in length")
    f = ctypes.c_uint64()
    _check(_lib.kv_backup(pool, host, pa, pb, a.size, stream, ctypes.byref(f)))
    return f.value


def kv_restore_layers(pool: int, host: int, host_slots, dst_pages, first_layer: int,
                      num_layers: int, stream=None) -> list:
    """One call, progressive per-layer fences (list of num_layers fences)."""
    a, pa = _ids(host_slots)
    b, pb = _ids(dst_pages)
    if a.size != b.size:
        raise ValueError("host_slots and dst_pages differ in length")
    fences = (ctypes.c_uint64 * max(1, num_layers))()
    _check(_lib.kv_restore_layers(pool, host, pa, pb, a.size, first_layer, num_layers, stream,
                                  fences))
    return list(fences[:num_layers])


def kv_backup_when_ready(pool: int, host: int, src_pages, host_slots, ready_word: int,
                         ready_value: int, ready_timeout_ns: int, stream=None) -> int:
    """BACKUP that starts on the GPU once the 64-bit word at `ready_word` reaches
    `ready_value` (bounded wait; on time-out it moves nothing and its fence reports ABORTED);
    returns the fence."""
    a, pa = _ids(src_pages)
    b, pb = _ids(host_slots)
    if a.size != b.size:
        raise ValueError("src_pages and host_slots differ in length")
    f = ctypes.c_uint64()
    _check(_lib.kv_backup_when_ready(pool, host, pa, pb, a.size, ready_word, ready_value,
                                     ready_timeout_ns, stream, ctypes.byref(f)))
    return f.value


def kv_restore_when_ready(pool: int, host: int, host_slots, dst_pages, ready_word: int,
                          ready_value: int, ready_timeout_ns: int, layer: int = -1,
                          stream=None) -> int:
    """RESTORE gated like kv_backup_when_ready on its host data having landed; returns the
    fence."""
    a, pa = _ids(host_slots)
    b, pb = _ids(dst_pages)
    if a.size != b.size:
        raise ValueError("host_slots and dst_pages differ in length")
    f = ctypes.c_uint64()
    _check(_lib.kv_restore_when_ready(pool, host, pa, pb, a.size, layer, ready_word, ready_value,
                                      ready_timeout_ns, stream, ctypes.byref(f)))
    return f.value


def kv_restore(pool: int, host: int, host_slots, dst_pages, layer: int = -1, stream=None) -> int:
    """RESTORE: page dst_pages[i] <- host slot host_slots[i], every layer (layer = -1) or one
    layer; returns the fence."""
    a, pa = _ids(host_slots)
    b, pb = _ids(dst_pages)
    if a.size != b.size:
        raise ValueError("host_slots and dst_pages differ in length")
    f = ctypes.c_uint64()
    _check(_lib.kv_restore(pool, host, pa, pb, a.size, layer, stream, ctypes.byref(f)))
    return f.value


def kv_device_gather(pool: int, buf: int, buf_bytes: int, buf_heads: int, src_pages,
                     stream=None, fence: bool = True) -> int:
    """Pool pages -> a device buffer in host-tier layout (HBM only); returns the fence
    (0 with fence=False: ordered by the stream only, no fence word)."""
    a, pa = _ids(src_pages)
    f = ctypes.c_uint64()
    _check(_lib.kv_device_gather(pool, buf, buf_bytes, buf_heads, pa, a.size, stream,
                                 ctypes.byref(f) if fence else None))
    return f.value


def kv_device_scatter(pool: int, buf: int, buf_bytes: int, buf_heads: int, dst_pages,
                      layer: int = -1, stream=None, fence: bool = True) -> int:
    """A device buffer in host-tier layout -> pool pages (every layer, or one); returns the
    fence (0 with fence=False: ordered by the stream only)."""
    a, pa = _ids(dst_pages)
    f = ctypes.c_uint64()
    _check(_lib.kv_device_scatter(pool, buf, buf_bytes, buf_heads, pa, a.size, layer, stream,
                                  ctypes.byref(f) if fence else None))
    return f.value


def kv_backup_staged_noalloc(pool: int, host: int, src_pages, host_slots, stream=None) -> None:
    """Allocation-free staged backup (see include/kvb.h); ordered on ``stream``, no fence."""
    a, pa = _ids(src_pages)
    b, pb = _ids(host_slots)
    if a.size != b.size:
        raise ValueError("src_pages and host_slots differ in length")
    _check(_lib.kv_backup_staged_noalloc(pool, host, pa, pb, a.size, stream))


def kv_op_validate(layout: kv_layout, num_slots: int, kind: int, a, b, layer: int = -1) -> int:
    """Returns the library's status for the op (does not raise for it); id lists of
    different lengths raise ValueError, as for the operations themselves."""
    a_, pa = _ids(a)
    b_, pb = _ids(b)
    if a_.size != b_.size:
        raise ValueError("the two id lists differ in length")
    return _lib.kv_op_validate(ctypes.byref(layout), num_slots, kind, pa, pb, a_.size, layer)


# ------------------------------------------------------------------ fences

def kv_fence_query(fence: int) -> int:
    """Status of a fence without waiting: KV_OK done, KV_ERR_TIMEOUT not yet, KV_ERR_ABORTED
    gave up."""
    return _lib.kv_fence_query(fence)


def kv_fence_wait(fence: int, timeout_ns: int = 60_000_000_000) -> None:
    """Waits (host) up to `timeout_ns` for a fence; raises KvError on time-out or abort."""
    _check(_lib.kv_fence_wait(fence, timeout_ns))


def kv_fence_stream_wait(fence: int, stream=None) -> None:
    """Makes `stream` wait on the GPU until the fence completes."""
    _check(_lib.kv_fence_stream_wait(fence, stream))


# --------------------------------------------------------------- utilities

def kv_config_get() -> kv_config:
    """The process-wide kv_config (mode, CTA cap, staging bytes, flags, CTA size)."""
    c = kv_config()
    _check(_lib.kv_config_get(ctypes.byref(c)))
    return c


def kv_config_set(mode: int = KV_MODE_ZERO_COPY, max_ctas: int = 0, staging_bytes: int = 0,
                  flags: int = 0, cta_threads: int = 0):
    """Sets the process-wide kv_config for operations issued afterwards."""
    _check(_lib.kv_config_set(ctypes.byref(kv_config(mode, max_ctas, staging_bytes, flags,
                                                     cta_threads))))


def kv_layout_page_bytes(layout: kv_layout) -> int:
    """Bytes of one page (L * C * T * H * B) of a layout."""
    out = ctypes.c_uint64()
    _check(_lib.kv_layout_page_bytes(ctypes.byref(layout), ctypes.byref(out)))
    return out.value


def kv_launch_count() -> int:
    """Kernels the library has launched so far (all devices)."""
    return _lib.kv_launch_count()


def kv_overlap_count() -> int:
    """Ops issued overlapped with the previous one on their stream so far."""
    return _lib.kv_overlap_count()


def kv_last_error() -> str:
    """Message of this thread's last failing call."""
    return _lib.kv_last_error().decode(errors="replace")


def kv_abi_version() -> int:
    """ABI version of the loaded library."""
    return _lib.kv_abi_version()


# ----------------------------------------------------------- descriptor ring

def make_ring_op(kind: int, a, b, pool_index: int = 0, layer: int = -1,
                 operation_id: int = 0, ready_index: int = 0, ready_value: int = 0,
                 ready_timeout_ms: int = 0) -> kv_ring_op:
    """A descriptor for the shared-memory ring: kind 0 BACKUP (a = pages, b = slots) or 1
    RESTORE (a = slots, b = pages).  ready_value != 0 gates it on ready word ready_index
    reaching that value (waited for on the GPU for at most ready_timeout_ms, 0 = 10 s)."""
    a_, _ = _ids(a)
    b_, _ = _ids(b)
    if a_.size != b_.size or a_.size > KV_RING_MAX_IDS:
        raise ValueError("id lists differ in length or exceed KV_RING_MAX_IDS")
    op = kv_ring_op()
    op.kind, op.pool_index, op.n, op.layer, op.operation_id = kind, pool_index, a_.size, layer, \
        operation_id
    op.ready_index, op.ready_value, op.ready_timeout_ms = ready_index, ready_value, \
        ready_timeout_ms
    ctypes.memmove(op.a, a_.ctypes.data, a_.nbytes) if a_.size else None
    ctypes.memmove(op.b, b_.ctypes.data, b_.nbytes) if b_.size else None
    return op


def kv_ring_create(name: str, slots: int) -> int:
    """Creates a named shared-memory descriptor ring of `slots` entries (the submitting side);
    returns its handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_ring_create(name.encode(), slots, ctypes.byref(out)))
    return out.value


def kv_ring_attach(name: str) -> int:
    """Attaches to a ring another process created (the serving side); returns its handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_ring_attach(name.encode(), ctypes.byref(out)))
    return out.value


def kv_ring_close(ring: int) -> None:
    """Closes a ring handle (the creator also unlinks the name)."""
    _check(_lib.kv_ring_close(ring))


def kv_ring_submit(ring: int, op: kv_ring_op, timeout_ns: int = 10_000_000_000) -> int:
    """Publishes a descriptor; returns its ticket (waits up to `timeout_ns` for a free slot)."""
    t = ctypes.c_uint64()
    _check(_lib.kv_ring_submit(ring, ctypes.byref(op), timeout_ns, ctypes.byref(t)))
    return t.value


def kv_ring_wait(ring: int, ticket: int, timeout_ns: int = 10_000_000_000) -> int:
    """Waits for a ticket; returns the operation's own status (raises on TIMEOUT etc.)."""
    s = ctypes.c_int()
    _check(_lib.kv_ring_wait(ring, ticket, timeout_ns, ctypes.byref(s)))
    return s.value


def kv_ring_serve(ring: int, pools, host: int, stream=None, max_ops: int = 1,
                  idle_timeout_ns: int = 1_000_000_000) -> int:
    """Serves up to `max_ops` descriptors through kv_backup / kv_restore on `stream`; the GPU
    completes each ticket; returns how many."""
    arr = (ctypes.c_void_p * max(1, len(pools)))(*pools)
    served = ctypes.c_uint32()
    _check(_lib.kv_ring_serve(ring, arr, len(pools), host, stream, max_ops, idle_timeout_ns,
                              ctypes.byref(served)))
    return served.value


def kv_ring_pop(ring: int, timeout_ns: int = 1_000_000_000):
    """Takes the next descriptor (server side); returns (ticket, op)."""
    op, t = kv_ring_op(), ctypes.c_uint64()
    _check(_lib.kv_ring_pop(ring, timeout_ns, ctypes.byref(op), ctypes.byref(t)))
    return t.value, op


def kv_ring_complete(ring: int, ticket: int, status: int = KV_OK) -> None:
    """Completes a ticket from the CPU with a status (server side)."""
    _check(_lib.kv_ring_complete(ring, ticket, status))


def kv_ring_serve_device(ring: int, pools, host: int, stream=None, max_ops: int = 1,
                         idle_timeout_ns: int = 1_000_000_000) -> int:
    """Starts the GPU-resident server on `stream`: it takes and moves up to `max_ops`
    descriptors (ending after `idle_timeout_ns` without one); returns the fence that completes
    when it has ended."""
    arr = (ctypes.c_void_p * max(1, len(pools)))(*pools)
    f = ctypes.c_uint64()
    _check(_lib.kv_ring_serve_device(ring, arr, len(pools), host, stream, max_ops,
                                     idle_timeout_ns, ctypes.byref(f)))
    return f.value


def kv_ring_ready_set(ring: int, index: int, value: int) -> None:
    """Sets ready word `index` of the ring to `value` from the CPU (either process)."""
    _check(_lib.kv_ring_ready_set(ring, index, value))


def kv_ring_ready_stream_set(ring: int, index: int, value: int, stream=None) -> None:
    """Sets ready word `index` to `value` from the GPU once the work before it on `stream`
    has finished."""
    _check(_lib.kv_ring_ready_stream_set(ring, index, value, stream))


def kv_ring_device_stop(ring: int) -> None:
    """Asks the ring's resident server to end before its next descriptor (returns at once)."""
    _check(_lib.kv_ring_device_stop(ring))


def kv_ring_device_result(ring: int):
    """(descriptors taken, server status) of the last resident server, once it has ended."""
    n, s = ctypes.c_uint32(), ctypes.c_int()
    _check(_lib.kv_ring_device_result(ring, ctypes.byref(n), ctypes.byref(s)))
    return n.value, s.value


# ------------------------------------------------------- L3 record store

def kv_l3_open(fd: int, base_offset: int, record_bytes: int, num_records: int,
               threads: int = 0) -> int:
    """An L3 record store over file descriptor `fd`: `num_records` records of `record_bytes`
    from `base_offset`; returns its handle."""
    out = ctypes.c_void_p()
    _check(_lib.kv_l3_open(fd, base_offset, record_bytes, num_records, threads,
                           ctypes.byref(out)))
    return out.value


def kv_l3_close(store: int) -> None:
    """Closes an L3 record store (stops its worker threads; the caller closes the fd)."""
    _check(_lib.kv_l3_close(store))


def kv_l3_put(store: int, host: int, host_slots: int, slots, records) -> None:
    """Host slots -> records; ``host`` is the address of the slot array."""
    a, pa = _ids(slots)
    b, pb = _ids(records)
    if a.size != b.size:
        raise ValueError("slots and records differ in length")
    _check(_lib.kv_l3_put(store, host, host_slots, pa, pb, a.size))


def kv_l3_get(store: int, host: int, host_slots: int, records, slots) -> None:
    """Records -> host slots."""
    a, pa = _ids(records)
    b, pb = _ids(slots)
    if a.size != b.size:
        raise ValueError("records and slots differ in length")
    _check(_lib.kv_l3_get(store, host, host_slots, pa, pb, a.size))


def kv_fault_inject(point: str, count: int = 1) -> None:
    """Arms a host-side fault point ("staging_alloc", "fence_reserve", "launch", "launch_nth",
    "ipc_open", "host_register"); count 0 disarms."""
    _check(_lib.kv_fault_inject(point.encode(), count))


def library():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib
