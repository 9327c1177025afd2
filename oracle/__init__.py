"""CPU oracle for paged KV-cache backup / restore (ctypes wrapper of kv_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (the CUDA library and its Python binding) never imports it, and it never
imports the product: the two share no code.  Only the seeded input generators
(``hierarchical_kv_cache_backup_gb300.workloads``, which hold none of the
method's arithmetic) feed both.

The arithmetic lives in ``kv_oracle.c``; its header states the definition it
restates and the pages it follows.  This module only marshals numpy buffers.
``numpy_statement.py`` states the same definition a second time with numpy
views and fancy indexing, sharing no code with the C file (the tests pin one
against the other).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "kv_oracle.c")
LIB = os.path.join(_HERE, "libkv_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kv_oracle.c with gcc into a shared object next to it."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC",
                        "-pthread", "-o", tmp, SRC], check=True)
        os.replace(tmp, LIB)
    return LIB


class Geom(ctypes.Structure):
    """Mirror of ``kvo_geom`` in kv_oracle.c."""

    _fields_ = [("L", ctypes.c_int64), ("C", ctypes.c_int64), ("P", ctypes.c_int64),
                ("T", ctypes.c_int64), ("H", ctypes.c_int64), ("B", ctypes.c_int64),
                ("page_first", ctypes.c_int32), ("dev_hnd", ctypes.c_int32),
                ("host_hnd", ctypes.c_int32), ("pad_", ctypes.c_int32)]


def geom(L, C, P, T, H, B, page_first=False, dev_hnd=False, host_hnd=False) -> Geom:
    return Geom(L, C, P, T, H, B, int(bool(page_first)), int(bool(dev_hnd)),
                int(bool(host_hnd)), 0)


def _bind(lib):
    i64, i32, vp, gp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(Geom)
    lib.kvo_dev_offset.argtypes = [gp, i64, i64, i64, i64, i64]
    lib.kvo_dev_offset.restype = i64
    lib.kvo_host_offset.argtypes = [gp, i64, i64, i64, i64, i64]
    lib.kvo_host_offset.restype = i64
    lib.kvo_page_bytes.argtypes = [gp]
    lib.kvo_page_bytes.restype = i64
    lib.kvo_backup.argtypes = [gp, vp, i64, vp, vp, vp, i64]
    lib.kvo_backup.restype = None
    lib.kvo_restore.argtypes = [gp, vp, i64, vp, vp, vp, i64, i32]
    lib.kvo_restore.restype = None
    lib.kvo_backup_mt.argtypes = [gp, vp, i64, vp, vp, vp, i64, ctypes.c_int]
    lib.kvo_backup_mt.restype = ctypes.c_int
    lib.kvo_restore_mt.argtypes = [gp, vp, i64, vp, vp, vp, i64, i32, ctypes.c_int]
    lib.kvo_restore_mt.restype = ctypes.c_int
    lib.kvo_l3_put.argtypes = [vp, i64, vp, vp, i64, vp, i64]
    lib.kvo_l3_put.restype = None
    lib.kvo_l3_get.argtypes = [vp, i64, i64, vp, vp, i64, vp]
    lib.kvo_l3_get.restype = None


def load(path: str | None = None):
    """Load the oracle (building it first if needed); ``path`` loads another build."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _bind(lib)
        return lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            _bind(lib)
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ids(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def dev_offset(g: Geom, p, l, c, t, h, lib=None) -> int:
    return (lib or load()).kvo_dev_offset(ctypes.byref(g), p, l, c, t, h)


def host_offset(g: Geom, s, l, c, t, h, lib=None) -> int:
    return (lib or load()).kvo_host_offset(ctypes.byref(g), s, l, c, t, h)


def page_bytes(g: Geom, lib=None) -> int:
    return (lib or load()).kvo_page_bytes(ctypes.byref(g))


def backup(g: Geom, pool: np.ndarray, host: np.ndarray, src, slots, pool_offset: int = 0,
           threads: int = 1, lib=None) -> int:
    """host[slots[i]] <- pool[src[i]] in place.  ``pool`` is the whole allocation
    (uint8); the pool itself starts ``pool_offset`` bytes in.  Returns threads used."""
    lib = lib or load()
    src, slots = _ids(src), _ids(slots)
    assert src.shape == slots.shape and pool.dtype == np.uint8 and host.dtype == np.uint8
    if threads <= 1:
        lib.kvo_backup(ctypes.byref(g), _ptr(pool), pool_offset, _ptr(host), _ptr(src),
                       _ptr(slots), src.size)
        return 1
    return lib.kvo_backup_mt(ctypes.byref(g), _ptr(pool), pool_offset, _ptr(host), _ptr(src),
                             _ptr(slots), src.size, threads)


def restore(g: Geom, pool: np.ndarray, host: np.ndarray, slots, dst, layer: int = -1,
            pool_offset: int = 0, threads: int = 1, lib=None) -> int:
    """pool[dst[i]] <- host[slots[i]] in place (one layer if ``layer`` >= 0)."""
    lib = lib or load()
    slots, dst = _ids(slots), _ids(dst)
    assert slots.shape == dst.shape and pool.dtype == np.uint8 and host.dtype == np.uint8
    if threads <= 1:
        lib.kvo_restore(ctypes.byref(g), _ptr(pool), pool_offset, _ptr(host), _ptr(slots),
                        _ptr(dst), slots.size, layer)
        return 1
    return lib.kvo_restore_mt(ctypes.byref(g), _ptr(pool), pool_offset, _ptr(host),
                              _ptr(slots), _ptr(dst), slots.size, layer, threads)


def l3_put(host: np.ndarray, record_bytes: int, slots, records, file_image: np.ndarray,
           base: int = 0, lib=None) -> None:
    """file_image[base + records[i]*rb : +rb] <- host[slots[i]*rb : +rb] in place."""
    lib = lib or load()
    slots, records = _ids(slots), _ids(records)
    assert slots.shape == records.shape and host.dtype == np.uint8
    assert file_image.dtype == np.uint8
    lib.kvo_l3_put(_ptr(host), record_bytes, _ptr(slots), _ptr(records), slots.size,
                   _ptr(file_image), base)


def l3_get(file_image: np.ndarray, record_bytes: int, records, slots, host: np.ndarray,
           base: int = 0, lib=None) -> None:
    """host[slots[i]*rb : +rb] <- file_image[base + records[i]*rb : +rb] in place."""
    lib = lib or load()
    records, slots = _ids(records), _ids(slots)
    assert slots.shape == records.shape and host.dtype == np.uint8
    assert file_image.dtype == np.uint8
    lib.kvo_l3_get(_ptr(file_image), base, record_bytes, _ptr(records), _ptr(slots),
                   slots.size, _ptr(host))
