"""Paged KV-cache backup / restore restated with numpy views and fancy indexing.

TEST INFRASTRUCTURE ONLY, like the rest of this package: a second statement of
the definition that ``kv_oracle.c`` states with explicit loops, sharing no code
with it.  The tests pin the C oracle against it, and the benchmark's CPU
baseline times it single-threaded beside the C oracle.

The definition ("[RFC][HiCache] Out-of-process HiCache data plane with
device-memory IPC", §Device IPC data path: BACKUP and RESTORE move the KV of
named pages between the device pool and host slots; "[PP + HiCache] Add PP
Prefetch Tickets", §PP Prefetch Ticket Path: a restore may cover one layer):
view the pool as X[p, l, c, t, h, :] and the host tier as Y[s, l, c, t, h, :]
(B bytes per head vector), whatever their layouts in memory; then

  backup:  Y[slots[i]] = X[src[i]]                     for every item i
  restore: X[dst[i]] = Y[slots[i]]                     (all layers), or
           X[dst[i], layer] = Y[slots[i], layer]       (one layer)

Every layout is a row-major array whose axes come in the order named below;
page-first HND is the TRT-LLM pool [NB, NL, 2, NH, BS, HS] ("LMCache
RawCudaIPCWrapper深度解析", §在项目中的实际接入方式).
"""
from __future__ import annotations

import numpy as np

# (order, heads) -> axis names of the device pool, row-major, before the byte axis.
DEV_AXES = {
    (0, 0): ("l", "c", "p", "t", "h"),   # layer-first NHD
    (0, 1): ("l", "c", "p", "h", "t"),   # layer-first HND
    (1, 0): ("p", "l", "c", "t", "h"),   # page-first NHD
    (1, 1): ("p", "l", "c", "h", "t"),   # page-first HND  (TRT-LLM 6-D view)
}
# host-tier heads -> axis names of the host tier (slot-major, page-contiguous)
HOST_AXES = {0: ("s", "l", "c", "t", "h"), 1: ("s", "l", "c", "h", "t")}
LAYOUTS = [(o, d, hh) for (o, d) in DEV_AXES for hh in (0, 1)]


def shape(axes, dims):
    return tuple(dims[a] for a in axes)


def dims(g, S=None):
    """Axis sizes of geometry ``g`` (attributes L, C, P, T, H), with S host slots."""
    d = {"l": g.L, "c": g.C, "p": g.P, "t": g.T, "h": g.H}
    if S is not None:
        d["s"] = S
    return d


def pool_from_logical(X, order, dev):
    """X[p, l, c, t, h, :] -> flat pool bytes in the given device layout."""
    src_axes = ("p", "l", "c", "t", "h")
    perm = [src_axes.index(a) for a in DEV_AXES[(order, dev)]] + [5]
    return np.ascontiguousarray(X.transpose(perm)).reshape(-1)


def logical_from_pool(pool, g, order, dev):
    """Flat pool bytes -> the view X[p, l, c, t, h, :] (no copy)."""
    axes = DEV_AXES[(order, dev)]
    arr = pool.reshape(shape(axes, dims(g)) + (g.B,))
    perm = [axes.index(a) for a in ("p", "l", "c", "t", "h")] + [5]
    return arr.transpose(perm)


def logical_from_host(host, g, S, hh):
    """Flat host-tier bytes of S slots -> the view Y[s, l, c, t, h, :] (no copy)."""
    axes = HOST_AXES[hh]
    arr = host.reshape(shape(axes, dims(g, S)) + (g.B,))
    perm = [axes.index(a) for a in ("s", "l", "c", "t", "h")] + [5]
    return arr.transpose(perm)


def host_from_logical(Y, hh):
    """Y[s, l, c, t, h, :] -> flat host-tier bytes in the given head order."""
    src_axes = ("s", "l", "c", "t", "h")
    perm = [src_axes.index(a) for a in HOST_AXES[hh]] + [5]
    return np.ascontiguousarray(Y.transpose(perm)).reshape(-1)


def backup(pool, g, order, dev, host, S, hh, src, slots):
    """The host tier after BACKUP of pages ``src`` into ``slots`` (a new array)."""
    X = logical_from_pool(pool, g, order, dev)
    Y = logical_from_host(host, g, S, hh).copy()
    Y[np.asarray(slots)] = X[np.asarray(src)]
    return host_from_logical(Y, hh)


def restore(pool, g, order, dev, host, S, hh, slots, dst, layer):
    """The pool after RESTORE of ``slots`` into pages ``dst`` (a new array); layer -1 = all."""
    X = logical_from_pool(pool, g, order, dev).copy()
    Y = logical_from_host(host, g, S, hh)
    if layer < 0:
        X[np.asarray(dst)] = Y[np.asarray(slots)]
    else:
        X[np.asarray(dst), layer] = Y[np.asarray(slots), layer]
    return pool_from_logical(X, order, dev)
