"""Pins that tie the CPU oracle to something other than itself.

Every pin takes the loaded oracle library as ``lib`` so the same battery can be
run against builds of the oracle with a planted mistake
(``test_oracle_mutations.py``): each planted mistake must trip at least one pin.

What pins what:
  * ``pin_offsets_row_major`` -- the layout readings are row-major views with
    named axes; numpy's ``ravel_multi_index`` (a library routine) gives the
    offset of every unit, independently of the oracle's arithmetic.
  * ``pin_backup_tags`` / ``pin_restore_tags`` -- brute force over tiny pools:
    every unit carries a tag naming its own coordinates, written through a
    numpy view in the layout's axis order; after the oracle runs, every byte of
    the destination is checked unit by unit in Python loops (moved units carry
    the right tag, every other byte is unchanged).
  * ``pin_trtllm_view`` -- the TRT-LLM statement ([NB, NL, 2, NH*BS*HS] viewed as
    [NB, NL, 2, NH, BS, HS], kv_layout HND) from the LMCache page, as a golden
    fixture.
  * ``pin_numpy_restatement`` -- the whole operation restated with numpy
    transposes and fancy indexing on random bytes (``oracle/numpy_statement.py``,
    a second, independent statement of the same definition).
  * ``pin_invariants`` -- restore(backup(x)) is the identity, base+offset
    addressing, layer-by-layer restore equals whole-prefix restore, every device
    layout of the same logical KV gives the same host tier, threaded = serial.
  * ``pin_page_bytes`` -- bytes per page of the five workloads, written out by hand.
  * ``pin_l3_records`` -- the L3 record store: numpy fancy indexing over a
    [records, record_bytes] view of the file image restates put and get; a tiny
    store is checked byte by byte against tags naming (slot, byte); put then get
    into other slots returns the original pages; untouched records, slots and
    the bytes around the store are unchanged.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np

import oracle
from oracle import numpy_statement as nps

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# The numpy statement (oracle/numpy_statement.py, no code shared with the C
# oracle): named-axis layouts, views and the two operations.
DEV_AXES, HOST_AXES, LAYOUTS = nps.DEV_AXES, nps.HOST_AXES, nps.LAYOUTS
_shape, _dims = nps.shape, nps.dims
_pool_from_logical, _logical_from_pool = nps.pool_from_logical, nps.logical_from_pool
_logical_from_host, _host_from_logical = nps.logical_from_host, nps.host_from_logical
_np_backup, _np_restore = nps.backup, nps.restore


def _geom(L, C, P, T, H, B, order, dev, host):
    return oracle.geom(L, C, P, T, H, B, page_first=order, dev_hnd=dev, host_hnd=host)


def _tag(coord, B, marker):
    """B bytes naming a unit: its five coordinates, a marker, then a byte-index ramp."""
    v = np.empty(B, dtype=np.uint8)
    v[:5] = coord
    v[5] = marker
    v[6:] = (np.arange(6, B) * 29 + sum(coord)) & 0xFF
    return v


# ----------------------------------------------------------------------- pins

def pin_offsets_row_major(lib):
    dims = dict(L=2, C=2, P=3, T=4, H=5, B=16)
    S = 3
    for order, dev, hh in LAYOUTS:
        g = _geom(dims["L"], dims["C"], dims["P"], dims["T"], dims["H"], dims["B"], order, dev, hh)
        d = _dims(g, S)
        dshape = _shape(DEV_AXES[(order, dev)], d)
        hshape = _shape(HOST_AXES[hh], d)
        for p, l, c, t, h in itertools.product(range(g.P), range(g.L), range(g.C), range(g.T),
                                               range(g.H)):
            coord = {"p": p, "l": l, "c": c, "t": t, "h": h}
            want = np.ravel_multi_index(tuple(coord[a] for a in DEV_AXES[(order, dev)]), dshape)
            got = oracle.dev_offset(g, p, l, c, t, h, lib=lib)
            assert got == want * g.B, ("device offset", order, dev, (p, l, c, t, h), got, want)
        for s, l, c, t, h in itertools.product(range(S), range(g.L), range(g.C), range(g.T),
                                               range(g.H)):
            coord = {"s": s, "l": l, "c": c, "t": t, "h": h}
            want = np.ravel_multi_index(tuple(coord[a] for a in HOST_AXES[hh]), hshape)
            got = oracle.host_offset(g, s, l, c, t, h, lib=lib)
            assert got == want * g.B, ("host offset", hh, (s, l, c, t, h), got, want)


def _tagged_pool(g, order, dev, marker):
    axes = DEV_AXES[(order, dev)]
    arr = np.zeros(_shape(axes, _dims(g)) + (g.B,), dtype=np.uint8)
    for p, l, c, t, h in itertools.product(range(g.P), range(g.L), range(g.C), range(g.T),
                                           range(g.H)):
        coord = {"p": p, "l": l, "c": c, "t": t, "h": h}
        arr[tuple(coord[a] for a in axes)] = _tag((p, l, c, t, h), g.B, marker)
    return arr.reshape(-1)


def _tagged_host(g, S, hh, marker):
    axes = HOST_AXES[hh]
    arr = np.zeros(_shape(axes, _dims(g, S)) + (g.B,), dtype=np.uint8)
    for s, l, c, t, h in itertools.product(range(S), range(g.L), range(g.C), range(g.T),
                                           range(g.H)):
        coord = {"s": s, "l": l, "c": c, "t": t, "h": h}
        arr[tuple(coord[a] for a in axes)] = _tag((s, l, c, t, h), g.B, marker)
    return arr.reshape(-1)


def _id_lists(P, S):
    """Every single page and every ordered pair of distinct pages, with slot choices."""
    out = []
    for k in (1, 2):
        for pages in itertools.permutations(range(P), k):
            slots = tuple((S - 1 - j * 2 - pages[0]) % S for j in range(k))
            if len(set(slots)) == k:
                out.append((pages, slots))
    return out


def pin_backup_tags(lib):
    L, C, P, T, H, B, S = 2, 2, 4, 3, 2, 16, 3
    for order, dev, hh in LAYOUTS:
        g = _geom(L, C, P, T, H, B, order, dev, hh)
        pool = _tagged_pool(g, order, dev, marker=0x11)
        pool_before = pool.copy()
        haxes = HOST_AXES[hh]
        for pages, slots in _id_lists(P, S):
            host = np.full(S * L * C * T * H * B, 0xEE, dtype=np.uint8)
            oracle.backup(g, pool, host, pages, slots, lib=lib)
            harr = host.reshape(_shape(haxes, _dims(g, S)) + (B,))
            moved = dict(zip(slots, pages))
            for s, l, c, t, h in itertools.product(range(S), range(L), range(C), range(T),
                                                   range(H)):
                coord = {"s": s, "l": l, "c": c, "t": t, "h": h}
                got = harr[tuple(coord[a] for a in haxes)]
                if s in moved:
                    want = _tag((moved[s], l, c, t, h), B, 0x11)
                else:
                    want = np.full(B, 0xEE, dtype=np.uint8)
                assert np.array_equal(got, want), ("backup", order, dev, hh, pages, slots,
                                                   (s, l, c, t, h))
            assert np.array_equal(pool, pool_before), "backup wrote to the pool"


def pin_restore_tags(lib):
    L, C, P, T, H, B, S = 2, 2, 4, 3, 2, 16, 3
    for order, dev, hh in LAYOUTS:
        g = _geom(L, C, P, T, H, B, order, dev, hh)
        host = _tagged_host(g, S, hh, marker=0x22)
        host_before = host.copy()
        daxes = DEV_AXES[(order, dev)]
        for (pages, slots), layer in itertools.product(_id_lists(P, S), (-1, 0, L - 1)):
            pool = _tagged_pool(g, order, dev, marker=0x11)
            oracle.restore(g, pool, host, slots, pages, layer=layer, lib=lib)
            parr = pool.reshape(_shape(daxes, _dims(g)) + (B,))
            filled = dict(zip(pages, slots))
            for p, l, c, t, h in itertools.product(range(P), range(L), range(C), range(T),
                                                   range(H)):
                coord = {"p": p, "l": l, "c": c, "t": t, "h": h}
                got = parr[tuple(coord[a] for a in daxes)]
                if p in filled and (layer < 0 or l == layer):
                    want = _tag((filled[p], l, c, t, h), B, 0x22)
                else:
                    want = _tag((p, l, c, t, h), B, 0x11)
                assert np.array_equal(got, want), ("restore", order, dev, hh, pages, slots,
                                                   layer, (p, l, c, t, h))
            assert np.array_equal(host, host_before), "restore wrote to the host tier"


def pin_trtllm_view(lib):
    with open(os.path.join(GOLDEN, "trtllm_pool_view.json")) as f:
        fx = json.load(f)
    assert fx["kv_layout"] == "HND" and fx["six_d"] == ["NB", "NL", 2, "NH", "BS", "HS"]
    for case in fx["cases"]:
        NB, NL, NH, BS, HS, eb = (case[k] for k in ("NB", "NL", "NH", "BS", "HS", "elem_bytes"))
        dt = {1: np.uint8, 2: np.uint16}[eb]
        # the 4-D tensor as the adapter registers it, elements numbered in memory order
        four = np.arange(NB * NL * 2 * NH * BS * HS, dtype=np.int64).astype(dt).reshape(
            NB, NL, 2, NH * BS * HS)
        six = four.reshape(NB, NL, 2, NH, BS, HS)        # the server's view
        raw = four.reshape(-1).view(np.uint8)
        g = oracle.geom(NL, 2, NB, BS, NH, HS * eb, page_first=True, dev_hnd=True)
        for nb, nl, kv, nh, bs in itertools.product(range(NB), range(NL), range(2), range(NH),
                                                    range(BS)):
            off = oracle.dev_offset(g, nb, nl, kv, bs, nh, lib=lib)
            got = raw[off:off + HS * eb]
            want = np.ascontiguousarray(six[nb, nl, kv, nh, bs]).view(np.uint8)
            assert np.array_equal(got, want), ("trtllm view", case, (nb, nl, kv, nh, bs))


def pin_numpy_restatement(lib, seed=7):
    r = np.random.default_rng(seed)
    shapes = [(3, 2, 17, 5, 3, 32), (1, 1, 9, 1, 1, 48), (4, 2, 6, 2, 7, 16), (2, 1, 11, 8, 1, 64)]
    for (L, C, P, T, H, B), (order, dev, hh) in itertools.product(shapes, LAYOUTS):
        g = _geom(L, C, P, T, H, B, order, dev, hh)
        S = P + 2
        n = min(P, 5)
        pool = r.integers(0, 256, P * L * C * T * H * B, dtype=np.uint8)
        host = r.integers(0, 256, S * L * C * T * H * B, dtype=np.uint8)
        src = r.permutation(P)[:n].astype(np.int32)
        slots = r.permutation(S)[:n].astype(np.int32)
        want = _np_backup(pool, g, order, dev, host, S, hh, src, slots)
        got = host.copy()
        oracle.backup(g, pool, got, src, slots, lib=lib)
        assert np.array_equal(got, want), ("numpy backup", (L, C, P, T, H, B), order, dev, hh)
        dst = r.permutation(P)[:n].astype(np.int32)
        for layer in (-1, L - 1):
            want = _np_restore(pool, g, order, dev, host, S, hh, slots, dst, layer)
            got = pool.copy()
            oracle.restore(g, got, host, slots, dst, layer=layer, lib=lib)
            assert np.array_equal(got, want), ("numpy restore", (L, C, P, T, H, B), order, dev,
                                               hh, layer)


def pin_invariants(lib, seed=11):
    r = np.random.default_rng(seed)
    L, C, P, T, H, B = 3, 2, 12, 4, 3, 32
    S, n = 8, 6
    X = r.integers(0, 256, (P, L, C, T, H, B), dtype=np.uint8)   # one logical KV content
    src = r.permutation(P)[:n].astype(np.int32)
    slots = r.permutation(S)[:n].astype(np.int32)
    others = np.setdiff1d(np.arange(P), src)
    dst = r.permutation(others)[:n].astype(np.int32)
    hosts = {}
    for order, dev, hh in LAYOUTS:
        g = _geom(L, C, P, T, H, B, order, dev, hh)
        pool = _pool_from_logical(X, order, dev)
        base = pool.copy()
        host = np.full(S * g.L * g.C * g.T * g.H * g.B, 0x5A, dtype=np.uint8)
        oracle.backup(g, pool, host, src, slots, lib=lib)
        # the same logical content gives the same host tier whatever the device layout
        key = hh
        if key in hosts:
            assert np.array_equal(hosts[key], host), ("layout independence", order, dev, hh)
        hosts[key] = host.copy()
        # base + offset: the same pool at a byte offset inside a larger allocation
        for off in (16, 48, 4096 + 48):
            alloc = np.full(off + pool.size + 64, 0x77, dtype=np.uint8)
            alloc[off:off + pool.size] = pool
            h2 = np.full_like(host, 0x5A)
            oracle.backup(g, alloc, h2, src, slots, pool_offset=off, lib=lib)
            assert np.array_equal(h2, host), ("base+offset backup", off)
            oracle.restore(g, alloc, h2, slots, dst, pool_offset=off, lib=lib)
            assert (alloc[:off] == 0x77).all() and (alloc[off + pool.size:] == 0x77).all(), \
                ("restore wrote outside the pool", off)
        # restore(backup(x)) onto the source pages is the identity
        scribbled = pool.copy()
        Xs = _logical_from_pool(scribbled, g, order, dev)
        Xs[src] = 0xA5
        oracle.restore(g, scribbled, host, slots, src, lib=lib)
        assert np.array_equal(scribbled, base), ("round trip", order, dev, hh)
        # restore into other pages: those pages now hold the source pages' content
        moved = pool.copy()
        oracle.restore(g, moved, host, slots, dst, lib=lib)
        Xm = _logical_from_pool(moved, g, order, dev)
        assert np.array_equal(Xm[dst], X[src]), ("restore elsewhere", order, dev, hh)
        keep = np.setdiff1d(np.arange(P), dst)
        assert np.array_equal(Xm[keep], X[keep]), ("untouched pages", order, dev, hh)
        # layer by layer over every layer equals one whole-prefix restore
        lw = pool.copy()
        for layer in range(L):
            oracle.restore(g, lw, host, slots, dst, layer=layer, lib=lib)
        assert np.array_equal(lw, moved), ("layer-wise", order, dev, hh)
        # threaded runs equal serial ones
        hmt = np.full_like(host, 0x5A)
        oracle.backup(g, pool, hmt, src, slots, threads=3, lib=lib)
        assert np.array_equal(hmt, host), ("threaded backup", order, dev, hh)
        pmt = pool.copy()
        oracle.restore(g, pmt, host, slots, dst, threads=4, lib=lib)
        assert np.array_equal(pmt, moved), ("threaded restore", order, dev, hh)
    # NHD and HND host tiers hold the same units, token and head axes swapped
    Yn = _logical_from_host(hosts[0], _geom(L, C, P, T, H, B, 0, 0, 0), S, 0)
    Yh = _logical_from_host(hosts[1], _geom(L, C, P, T, H, B, 0, 0, 1), S, 1)
    assert np.array_equal(Yn, Yh), "host NHD vs HND"


def pin_page_bytes(lib):
    with open(os.path.join(GOLDEN, "workload_bytes.json")) as f:
        fx = json.load(f)
    for name, d in fx.items():
        if name == "citation":
            continue
        g = oracle.geom(d["L"], d["C"], 1, d["T"], d["H"], d["B"])
        assert oracle.page_bytes(g, lib=lib) == d["page_bytes"], name


def pin_l3_records(lib, seed=23):
    r = np.random.default_rng(seed)
    # (1) restated with numpy: the store is file[base : base + R*rb] viewed [R, rb]
    for rb, S, R, base, n in [(16, 5, 7, 0, 3), (48, 9, 12, 32, 9), (256, 4, 40, 4096 + 16, 4),
                              (64, 30, 30, 8, 30)]:
        host = r.integers(0, 256, S * rb, dtype=np.uint8)
        image = r.integers(0, 256, base + R * rb + 64, dtype=np.uint8)
        slots = r.integers(0, S, n).astype(np.int32)          # a put may read a slot twice
        records = r.permutation(R)[:n].astype(np.int32)
        want = image.copy()
        want[base:base + R * rb].reshape(R, rb)[records] = host.reshape(S, rb)[slots]
        got = image.copy()
        oracle.l3_put(host, rb, slots, records, got, base, lib=lib)
        assert np.array_equal(got, want), ("numpy put", rb, S, R, base, n)
        m = min(n, S)
        gslots = r.permutation(S)[:m].astype(np.int32)
        grecs = r.integers(0, R, m).astype(np.int32)          # a get may read a record twice
        wanth = host.copy()
        wanth.reshape(S, rb)[gslots] = image[base:base + R * rb].reshape(R, rb)[grecs]
        goth = host.copy()
        oracle.l3_get(image, rb, grecs, gslots, goth, base, lib=lib)
        assert np.array_equal(goth, wanth), ("numpy get", rb, S, R, base, m)
    # (2) brute force on a tiny store: every byte checked against its tag
    rb, S, R, base = 16, 3, 4, 5
    host = np.array([(s * 16 + b) & 0xFF for s in range(S) for b in range(rb)], dtype=np.uint8)
    for slots in itertools.permutations(range(S), 2):
        for records in itertools.permutations(range(R), 2):
            image = np.full(base + R * rb + 3, 0xEE, dtype=np.uint8)
            oracle.l3_put(host, rb, list(slots), list(records), image, base, lib=lib)
            for pos in range(image.size):
                rec, b = divmod(pos - base, rb)
                if pos >= base and rec < R and rec in records:
                    s = slots[records.index(rec)]
                    assert image[pos] == s * 16 + b, ("tag put", slots, records, pos)
                else:
                    assert image[pos] == 0xEE, ("untouched put", slots, records, pos)
            back = np.full(S * rb, 0xDD, dtype=np.uint8)
            oracle.l3_get(image, rb, list(records), list(slots[::-1]), back, base, lib=lib)
            for pos in range(back.size):
                s, b = divmod(pos, rb)
                if s in slots[::-1]:
                    rec = records[list(slots[::-1]).index(s)]
                    src = slots[records.index(rec)]
                    assert back[pos] == src * 16 + b, ("tag get", slots, records, pos)
                else:
                    assert back[pos] == 0xDD, ("untouched get", slots, records, pos)
    # (3) put then get into other slots returns the pages
    rb, S, R, n = 128, 10, 25, 5
    host = r.integers(0, 256, S * rb, dtype=np.uint8)
    image = np.zeros(R * rb, dtype=np.uint8)
    src = r.permutation(S)[:n].astype(np.int32)
    recs = r.permutation(R)[:n].astype(np.int32)
    oracle.l3_put(host, rb, src, recs, image, lib=lib)
    back = host.copy()
    dst = np.array([s for s in range(S) if s not in src][:n], dtype=np.int32)
    oracle.l3_get(image, rb, recs, dst, back, lib=lib)
    hv, bv = host.reshape(S, rb), back.reshape(S, rb)
    assert np.array_equal(bv[dst], hv[src]), "round trip through records"
    keep = np.setdiff1d(np.arange(S), dst)
    assert np.array_equal(bv[keep], hv[keep]), "slots not named stay unchanged"


ALL_PINS = [pin_offsets_row_major, pin_backup_tags, pin_restore_tags, pin_trtllm_view,
            pin_numpy_restatement, pin_invariants, pin_page_bytes, pin_l3_records]
