"""Randomised checks of the oracle against the numpy restatement of the
definition (transposes and fancy indexing over named axes), over geometries,
layouts, id lists and layers drawn by hypothesis, beyond the fixed shapes of
the pin battery.  Skipped where hypothesis is not installed."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
import oracle_pins as pins  # noqa: E402


@st.composite
def cases(draw):
    L = draw(st.integers(1, 4))
    C = draw(st.integers(1, 2))
    P = draw(st.integers(1, 9))
    T = draw(st.integers(1, 5))
    H = draw(st.integers(1, 4))
    B = 16 * draw(st.integers(1, 3))
    order, dev, hh = draw(st.sampled_from(pins.LAYOUTS))
    S = draw(st.integers(1, P + 3))
    n = draw(st.integers(0, min(P, S)))
    src = draw(st.lists(st.integers(0, P - 1), min_size=n, max_size=n))           # may repeat
    slots = draw(st.permutations(list(range(S))))[:n]                              # distinct
    dst = draw(st.permutations(list(range(P))))[:n]                                # distinct
    layer = draw(st.sampled_from([-1] + list(range(L))))
    seed = draw(st.integers(0, 2**31 - 1))
    return (L, C, P, T, H, B, order, dev, hh, S, np.array(src, np.int32),
            np.array(slots, np.int32), np.array(dst, np.int32), layer, seed)


@settings(max_examples=150, deadline=None)
@given(cases())
def test_backup_and_restore_match_the_numpy_statement(case):
    L, C, P, T, H, B, order, dev, hh, S, src, slots, dst, layer, seed = case
    g = pins._geom(L, C, P, T, H, B, order, dev, hh)
    r = np.random.default_rng(seed)
    pool = r.integers(0, 256, P * L * C * T * H * B, dtype=np.uint8)
    host = r.integers(0, 256, S * L * C * T * H * B, dtype=np.uint8)
    want = pins._np_backup(pool, g, order, dev, host, S, hh, src, slots)
    got = host.copy()
    oracle.backup(g, pool, got, src, slots)
    assert np.array_equal(got, want)
    want = pins._np_restore(pool, g, order, dev, host, S, hh, slots, dst, layer)
    got = pool.copy()
    oracle.restore(g, got, host, slots, dst, layer=layer)
    assert np.array_equal(got, want)


@settings(max_examples=100, deadline=None)
@given(rb=st.sampled_from([16, 48, 64, 4096]), S=st.integers(1, 12), R=st.integers(1, 12),
       base=st.integers(0, 3).map(lambda k: 16 * k), data=st.data())
def test_l3_put_and_get_match_fancy_indexing(rb, S, R, base, data):
    n = data.draw(st.integers(0, min(S, R)))
    slots = np.array(data.draw(st.lists(st.integers(0, S - 1), min_size=n, max_size=n)), np.int32)
    recs = np.array(data.draw(st.permutations(list(range(R))))[:n], np.int32)
    r = np.random.default_rng(data.draw(st.integers(0, 2**31 - 1)))
    host = r.integers(0, 256, S * rb, dtype=np.uint8)
    image = r.integers(0, 256, base + R * rb + 8, dtype=np.uint8)
    want = image.copy()
    want[base:base + R * rb].reshape(R, rb)[recs] = host.reshape(S, rb)[slots]
    got = image.copy()
    oracle.l3_put(host, rb, slots, recs, got, base)
    assert np.array_equal(got, want)
    gslots = np.array(data.draw(st.permutations(list(range(S))))[:n], np.int32)
    back = host.copy()
    wantb = host.copy()
    wantb.reshape(S, rb)[gslots] = want[base:base + R * rb].reshape(R, rb)[recs]
    oracle.l3_get(want, rb, recs, gslots, back, base)
    assert np.array_equal(back, wantb)
