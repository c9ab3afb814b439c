"""The persistent decode path's weighted split of the tile list, on the host.

The split kernel gives CTA c the tiles [starts[c], starts[c + 1]) and the merge
kernel picks, for every (sequence, KV head) row, the CTAs whose partials hold
that row's cold and hot tiles; both run the functions that the host hook
``tq_debug_split_plan`` runs here.  Checked: the ranges partition the list in
order; every tile lies in the range of the CTA its price puts it in; the merge
reads exactly the CTAs whose range meets a row part (a missing one drops tiles
from the softmax, an extra one reads a partial nobody wrote); and no CTA's load
(tiles plus the price of the segments it starts) exceeds an equal share by more
than one segment price.
"""
import numpy as np
import pytest

from bit_kv_cache_10_gb300 import native as N
from bit_kv_cache_10_gb300 import synth


def _list(tc, th, hkv):
    """Per tile: (row, part) in list order."""
    row, part = [], []
    for v in range(len(tc)):
        for h in range(hkv):
            r = v * hkv + h
            row += [r] * (tc[v] + th[v])
            part += [0] * tc[v] + [1] * th[v]
    return np.array(row, np.int64), np.array(part, np.int64)


def _check(tc, th, hkv, grid, kc=40, kh=40):
    tc = np.asarray(tc, np.int32)
    th = np.asarray(th, np.int32)
    starts, seg = N.tq_debug_split_plan(tc, th, hkv, grid, kc, kh)
    total = int(hkv * (tc.astype(np.int64) + th).sum())
    rows = len(tc) * hkv
    assert starts[0] == 0 and starts[grid] == total
    assert np.all(np.diff(starts) >= 0)
    row, part = _list(tc, th, hkv)
    cta = np.searchsorted(starts, np.arange(total), side="right") - 1  # CTA whose range holds tile t
    assert np.all((cta >= 0) & (cta < grid))
    # the price of tile t, from its definition: its index, kc per cold segment
    # and kh per hot segment started at or before it
    cost = np.arange(total) + kc * (row + 1) + kh * (row + part)
    C = total + (kc + kh) * rows
    if total:
        assert np.all(np.diff(cost) > 0) and cost[-1] < C
        np.testing.assert_array_equal(cta, cost * grid // C)
    # merge: exactly the CTAs that took tiles of each row part
    want = np.zeros((2 * rows, grid), np.uint8)
    want[2 * row + part, cta] = 1
    np.testing.assert_array_equal(seg, want)
    # load of each CTA: its tiles plus the price of every segment it starts (its first one included)
    seg_id = 2 * row + part
    load = np.zeros(grid)
    for c in range(grid):
        s = seg_id[starts[c]:starts[c + 1]]
        if len(s):
            u = np.unique(s)
            load[c] = len(s) + kc * np.count_nonzero(u % 2 == 0) + kh * np.count_nonzero(u % 2 == 1)
    assert load.max() <= C / grid + max(kc, kh) + 1 + 1e-9
    if kc == 0 and kh == 0:  # no prices: equal counts of tiles, ceil(c total / grid) onwards
        np.testing.assert_array_equal(starts, -(-np.arange(grid + 1) * total // grid))
    return starts, load


@pytest.mark.parametrize("seed", range(12))
def test_random_lists(seed):
    rng = np.random.default_rng(seed)
    nv = int(rng.integers(1, 40))
    hkv = int(rng.integers(1, 9))
    grid = int(rng.choice([1, 2, 7, 64, 152, 200]))
    tc = rng.integers(0, 300, nv)
    th = rng.integers(0, 17, nv)
    tc[rng.random(nv) < 0.2] = 0  # sequences without cold tiles, or empty ones
    th[rng.random(nv) < 0.2] = 0
    kc, kh = (int(x) for x in rng.choice([0, 1, 7, 40, 300], 2))
    _check(tc, th, hkv, grid, kc, kh)


def test_fewer_tiles_than_ctas_and_empty_lists():
    _check([0], [0], 1, 152)
    _check([0, 0, 0], [0, 0, 0], 8, 7)
    _check([1], [0], 1, 152)
    _check([0, 3], [1, 0], 2, 152)
    _check([5, 0, 2], [1, 1, 0], 4, 1)
    # fewer price units than CTAs: consecutive prices of a row skip CTAs
    _check([10], [0], 1, 152)
    _check([7], [5], 1, 152)
    _check([3, 9], [2, 4], 1, 200)
    _check([3, 9], [2, 4], 1, 200, 0, 0)
    _check([0, 0], [0, 0], 3, 5, 0, 0)
    _check([4, 0], [0, 2], 2, 3, 0, 0)


def test_long_context_decode_balance():
    """The long-context 3.5-bit decode: B4, 8 KV heads, lengths U[65536, 131072],
    256-token hot window, 152 CTAs.  An equal count of tiles per CTA left the
    CTAs that cross a row end with two segment starts more than the rest; the
    weighted split evens their loads."""
    lens = synth.seq_lengths(42, 4, 65536, 131072)
    W = 256
    ce = lens - np.minimum(W, lens)
    tc = (ce + 15) // 16
    th = (lens - ce + 15) // 16
    starts, load = _check(tc, th, 8, 152, 40, 40)
    assert load.max() / load.mean() < 1.01
    tiles = np.diff(starts)
    assert tiles.max() - tiles.min() >= 40  # CTAs that start extra segments take fewer tiles
