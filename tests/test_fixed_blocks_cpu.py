"""Pins of the oracle's fixed blocks (the deterministic baseline of the
fine-tuning experiment, Experimental validation): textbook grids and the
shift rule, independent of any library code."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("n,w", [(1, 1), (10, 3), (64, 32), (100, 7), (1000, 128), (50, 50), (50, 80)])
def test_one_grid_is_range(n, w):
    off, st = oracle.bins_fixed(n, [w], 1)
    assert list(off) == [0, len(st)]
    assert list(st) == list(range(0, n, w)) + [n]


@pytest.mark.parametrize("n,w,s", [(100, 7, 3), (257, 32, 4), (1000, 10, 10), (500, 3, 5), (64, 100, 2)])
def test_shifted_grids(n, w, s):
    off, st = oracle.bins_fixed(n, [w], s)
    for t in range(s):
        row = st[off[t]:off[t + 1]]
        o = t * w // s
        assert row[0] == 0 and row[-1] == n
        d = np.diff(row)
        assert (d > 0).all()                       # contiguous, strictly increasing
        inner = row[1:-1]
        if o > 0 and o < n:
            assert inner[0] == o                   # first block [0, o)
        # every start but 0 lies on the grid o + k w, and no grid point is missed
        grid = [x for x in range(o, n, w) if x > 0]
        assert list(inner) == grid
        if len(d) > 2:
            assert (d[1:-1] == w).all()            # interior blocks are full


def test_offsets_are_evenly_spaced():
    w, s = 20, 4
    off, st = oracle.bins_fixed(200, [w], s)
    firsts = [st[off[t] + 1] for t in range(s)]
    assert firsts == [20, 5, 10, 15]              # t = 0 starts its second block at w


def test_width_one_is_all_singletons():
    n = 37
    off, st = oracle.bins_fixed(n, [1, 1], 3)
    for hs in range(6):
        assert list(st[off[hs]:off[hs + 1]]) == list(range(n + 1))
