"""CPU checks of the test helpers that compare per-tile lists whatever the order of the lists
in the sorted array (the render path may lay the tiles' lists out in another order than the
tile ids)."""
import numpy as np
import pytest

from parity import assert_same_tile_lists, tile_lists_in_tile_order


def _lists(rng, tiles=50, max_len=9):
    lens = rng.integers(0, max_len, tiles)
    lists = [rng.integers(0, 1000, l).astype(np.uint32) for l in lens]
    return lists


def _pack(lists, tile_order):
    """Sorted array with the lists placed in tile_order, and the ranges by tile id."""
    ranges = np.zeros((len(lists), 2), np.uint32)
    out, at = [], 0
    for t in tile_order:
        ranges[t] = (at, at + len(lists[t]))
        out.append(lists[t])
        at += len(lists[t])
    return np.concatenate(out) if out else np.zeros(0, np.uint32), ranges


def test_tile_order_layout_does_not_matter():
    rng = np.random.default_rng(3)
    lists = _lists(rng)
    a, ra = _pack(lists, range(len(lists)))
    b, rb = _pack(lists, rng.permutation(len(lists)))
    assert_same_tile_lists(b, rb, a, ra)
    got, lens = tile_lists_in_tile_order(b, rb)
    np.testing.assert_array_equal(got, np.concatenate(lists))
    np.testing.assert_array_equal(lens, [len(l) for l in lists])


def test_a_changed_list_is_caught():
    rng = np.random.default_rng(4)
    lists = _lists(rng)
    a, ra = _pack(lists, range(len(lists)))
    t = next(i for i, l in enumerate(lists) if len(l) >= 2)
    swapped = [l.copy() for l in lists]
    swapped[t][[0, 1]] = swapped[t][[1, 0]]
    if np.array_equal(swapped[t], lists[t]):
        swapped[t][0] += 1
    b, rb = _pack(swapped, rng.permutation(len(lists)))
    with pytest.raises(AssertionError):
        assert_same_tile_lists(b, rb, a, ra)


def test_overlapping_or_gapped_ranges_are_caught():
    rng = np.random.default_rng(5)
    lists = _lists(rng)
    a, ra = _pack(lists, range(len(lists)))
    bad = ra.copy()
    t = next(i for i in range(len(lists)) if bad[i, 1] > bad[i, 0])
    bad[t, 0] += 1   # a gap before tile t's list
    with pytest.raises(AssertionError):
        tile_lists_in_tile_order(a, bad)
