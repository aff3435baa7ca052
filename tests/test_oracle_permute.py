"""Oracle pins for the token permutation: sort-based brute force and invariants."""
import numpy as np

import oracle as O


def _brute(ids, E):
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    nvalid = int(valid.sum())
    sorted_assign = np.full(flat.size, -1, np.int64)
    sorted_assign[:nvalid] = order[:nvalid]
    offsets = np.concatenate([[0], np.cumsum(np.bincount(flat[valid], minlength=E))])
    pos = np.full(flat.size, -1, np.int64)
    pos[order[:nvalid]] = np.arange(nvalid)
    return offsets, sorted_assign, pos


def test_permute_matches_stable_sort():
    rng = np.random.default_rng(0)
    for T, k, E in [(1, 1, 1), (32, 2, 8), (37, 8, 256), (100, 3, 5), (0, 4, 16)]:
        ids = rng.integers(0, E, (T, k)).astype(np.int32)
        off, sa, pos, dropped = O.permute(ids, E)
        boff, bsa, bpos = _brute(ids, E)
        assert dropped == 0
        assert np.array_equal(off, boff) and np.array_equal(sa, bsa) and np.array_equal(pos, bpos)
        assert off[-1] == T * k and np.all(np.diff(off) >= 0)
        if T:
            assert np.array_equal(sa[pos], np.arange(T * k))


def test_permute_drops_out_of_range_ids():
    ids = np.array([[0, 5], [-1, 2], [7, 2]], np.int32)
    off, sa, pos, dropped = O.permute(ids, 6)
    assert dropped == 2
    assert list(pos) == [0, 3, -1, 1, -1, 2]
    assert list(off) == [0, 1, 1, 3, 3, 3, 4]
    assert list(sa) == [0, 3, 5, 1, -1, -1]


def test_permute_duplicate_ids_are_separate_assignments():
    ids = np.array([[3, 3, 3], [3, 1, 3]], np.int32)
    off, sa, pos, _ = O.permute(ids, 4)
    assert list(off) == [0, 0, 1, 1, 6]
    assert list(sa) == [4, 0, 1, 2, 3, 5]
