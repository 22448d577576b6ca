"""Pins of the oracle's indexer and top-k against brute force and closed forms."""
import itertools

import numpy as np
import pytest

from oracle import indexer_scores, indexer_scores_many, topk_select


def _loop_scores(keys, q):
    # plain Python double loop, the definition written out
    return [sum(int(a) * int(b) for a, b in zip(row, q)) for row in keys]


def test_indexer_matches_python_loop():
    rng = np.random.default_rng(1)
    for d in (4, 16, 64, 128):
        keys = rng.integers(-128, 128, size=(37, d), dtype=np.int8)
        q = rng.integers(-128, 128, size=d, dtype=np.int8)
        assert indexer_scores(keys, q).tolist() == _loop_scores(keys, q)


def test_indexer_closed_forms():
    q = np.arange(-64, 64, dtype=np.int8)
    keys = np.full((5, 128), 3, dtype=np.int8)
    assert (indexer_scores(keys, q) == 3 * int(q.astype(np.int64).sum())).all()
    # extreme magnitudes: -128 * -128 * d, and the int8 wrap must not happen
    keys = np.full((2, 128), -128, dtype=np.int8)
    qq = np.full(128, -128, dtype=np.int8)
    assert indexer_scores(keys, qq).tolist() == [128 * 128 * 128] * 2
    # one-hot query picks one key column
    keys = np.random.default_rng(2).integers(-127, 128, size=(9, 64), dtype=np.int8)
    e = np.zeros(64, dtype=np.int8)
    e[17] = 1
    assert indexer_scores(keys, e).tolist() == keys[:, 17].astype(int).tolist()


def test_indexer_float32_path_is_exact():
    rng = np.random.default_rng(3)
    keys = rng.integers(-128, 128, size=(4099, 128), dtype=np.int8)
    qs = rng.integers(-128, 128, size=(7, 128), dtype=np.int8)
    many = indexer_scores_many(keys, qs)
    for t in range(7):
        assert np.array_equal(many[:, t], indexer_scores(keys, qs[t]))
    # worst case magnitude: every partial sum still exact
    keys = np.full((3, 128), -128, dtype=np.int8)
    qs = np.full((1, 128), -128, dtype=np.int8)
    assert indexer_scores_many(keys, qs)[:, 0].tolist() == [2 ** 21] * 3


def _brute_topk(scores, k):
    """Enumerate every k-subset; keep the one where each member beats each
    non-member (higher score, or equal score and lower position)."""
    n = len(scores)
    k = min(k, n)
    found = []
    for sub in itertools.combinations(range(n), k):
        inside = set(sub)
        ok = all(scores[i] > scores[j] or (scores[i] == scores[j] and i < j)
                 for i in inside for j in range(n) if j not in inside)
        if ok:
            found.append(list(sub))
    assert len(found) == 1
    return found[0]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(4)
    for _ in range(300):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 10))
        s = rng.integers(-3, 4, size=n)        # few distinct values: many ties
        assert topk_select(s, k).tolist() == _brute_topk(s.tolist(), k)


def test_topk_special_cases():
    # all equal -> lowest positions
    assert topk_select(np.zeros(100, dtype=np.int64), 7).tolist() == list(range(7))
    # k >= N -> everything, ascending
    assert topk_select(np.array([5, -1, 9]), 8).tolist() == [0, 1, 2]
    # empty
    assert topk_select(np.array([], dtype=np.int64), 4).tolist() == []
    # strictly decreasing -> first k; strictly increasing -> last k
    assert topk_select(np.arange(50, 0, -1), 5).tolist() == [0, 1, 2, 3, 4]
    assert topk_select(np.arange(50), 5).tolist() == [45, 46, 47, 48, 49]
    # result is ascending and unique
    s = np.random.default_rng(5).integers(-1000, 1000, size=5000)
    sel = topk_select(s, 300)
    assert (np.diff(sel) > 0).all() and sel.size == 300
    thr = s[sel].min()
    assert (s[np.setdiff1d(np.arange(5000), sel)] <= thr).all()


@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_tie_at_threshold(k):
    s = np.array([5, 7, 7, 7, 1, 7])
    # one 7 cannot be excluded when k=3... the three lowest positions of the 7s
    expect = {1: [1], 2: [1, 2], 3: [1, 2, 3]}[k]
    assert topk_select(s, k).tolist() == expect
