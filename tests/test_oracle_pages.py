"""Pins of the oracle's Quest-style page selection (pages of P positions, scored
by the upper bound that their per-dimension key minima and maxima give):

* a page of one position is that position: with P = 1 the page selection is
  the token-level top-k of the exact scores;
* the bound holds: every page's score is at least q . k of each of its keys,
  and equals it for a page that holds one key (brute force);
* a plain double loop reproduces the scores; the bounds of a page are the
  element-wise extremes of its keys, the last partial page included;
* ties go to the lower page, positions come out ascending and stop at N.
"""
import numpy as np

from oracle import indexer_scores, page_bounds, page_scores, page_select, topk_select


def test_page_of_one_position_is_the_token_selection():
    rng = np.random.default_rng(21)
    keys = rng.integers(-127, 128, size=(500, 64), dtype=np.int8)
    q = rng.integers(-127, 128, size=64, dtype=np.int8)
    pages, pos = page_select(keys, q, 1, 40)
    assert np.array_equal(pos, topk_select(indexer_scores(keys, q), 40))
    assert np.array_equal(pages, pos)


def test_the_bound_holds_and_is_tight_for_single_keys():
    rng = np.random.default_rng(22)
    keys = rng.integers(-128, 128, size=(333, 32), dtype=np.int8)
    q = rng.integers(-128, 128, size=32, dtype=np.int8)
    for P in (2, 8, 16):
        kmin, kmax = page_bounds(keys, P)
        U = page_scores(kmin, kmax, q)
        s = indexer_scores(keys, q)
        for j in range(U.size):
            blk = s[j * P:(j + 1) * P]
            assert U[j] >= blk.max()
            if blk.size == 1:
                assert U[j] == blk[0]


def test_plain_loop_scores_and_partial_last_page():
    rng = np.random.default_rng(23)
    keys = rng.integers(-128, 128, size=(37, 16), dtype=np.int8)
    q = rng.integers(-128, 128, size=16, dtype=np.int8)
    P = 8
    kmin, kmax = page_bounds(keys, P)
    assert kmin.shape == (5, 16)
    assert np.array_equal(kmin[4], keys[32:].min(axis=0)) and np.array_equal(kmax[4], keys[32:].max(axis=0))
    U = page_scores(kmin, kmax, q)
    for j in range(5):
        u = 0
        for d in range(16):
            u += max(int(q[d]) * int(kmin[j, d]), int(q[d]) * int(kmax[j, d]))
        assert U[j] == u


def test_ties_take_the_lower_page_and_positions_stop_at_n():
    keys = np.zeros((45, 16), np.int8)   # every bound is 0: all pages tie
    q = np.ones(16, np.int8)
    pages, pos = page_select(keys, q, 16, 32)
    assert pages.tolist() == [0, 1] and pos.tolist() == list(range(32))
    keys[40] = 5                          # the last (partial) page now leads
    pages, pos = page_select(keys, q, 16, 32)
    assert pages.tolist() == [0, 2] and pos.tolist() == list(range(16)) + list(range(32, 45))
