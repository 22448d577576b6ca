"""Pins of the oracle's LRU hot cache and Belady bound.

* a hand-worked trace (tests/golden/lru_trace_b3.txt);
* the textbook paging example (tests/golden/paging_textbook.txt);
* exhaustive replay of every trace over tiny universes against a second
  formulation written here from the rule (a recency list, not stamps);
* cold misses = number of distinct positions when B covers them;
* misses never below Belady's MIN, and MIN equal to a brute-force optimum;
* structural invariants of page table / reverse map / stamps.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import LRUHotCache, belady_misses
from tests.conftest import GOLDEN


def _read_lru_golden():
    steps, page = [], None
    B = None
    for line in open(os.path.join(GOLDEN, "lru_trace_b3.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("B "):
            B = int(line.split()[1])
        elif line.startswith("page"):
            page = [int(x) for x in line.split()[1:]]
        else:
            f = [c.split() for c in line.split("|")]
            steps.append(dict(sel=[int(x) for x in f[1]], slots=[int(x) for x in f[2]],
                              hits=int(f[3][0]), misses=int(f[4][0]),
                              reverse=[int(x) for x in f[5]], stamp=[int(x) for x in f[6]]))
    return B, steps, page


def test_hand_worked_trace():
    B, steps, page = _read_lru_golden()
    c = LRUHotCache(B)
    for st in steps:
        r = c.step(st["sel"])
        assert r["slot_of_sel"].tolist() == st["slots"]
        assert (r["hits"], r["misses"]) == (st["hits"], st["misses"])
        pg, rev, stamp, _ = c.snapshot(len(page))
        assert rev.tolist() == st["reverse"]
        assert stamp.tolist() == st["stamp"]
    assert c.snapshot(len(page))[0].tolist() == page
    assert c.step_no == len(steps)


def _read_paging():
    d = {}
    for line in open(os.path.join(GOLDEN, "paging_textbook.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            d[k] = [int(x) for x in v]
    return d


def test_textbook_paging_example():
    d = _read_paging()
    frames = d["frames"][0]
    trace = [[r] for r in d["refs"]]
    assert belady_misses(trace, frames) == d["opt_faults"][0]
    c = LRUHotCache(frames)
    misses = sum(c.step(s)["misses"] for s in trace)
    assert misses == d["lru_faults"][0]


class RecencyListLRU:
    """Second formulation: slots kept in a list from least to most recently
    used (never-used slots first, in slot order).  A call moves the slots it
    used to the end, in slot order; victims are the first unpinned slots."""

    def __init__(self, B):
        self.order = list(range(B))
        self.pos_of = [-1] * B
        self.where = {}
        self.last = [-1] * B
        self.t = 0

    def step(self, sel):
        hits = {self.where[p] for p in sel if p in self.where}
        miss = [p for p in sorted(sel) if p not in self.where]
        free = [s for s in self.order if s not in hits][:len(miss)]
        for p, s in zip(miss, free):
            if self.pos_of[s] >= 0:
                self.where.pop(self.pos_of[s])
            self.pos_of[s] = p
            self.where[p] = s
        used = hits | set(free)
        self.order = [s for s in self.order if s not in used] + sorted(used)
        for s in used:
            self.last[s] = self.t
        self.t += 1
        return [self.where[p] for p in sorted(sel)], len(sel) - len(miss), len(miss)


def _all_traces(n_pos, max_k, T):
    subsets = [list(c) for r in range(0, max_k + 1) for c in itertools.combinations(range(n_pos), r)]
    return itertools.product(subsets, repeat=T)


@pytest.mark.parametrize("n_pos,B,T", [(4, 1, 4), (4, 2, 4), (5, 2, 3), (5, 3, 3), (6, 3, 3)])
def test_exhaustive_against_recency_list(n_pos, B, T):
    count = 0
    for trace in _all_traces(n_pos, B, T):
        a, b = LRUHotCache(B), RecencyListLRU(B)
        for sel in trace:
            ra = a.step(sel)
            sb, hb, mb = b.step(sel)
            assert ra["slot_of_sel"].tolist() == sb
            assert (ra["hits"], ra["misses"]) == (hb, mb)
            assert a.slot_pos == b.pos_of and a.slot_stamp == b.last
        count += 1
    assert count > 100


def _random_trace(rng, n_pos, k, T, walk=True):
    trace, cur = [], rng.choice(n_pos, size=k, replace=False)
    for _ in range(T):
        if walk:   # replace a few positions per step: locality like the pages describe
            keep = rng.random(k) > 0.2
            new = rng.choice(n_pos, size=k, replace=False)
            merged = list(dict.fromkeys(list(cur[keep]) + list(new)))[:k]
            cur = np.array(merged)
        else:
            cur = rng.choice(n_pos, size=k, replace=False)
        trace.append(sorted(int(x) for x in cur))
    return trace


def test_cold_misses_equal_distinct_when_cache_is_large():
    rng = np.random.default_rng(7)
    for _ in range(50):
        trace = _random_trace(rng, 60, 8, 12)
        distinct = len({p for s in trace for p in s})
        c = LRUHotCache(distinct + int(rng.integers(0, 5)))
        assert sum(c.step(s)["misses"] for s in trace) == distinct


def test_misses_never_below_belady():
    rng = np.random.default_rng(8)
    for _ in range(200):
        k = int(rng.integers(1, 6))
        B = k + int(rng.integers(0, 6))
        trace = _random_trace(rng, 30, k, 15, walk=bool(rng.integers(0, 2)))
        c = LRUHotCache(B)
        lru = sum(c.step(s)["misses"] for s in trace)
        assert lru >= belady_misses(trace, B)


def _brute_opt(seq, B):
    """Minimum misses over every demand-paging eviction choice (tiny inputs)."""
    best = [len(seq) + 1]

    def go(i, res, m):
        if m >= best[0]:
            return
        if i == len(seq):
            best[0] = m
            return
        p = seq[i]
        if p in res:
            go(i + 1, res, m)
        elif len(res) < B:
            go(i + 1, res | {p}, m + 1)
        else:
            for v in res:
                go(i + 1, (res - {v}) | {p}, m + 1)

    go(0, frozenset(), 0)
    return best[0]


def test_belady_equals_brute_force_optimum():
    rng = np.random.default_rng(9)
    for _ in range(300):
        n = int(rng.integers(2, 7))
        B = int(rng.integers(1, 4))
        seq = [int(x) for x in rng.integers(0, n, size=int(rng.integers(1, 11)))]
        assert belady_misses([[p] for p in seq], B) == _brute_opt(seq, B)


def test_invariants_on_random_walk():
    rng = np.random.default_rng(10)
    B, k = 16, 8
    c = LRUHotCache(B)
    for t, sel in enumerate(_random_trace(rng, 200, k, 60)):
        r = c.step(sel)
        page, rev, stamp, step = c.snapshot(200)
        assert step == t + 1
        for p in sel:                           # every selected row is resident
            assert page[p] >= 0
        assert (stamp[r["slot_of_sel"]] == t).all()
        for s in range(B):                      # reverse o page = identity
            if rev[s] >= 0:
                assert page[rev[s]] == s
        assert (page >= 0).sum() == (rev >= 0).sum() <= B
        assert len(set(page[page >= 0].tolist())) == (page >= 0).sum()
        assert ((rev < 0) == (stamp < 0)).all()


def test_k_equals_B_every_unhit_slot_is_a_victim():
    c = LRUHotCache(4)
    c.step([0, 1, 2, 3])
    r = c.step([2, 3, 4, 5])
    assert r["hits"] == 2 and r["misses"] == 2
    assert r["slot_of_sel"].tolist() == [2, 3, 0, 1]   # 2,3 keep slots 2,3; 4,5 take 0,1
    r = c.step([10, 11, 12, 13])
    assert r["misses"] == 4 and r["slot_of_sel"].tolist() == [0, 1, 2, 3]
