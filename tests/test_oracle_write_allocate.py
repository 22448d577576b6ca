"""Pins of the oracle's write-allocate variant (the token a decode call appends
counts as used by that call):

* a hand-worked trace (tests/golden/lru_write_allocate_b3.txt);
* exhaustive replay of every trace over tiny universes against a second
  formulation written here from the rule (a recency list, not stamps), for the
  LRU and FIFO rules;
* special cases: a selected new token is a plain miss (no alloc), so the
  variant equals write-around whenever every call selects its own token; every
  appended position is resident right after its call.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import FIFOHotCache, LRUHotCache
from tests.conftest import GOLDEN


def _read():
    steps, page, B = [], None, None
    for line in open(os.path.join(GOLDEN, "lru_write_allocate_b3.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("B "):
            B = int(line.split()[1])
        elif line.startswith("page"):
            page = [int(x) for x in line.split()[1:]]
        else:
            f = [c.split() for c in line.split("|")]
            steps.append(dict(app=int(f[1][0]), sel=[int(x) for x in f[2]], slots=[int(x) for x in f[3]],
                              hits=int(f[4][0]), misses=int(f[5][0]), allocs=int(f[6][0]),
                              reverse=[int(x) for x in f[7]], stamp=[int(x) for x in f[8]]))
    return B, steps, page


def test_hand_worked_trace():
    B, steps, page = _read()
    c = LRUHotCache(B)
    for st in steps:
        r = c.step(st["sel"], allocate=st["app"])
        assert r["slot_of_sel"].tolist() == st["slots"]
        assert (r["hits"], r["misses"], r["allocs"]) == (st["hits"], st["misses"], st["allocs"])
        _, rev, stamp, _ = c.snapshot(len(page))
        assert rev.tolist() == st["reverse"] and stamp.tolist() == st["stamp"]
    assert c.snapshot(len(page))[0].tolist() == page


class RecencyList:
    """Second formulation: slots from least to most recently used (never-used
    slots first, in slot order); a call's used set is its selection plus the
    token it appended; LRU moves every used slot to the end in slot order, FIFO
    only the filled ones; victims are the first unpinned slots of the list."""

    def __init__(self, B, fifo=False):
        self.order = list(range(B))
        self.pos_of = [-1] * B
        self.where = {}
        self.last = [-1] * B
        self.t = 0
        self.fifo = fifo

    def step(self, sel, new):
        want = sorted(set(sel) | {new})
        pinned = {self.where[p] for p in want if p in self.where}
        miss = [p for p in want if p not in self.where]
        free = [s for s in self.order if s not in pinned][:len(miss)]
        for p, s in zip(miss, free):
            if self.pos_of[s] >= 0:
                self.where.pop(self.pos_of[s])
            self.pos_of[s] = p
            self.where[p] = s
        moved = set(free) if self.fifo else pinned | set(free)
        self.order = [s for s in self.order if s not in moved] + sorted(moved)
        for s in moved:
            self.last[s] = self.t
        self.t += 1
        n_miss_sel = sum(1 for p in sel if p in miss)
        return [self.where[p] for p in sorted(sel)], len(sel) - n_miss_sel, n_miss_sel


@pytest.mark.parametrize("cls,fifo", [(LRUHotCache, False), (FIFOHotCache, True)])
@pytest.mark.parametrize("n_pos,B,T", [(3, 2, 3), (3, 3, 3), (4, 3, 3)])
def test_exhaustive_against_recency_list(cls, fifo, n_pos, B, T):
    # step t appends position n_pos + t and may select any positions up to it
    count = 0
    per_step = [[list(c) for r in range(0, B) for c in itertools.combinations(range(n_pos + t + 1), r)]
                for t in range(T)]
    for trace in itertools.product(*per_step):
        a, b = cls(B), RecencyList(B, fifo)
        for t, sel in enumerate(trace):
            new = n_pos + t
            ra = a.step(sel, allocate=new)
            sb, hb, mb = b.step(sel, new)
            assert ra["slot_of_sel"].tolist() == sb
            assert (ra["hits"], ra["misses"]) == (hb, mb)
            assert a.slot_pos == b.pos_of and a.slot_stamp == b.last
            assert new in a.page, "the appended token is resident after its call"
        count += 1
    assert count > 100


def test_selected_new_token_is_a_plain_miss():
    rng = np.random.default_rng(5)
    B, n0 = 6, 10
    wa, wr = LRUHotCache(B), LRUHotCache(B)
    for t in range(40):
        new = n0 + t
        others = rng.choice(new, size=int(rng.integers(0, B - 1)), replace=False)
        sel = sorted(set(int(x) for x in others) | {new})
        ra, rr = wa.step(sel, allocate=new), wr.step(sel)
        assert ra["allocs"] == 0
        assert ra["slot_of_sel"].tolist() == rr["slot_of_sel"].tolist()
        assert (ra["hits"], ra["misses"]) == (rr["hits"], rr["misses"])
    assert wa.slot_pos == wr.slot_pos and wa.slot_stamp == wr.slot_stamp
