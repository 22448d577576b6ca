"""Pins of the oracle's FIFO hot cache (the comparison policy of the HiSparse
summary's miss-rate ablation).

* the textbook paging example (tests/golden/paging_textbook.txt: FIFO 15 faults);
* Belady's anomaly (tests/golden/paging_belady_anomaly.txt: FIFO 9 faults with
  3 frames, 10 with 4; LRU 10 and 8; the optimum 7 and 6), which also tells
  FIFO and LRU apart;
* exhaustive replay of every trace over tiny universes against a second
  formulation written here from the rule (an insertion queue, not stamps);
* misses never below Belady's MIN; FIFO = LRU on traces without hits;
* structural invariants, and hits keeping their fill stamp.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import FIFOHotCache, LRUHotCache, belady_misses
from tests.conftest import GOLDEN
from tests.test_oracle_lru import _random_trace


def _read(name):
    d = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            d[k] = [int(x) for x in v]
    return d


def _faults(cls, refs, frames):
    c = cls(frames)
    return sum(c.step([r])["misses"] for r in refs)


def test_textbook_paging_example():
    d = _read("paging_textbook.txt")
    assert _faults(FIFOHotCache, d["refs"], d["frames"][0]) == d["fifo_faults"][0]


def test_belady_anomaly():
    d = _read("paging_belady_anomaly.txt")
    refs = d["refs"]
    for f in (3, 4):
        assert _faults(FIFOHotCache, refs, f) == d[f"frames{f}_fifo"][0]
        assert _faults(LRUHotCache, refs, f) == d[f"frames{f}_lru"][0]
        assert belady_misses([[r] for r in refs], f) == d[f"frames{f}_opt"][0]


class InsertionQueueFIFO:
    """Second formulation: slots kept in a queue from the oldest fill to the
    newest (never-filled slots first, in slot order).  A call moves only the
    slots it filled to the back, in slot order; hits stay where they are;
    victims are the first unpinned slots of the queue."""

    def __init__(self, B):
        self.queue = list(range(B))
        self.pos_of = [-1] * B
        self.where = {}
        self.filled_at = [-1] * B
        self.t = 0

    def step(self, sel):
        hits = {self.where[p] for p in sel if p in self.where}
        miss = [p for p in sorted(sel) if p not in self.where]
        free = [s for s in self.queue if s not in hits][:len(miss)]
        for p, s in zip(miss, free):
            if self.pos_of[s] >= 0:
                self.where.pop(self.pos_of[s])
            self.pos_of[s] = p
            self.where[p] = s
        self.queue = [s for s in self.queue if s not in set(free)] + sorted(free)
        for s in free:
            self.filled_at[s] = self.t
        self.t += 1
        return [self.where[p] for p in sorted(sel)], len(sel) - len(miss), len(miss)


def _all_traces(n_pos, max_k, T):
    subsets = [list(c) for r in range(0, max_k + 1) for c in itertools.combinations(range(n_pos), r)]
    return itertools.product(subsets, repeat=T)


@pytest.mark.parametrize("n_pos,B,T", [(4, 1, 4), (4, 2, 4), (5, 2, 3), (5, 3, 3), (6, 3, 3)])
def test_exhaustive_against_insertion_queue(n_pos, B, T):
    count = 0
    for trace in _all_traces(n_pos, B, T):
        a, b = FIFOHotCache(B), InsertionQueueFIFO(B)
        for sel in trace:
            ra = a.step(sel)
            sb, hb, mb = b.step(sel)
            assert ra["slot_of_sel"].tolist() == sb
            assert (ra["hits"], ra["misses"]) == (hb, mb)
            assert a.slot_pos == b.pos_of and a.slot_stamp == b.filled_at
        count += 1
    assert count > 100


def test_misses_never_below_belady_and_equal_lru_without_hits():
    rng = np.random.default_rng(11)
    for _ in range(200):
        k = int(rng.integers(1, 6))
        B = k + int(rng.integers(0, 6))
        trace = _random_trace(rng, 30, k, 15, walk=bool(rng.integers(0, 2)))
        c = FIFOHotCache(B)
        assert sum(c.step(s)["misses"] for s in trace) >= belady_misses(trace, B)
    # every step selects positions never seen before: no hits, and the fill order
    # is the use order, so FIFO and LRU make the same choices
    for _ in range(50):
        B = int(rng.integers(1, 8))
        k = int(rng.integers(1, B + 1))
        trace = [list(range(t * k, (t + 1) * k)) for t in range(10)]
        a, b = FIFOHotCache(B), LRUHotCache(B)
        for s in trace:
            assert a.step(s)["slot_of_sel"].tolist() == b.step(s)["slot_of_sel"].tolist()
        assert a.slot_stamp == b.slot_stamp


def test_hits_keep_their_fill_stamp_and_invariants():
    c = FIFOHotCache(3)
    c.step([0, 1, 2])          # fills slots 0, 1, 2 at step 0
    r = c.step([0, 5])         # 0 hits (stays stamped 0); 5 evicts the oldest unpinned: slot 1
    assert r["slot_of_sel"].tolist() == [0, 1] and c.slot_stamp == [0, 1, 0]
    r = c.step([0, 9])         # LRU would now evict slot 2; FIFO evicts slot 2 too
    assert r["slot_of_sel"].tolist() == [0, 2] and c.slot_stamp == [0, 1, 2]
    r = c.step([7])            # slot 0 holds the oldest fill although it was just used
    assert r["slot_of_sel"].tolist() == [0] and c.slot_pos == [7, 5, 9]
    rng = np.random.default_rng(12)
    B, k = 16, 8
    c = FIFOHotCache(B)
    for t, sel in enumerate(_random_trace(rng, 200, k, 60)):
        r = c.step(sel)
        page, rev, stamp, step = c.snapshot(200)
        assert step == t + 1
        for p in sel:
            assert page[p] >= 0
        assert (stamp[r["slot_of_sel"]] <= t).all()
        assert all(stamp[v] == t for _, v in r["fills"])
        for s in range(B):
            if rev[s] >= 0:
                assert page[rev[s]] == s
        assert ((rev < 0) == (stamp < 0)).all()
