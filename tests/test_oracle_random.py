"""Pins of the oracle's random-replacement hot cache (the other comparison
policy of the HiSparse summary's miss-rate ablation).

* the generator: SplitMix64's published outputs from state 0
  (tests/golden/splitmix64_state0.txt);
* never-filled slots are taken first; after that the victims are a uniformly
  random subset of the unpinned slots (frequency of each slot over many calls,
  chi-square bound), never a pinned slot, filled in ascending slot order;
* the victim set against a second formulation (numpy lexsort of the keys);
* misses never below Belady's MIN; cold misses only when B covers every position;
* k = B: every unhit slot is a victim; structural invariants.
"""
import os

import numpy as np

from oracle import LRUHotCache, RandomHotCache, belady_misses, splitmix64
from tests.conftest import GOLDEN
from tests.test_oracle_lru import _random_trace


def _golden():
    d = {}
    for line in open(os.path.join(GOLDEN, "splitmix64_state0.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            d[k] = int(v, 16)
    return d


def test_generator_matches_the_published_outputs():
    d = _golden()
    for n in (1, 2, 3):
        assert splitmix64(d["state"], n) == d[f"out{n}"]


def _cache(B, seed=7, request=3, layer=1, n_layers=4):
    return RandomHotCache(B, seed=seed, request=request, layer=layer, n_layers=n_layers)


def test_victims_are_the_smallest_keys_against_lexsort():
    rng = np.random.default_rng(20)
    for _ in range(100):
        B = int(rng.integers(2, 40))
        k = int(rng.integers(1, B + 1))
        c = _cache(B, seed=int(rng.integers(0, 2**32)))
        for t, sel in enumerate(_random_trace(rng, 3 * B, k, 6)):
            before = dict(c.page)
            filled = np.array(c.slot_pos) >= 0
            hits = {before[p] for p in sel if p in before}
            r = c.step(sel)
            free = np.array([s for s in range(B) if s not in hits], dtype=np.int64)
            keys = np.array([c.key(t, int(s)) if filled[s] else 0 for s in free], dtype=np.int64)
            order = np.lexsort((free, keys, filled[free]))   # never-filled first, then key, then slot
            want = sorted(free[order[:r["misses"]]].tolist())
            got = sorted(v for _, v in r["fills"])
            assert got == want
            # misses (ascending positions) fill the victims in ascending slot order
            assert [v for _, v in r["fills"]] == want
            assert not (set(got) & hits)


def test_victims_are_uniform_over_unpinned_slots():
    B, m = 16, 4
    c = _cache(B, seed=12345)
    c.step(list(range(B)))                   # fill every slot
    counts = np.zeros(B)
    pinned = {0, 1, 2, 3}
    T = 4000
    nxt = 1000
    for _ in range(T):
        # positions 0..3 stay selected (pinned in slots 0..3), plus m new ones
        sel = sorted([0, 1, 2, 3] + list(range(nxt, nxt + m)))
        nxt += m
        r = c.step(sel)
        for _, v in r["fills"]:
            counts[v] += 1
    assert counts[list(pinned)].sum() == 0
    free = [s for s in range(B) if s not in pinned]
    expect = T * m / len(free)
    chi2 = (((counts[free] - expect) ** 2) / expect).sum()
    assert chi2 < 40.0   # 11 degrees of freedom: P(chi2 > 40) < 1e-4


def test_misses_bounds_and_invariants():
    rng = np.random.default_rng(21)
    for _ in range(100):
        k = int(rng.integers(1, 6))
        B = k + int(rng.integers(0, 6))
        trace = _random_trace(rng, 30, k, 15, walk=bool(rng.integers(0, 2)))
        c = _cache(B, seed=int(rng.integers(0, 2**32)))
        assert sum(c.step(s)["misses"] for s in trace) >= belady_misses(trace, B)
    for _ in range(30):
        trace = _random_trace(rng, 60, 8, 12)
        distinct = len({p for s in trace for p in s})
        c = _cache(distinct + int(rng.integers(0, 5)))
        assert sum(c.step(s)["misses"] for s in trace) == distinct
    c = _cache(4)
    c.step([0, 1, 2, 3])
    r = c.step([2, 3, 4, 5])                 # k = B: the two unpinned slots are the victims
    assert sorted(v for _, v in r["fills"]) == [0, 1]
    c = _cache(16)
    for t, sel in enumerate(_random_trace(rng, 200, 8, 40)):
        r = c.step(sel)
        page, rev, stamp, step = c.snapshot(200)
        assert step == t + 1 and (stamp[r["slot_of_sel"]] == t).all()
        for p in sel:
            assert page[p] >= 0
        for s in range(16):
            if rev[s] >= 0:
                assert page[rev[s]] == s


def test_differs_from_lru():
    rng = np.random.default_rng(22)
    trace = _random_trace(rng, 400, 32, 30)
    a, b = _cache(48), LRUHotCache(48)
    sa = [a.step(s)["slot_of_sel"].tolist() for s in trace]
    sb = [b.step(s)["slot_of_sel"].tolist() for s in trace]
    assert sa != sb
