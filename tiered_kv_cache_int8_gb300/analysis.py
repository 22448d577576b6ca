"""Host-side analysis of a selection trace produced by the library: the offline
optimum's miss count (Belady's MIN), the floor the HiSparse summary ("论文1：
HiSparse") sets the replacement policies against (LRU 13.4 %, random 16.1 %,
FIFO 17.2 % against Belady 8.2 % at B = 4096).

A decode step selects a set of positions; the trace is serialised step by step,
ascending inside a step, and MIN evicts the resident position whose next use is
farthest (never again = farthest of all).  Any batched schedule of the same
trace is also a serial one, so this count is a lower bound for every policy.

Formulation: a forward queue of use times per position gives each reference's
next use as the queue's new head, and the resident positions are kept in a list
sorted by (next use, position), so the victim is always the list's last entry.
"""
from __future__ import annotations

from bisect import bisect_left, insort
from collections import deque


def belady_misses(steps, n_slots: int) -> int:
    """Misses of Belady's MIN with ``n_slots`` slots on the step-serialised trace.

    steps: iterable of iterables of positions (each step's selection)."""
    if n_slots < 1:
        raise ValueError("n_slots must be >= 1")
    refs = [p for s in steps for p in sorted(int(x) for x in s)]
    uses: dict[int, deque] = {}
    for t, p in enumerate(refs):
        uses.setdefault(p, deque()).append(t)
    horizon = len(refs)
    resident: list[tuple[int, int]] = []   # (next use, position), ascending
    key_of: dict[int, int] = {}            # resident position -> its next use
    misses = 0
    for p in refs:
        q = uses[p]
        q.popleft()                                   # this reference
        nxt = q[0] if q else horizon + p              # never again: beyond the trace, distinct
        if p in key_of:
            del resident[bisect_left(resident, (key_of[p], p))]
        else:
            misses += 1
            if len(key_of) == n_slots:
                _, victim = resident.pop()            # farthest next use
                del key_of[victim]
        insort(resident, (nxt, p))
        key_of[p] = nxt
    return misses
