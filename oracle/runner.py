"""Replays a synthetic workload through the CPU oracle, one (request, layer) at a time.

TEST INFRASTRUCTURE (see ``hisparse_oracle``): used by the tests, the smoke
check and the benchmark's CPU-baseline leg only.

Per (request r, layer l) and decode step t = 0..T-1 (HiSparse summary, "论文1：
HiSparse"): the token of step t is appended first (position N0_r + t, index key
and K/V row from the generator), then every position < N0_r + t + 1 is scored,
the top-k selected, the LRU cache stepped, and attention taken over the selected
rows.  Requests and layers are independent: each (request, layer) has its own
cache and its own step counter.
"""
from __future__ import annotations

import numpy as np

import workload as wl

from .hisparse_oracle import (FIFOHotCache, LRUHotCache, RandomHotCache, belady_misses,
                              indexer_scores_many, sparse_attention, topk_select)


def replay_request_layer(w: wl.Workload, req: int, layer: int, steps: int | None = None, *,
                         attention_steps=None, kv_prefill: np.ndarray | None = None,
                         keep_trace: bool = True, replacement: str = "lru", seed: int = 0) -> dict:
    """Oracle results of decode steps 0..steps-1 of one (request, layer).

    attention_steps: None (no attention), "all", or an iterable of step numbers
    whose attention outputs are wanted (float64 [H_q, d_v]); replacement: "lru"
    (the pages' policy), "fifo" or "random" (their comparison policies; seed for
    the last)."""
    T = w.steps if steps is None else steps
    n0 = int(w.contexts()[req])
    keys = wl.idx_keys_upto(w, req, layer, T)
    walk = wl.query_walk(w, req, layer, T)
    scores = indexer_scores_many(keys, walk)           # [N0+T, T], exact integers
    if replacement == "random":
        cache = RandomHotCache(w.hot_slots, seed=seed, request=req, layer=layer, n_layers=w.n_layers)
    else:
        cache = {"lru": LRUHotCache, "fifo": FIFOHotCache}[replacement](w.hot_slots)
    if attention_steps == "all":
        att = set(range(T))
    elif attention_steps is None:
        att = set()
    else:
        att = set(int(t) for t in attention_steps)
    if att and kv_prefill is None:
        kv_prefill = wl.prefill_kv(w, req, layer)
    res = {"sel": [], "slot_of_sel": [], "hits": [], "misses": [], "out": {}}
    for t in range(T):
        n = n0 + t + 1
        sel = topk_select(scores[:n, t], w.top_k)
        st = cache.step(sel)
        if keep_trace:
            res["sel"].append(sel)
            res["slot_of_sel"].append(st["slot_of_sel"])
        res["hits"].append(st["hits"])
        res["misses"].append(st["misses"])
        if t in att:
            rows = np.empty((sel.size, w.row_elems), dtype=np.uint16)
            pre = sel < n0
            rows[pre] = kv_prefill[sel[pre]]
            for i in np.nonzero(~pre)[0]:
                rows[i] = wl.step_kv_row(w, req, layer, int(sel[i] - n0))
            q = wl.step_query(w, req, layer, t)
            res["out"][t] = sparse_attention(q, rows, h_kv=w.h_kv, d_qk=w.d_qk, d_v=w.d_v,
                                             v_offset=w.v_offset)
    res["cache"] = cache
    res["n_final"] = n0 + T
    return res


def belady_for(res: dict, n_slots: int) -> int:
    return belady_misses(res["sel"], n_slots)
