"""Full-size workloads through the decode path the benchmark times (fused
append, the default fetch placement, the library's own launch shapes), against
the CPU oracle.

Every selection of every (request, layer, step) and every (request, layer)'s
hit and miss totals are compared bit-exactly; the page table, reverse map,
stamps, LRU order and counters after every step of sampled (request, layer)
pairs; attention outputs of sampled steps within the fp tolerance.  The
comparison replacement policies (FIFO, random) run at full batch size too.  The oracle
scores all positions in float32 BLAS, exact because every partial sum is an
integer below 2^24.
"""
import numpy as np
import pytest

import workload as wl
from oracle import FIFOHotCache, LRUHotCache, RandomHotCache, indexer_scores_many, sparse_attention, topk_select
from tests.harness import MAX_ABS, REL_L2, StepInputs, attention_error, make_cache, prefill, run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_int8_gb300.build import build
    build()
    yield


def check_full(w, steps, meta_pairs, attn_pairs, replacement="lru", seed=0):
    cache = make_cache(w, steps, replacement=replacement, replacement_seed=seed)
    prefill(cache, w)
    inp = StepInputs(w, steps)
    got = run_steps(cache, w, inp, steps, fused=True, meta_pairs=meta_pairs)
    n0 = w.contexts()
    checked_attn = 0
    for l in range(w.n_layers):
        for r in range(w.n_requests):
            keys = wl.idx_keys_upto(w, r, l, steps)
            scores = indexer_scores_many(keys, wl.query_walk(w, r, l, steps))
            if replacement == "random":
                lru = RandomHotCache(w.hot_slots, seed=seed, request=r, layer=l, n_layers=w.n_layers)
            else:
                lru = {"lru": LRUHotCache, "fifo": FIFOHotCache}[replacement](w.hot_slots)
            hits = misses = 0
            for t in range(steps):
                n = int(n0[r]) + t + 1
                sel = topk_select(scores[:n, t], w.top_k)
                st = lru.step(sel)
                hits += st["hits"]
                misses += st["misses"]
                g_sel = got["sel"][l, t][r]
                assert np.array_equal(g_sel[:sel.size], sel), f"selection r{r} l{l} t{t}"
                assert (g_sel[sel.size:] == -1).all()
                if (r, l) in meta_pairs:
                    page, rev, stamp, order, (length, step, h, m) = got["meta"][l, t][r]
                    o_page, o_rev, o_stamp, _ = lru.snapshot(n)
                    assert length == n and step == t + 1 and (h, m) == (hits, misses), f"counters r{r} l{l} t{t}"
                    assert np.array_equal(page, o_page), f"page table r{r} l{l} t{t}"
                    assert np.array_equal(rev, o_rev), f"reverse map r{r} l{l} t{t}"
                    assert np.array_equal(stamp, o_stamp), f"stamps r{r} l{l} t{t}"
                    assert order.tolist() == sorted(range(w.hot_slots), key=lambda s: (stamp[s], s))
                if (r, l) in attn_pairs:
                    ref = sparse_attention(wl.step_query(w, r, l, t), wl.kv_rows_at(w, r, l, sel), h_kv=w.h_kv,
                                           d_qk=w.d_qk, d_v=w.d_v, v_offset=w.v_offset)
                    ma, rel = attention_error(got["out"][l, t][r], ref)
                    assert ma <= MAX_ABS and rel <= REL_L2, f"attention r{r} l{l} t{t}: {ma} {rel}"
                    checked_attn += 1
            _, _, _, _, (length, step, h, m) = cache.snapshot(r, l, 1)
            assert (h, m) == (hits, misses), f"hit/miss totals r{r} l{l}"
    assert checked_attn > 0
    assert cache.stats()["device_error"] == 0
    cache.close()


def test_batch16_32k_full():
    w = wl.WORKLOADS["batch16_32k"]   # 16 requests x 4 layers x 32K, GQA 32/8, k 2048, B 4096
    check_full(w, 5, meta_pairs={(0, 0), (7, 2), (15, 3)}, attn_pairs={(0, 0), (9, 1), (15, 3)})


def test_mixed_8k_200k_full():
    w = wl.WORKLOADS["mixed_8k_200k"]   # 64 requests x 2 layers, 8K..200K log-uniform
    n0 = w.contexts()
    lo, hi = int(np.argmin(n0)), int(np.argmax(n0))
    check_full(w, 3, meta_pairs={(lo, 0), (hi, 1), (31, 0)}, attn_pairs={(lo, 1), (hi, 0), (5, 1)})


def test_stress_128k_smallest_B_full():
    w = wl.stress_point(2048, 0.3)   # 64 requests x 2 layers x 128K, B = k = 2048, low locality
    check_full(w, 3, meta_pairs={(0, 0), (63, 1)}, attn_pairs={(1, 0), (62, 1)})


def test_mla_128k_full():
    w = wl.WORKLOADS["mla_128k"]   # 32 requests x 2 layers x 128K, latent 576 / 512, 128 heads
    check_full(w, 3, meta_pairs={(0, 0), (31, 1)}, attn_pairs={(0, 1), (17, 0), (31, 1)})


@pytest.mark.parametrize("replacement", ["fifo", "random"])
def test_comparison_policies_full(replacement):
    # batch 16 x 4 layers x 32K with B a little above k and a fast-moving query, so
    # every step evicts and the policies choose among several hundred free slots
    w = wl.make_workload("batch16_32k", hot_slots=2304, sigma=0.3)
    check_full(w, 4, meta_pairs={(0, 0), (8, 2), (15, 3)}, attn_pairs={(3, 1), (15, 3)},
               replacement=replacement, seed=2026)
