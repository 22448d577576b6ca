"""Quest-style page selection (page_size > 1) through the C ABI against the
oracle: the selected positions (every position of each selected page below the
length, ascending), per-step page hits and misses, the page table over pages,
the reverse map, stamps and order of the page slots, and the attention output
(max-abs <= 2e-2, relative L2 <= 5e-3 against fp64).  Covers partial last pages,
contexts shorter than k, appends through hs_append and through the decode call,
every fetch mode, the three replacement policies and ties between pages."""
import numpy as np
import pytest

import workload as wl
from oracle import FIFOHotCache, LRUHotCache, RandomHotCache, page_select, sparse_attention
from tests.harness import MAX_ABS, REL_L2, StepInputs, attention_error, make_cache, prefill, run_steps, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_int8_gb300.build import build
    build()
    yield


def page_cache(w, r, l, n_slots, replacement, seed):
    if replacement == "random":
        return RandomHotCache(n_slots, seed=seed, request=r, layer=l, n_layers=w.n_layers)
    return {"lru": LRUHotCache, "fifo": FIFOHotCache}[replacement](n_slots)


def page_oracle(w, r, l, steps, P, replacement="lru", seed=0):
    """Per step: (pages, positions, cache step result, cache snapshot over pages)."""
    keys = wl.idx_keys_upto(w, r, l, steps)
    walk = wl.query_walk(w, r, l, steps)
    cache = page_cache(w, r, l, w.hot_slots // P, replacement, seed)
    n0 = int(w.contexts()[r])
    out = []
    for t in range(steps):
        n = n0 + t + 1
        pages, pos = page_select(keys[:n], walk[t], P, w.top_k)
        st = cache.step(pages)
        out.append((pages, pos, st, cache.snapshot((n + P - 1) // P)))
    return out


def page_parity(w, steps, P, fetch_mode=2, fused=False, replacement="lru", seed=0):
    cache = make_cache(w, steps, fetch_mode=fetch_mode, replacement=replacement, replacement_seed=seed,
                       page_size=P)
    prefill(cache, w)
    inp = StepInputs(w, steps)
    got = run_steps(cache, w, inp, steps, collect_meta=True, fused=fused)
    BU = w.hot_slots // P
    for l in range(w.n_layers):
        for r in range(w.n_requests):
            prev_h = prev_m = 0
            for t, (pages, pos, st, snap) in enumerate(page_oracle(w, r, l, steps, P, replacement, seed)):
                g_sel = got["sel"][l, t][r]
                assert np.array_equal(g_sel[:pos.size], pos), f"selection r{r} l{l} t{t}"
                assert (g_sel[pos.size:] == -1).all()
                page, rev, stamp, order, (length, step, hits, misses) = got["meta"][l, t][r]
                assert length == int(w.contexts()[r]) + t + 1 and step == t + 1
                assert (hits - prev_h, misses - prev_m) == (st["hits"], st["misses"]), f"hit/miss r{r} l{l} t{t}"
                prev_h, prev_m = hits, misses
                o_page, o_rev, o_stamp, _ = snap
                n_pages = o_page.size
                assert np.array_equal(page[:n_pages], o_page), f"page table r{r} l{l} t{t}"
                assert (page[n_pages:] == -1).all()
                assert np.array_equal(rev[:BU], o_rev), f"reverse map r{r} l{l} t{t}"
                assert np.array_equal(stamp[:BU], o_stamp), f"stamps r{r} l{l} t{t}"
                assert order[:BU].tolist() == sorted(range(BU), key=lambda s: (stamp[s], s))
                ref = sparse_attention(wl.step_query(w, r, l, t), wl.kv_rows_at(w, r, l, pos), h_kv=w.h_kv,
                                       d_qk=w.d_qk, d_v=w.d_v, v_offset=w.v_offset)
                ma, rel = attention_error(got["out"][l, t][r], ref)
                assert ma <= MAX_ABS and rel <= REL_L2, f"attention r{r} l{l} t{t}: {ma} {rel}"
    st = cache.stats()
    assert st["device_error"] == 0
    cache.close()
    return got


@pytest.mark.parametrize("fetch_mode,fused", [(0, False), (1, False), (2, True), (1, True)])
def test_pages_of_16_match_the_oracle(fetch_mode, fused):
    # 3 requests x 2 layers, 5003 positions (a partial last page), d_idx 64,
    # k 256 = 16 pages, B 512 = 32 page slots
    w = wl.make_workload("tiny", n_requests=3, n_layers=2, context=5003, top_k=256, hot_slots=512, steps=6)
    page_parity(w, 6, 16, fetch_mode=fetch_mode, fused=fused)


def test_pages_of_64_with_wide_keys():
    # d_idx 128 (bounds rows of 256 bytes), k 512 = 8 pages, B 1024 = 16 page slots
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=9001, top_k=512, hot_slots=1024,
                         steps=5)
    page_parity(w, 5, 64, fused=True)


def test_pages_with_mixed_lengths_and_short_contexts():
    # contexts from 100 to 6000: some below k (every page attended), pages of 8
    w = wl.make_workload("mixed_8k_200k", n_requests=6, context_range=(100, 6000), top_k=256, hot_slots=384,
                         steps=4, d_idx=64)
    page_parity(w, 4, 8, fused=True)


@pytest.mark.parametrize("replacement,seed", [("fifo", 0), ("random", 0xBEEF)])
def test_pages_under_other_replacement_policies(replacement, seed):
    w = wl.make_workload("tiny", n_requests=2, n_layers=1, context=3000, top_k=128, hot_slots=256, steps=6)
    page_parity(w, 6, 16, replacement=replacement, seed=seed)


def test_page_ties_take_the_lower_pages():
    """Every key zero: every page bound is zero and all pages tie, so pages
    0 .. k/P - 1 are selected; one key made large moves its page in."""
    from tiered_kv_cache_int8_gb300 import HiSparseCache
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    P, K, n = 16, 64, 1000
    cache = HiSparseCache(n_layers=1, max_requests=1, max_context=2048, h_q=8, h_kv=1, d_qk=128, d_v=128,
                          d_idx=64, top_k=K, hot_slots=128, page_size=P)
    rows = torch.zeros((1, n, cache.row_elems), dtype=torch.int16, device=dev)
    keys = torch.zeros((1, n, 64), dtype=torch.int8, device=dev)
    keys[0, 999, :] = 3            # the last (partial) page holds the only non-zero key
    cache.append(0, rows, keys)
    q_idx = torch.ones((1, 64), dtype=torch.int8, device=dev)
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device=dev)
    sel = torch.full((1, K), -7, dtype=torch.int32, device=dev)
    cache.decode_layer(0, q_idx, q, sel_out=sel)
    got = sel.cpu().numpy()[0]
    want = list(range(0, 3 * P)) + list(range(62 * P, n))   # pages 0, 1, 2 and the partial page 62
    assert got[:len(want)].tolist() == want and (got[len(want):] == -1).all()
    assert cache.stats()["device_error"] == 0
    cache.close()
