"""CUDA path against the CPU oracle, through the C ABI (binding in
tiered_kv_cache_int8_gb300.hs).

Bit-exact: selected positions, per-step hits and misses, page table, reverse
map, last-use stamps, step counters.  Attention: max-abs <= 2e-2 and relative
L2 <= 5e-3 against fp64.  Sizes span several tiles and ragged tails; the edge
cases (k >= N, empty request, ties, request subsets, bad ids, capacity, the
largest shapes: d_idx 256, k = B = 8192, B = 16384) are covered below; full-size
workloads are in test_gpu_full.py.
"""
import numpy as np
import pytest

import workload as wl
from oracle import (FIFOHotCache, LRUHotCache, RandomHotCache, indexer_scores_many, indexer_scores_multihead,
                    sparse_attention, topk_select)
from tests.harness import MAX_ABS, REL_L2, StepInputs, attention_error, make_cache, prefill, run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiered_kv_cache_int8_gb300.build import build
    build()
    yield


def oracle_cache(w, r, l, n_slots, replacement="lru", seed=0):
    if replacement == "random":
        return RandomHotCache(n_slots, seed=seed, request=r, layer=l, n_layers=w.n_layers)
    return {"lru": LRUHotCache, "fifo": FIFOHotCache}[replacement](n_slots)


def oracle_steps(w, r, l, steps, n_slots=None, replacement="lru", seed=0, write_allocate=False):
    """Per step: (sel, step result, snapshot) from the oracle (with write_allocate,
    the position each step appends counts as used by that step)."""
    keys = wl.idx_keys_upto(w, r, l, steps)
    if w.idx_heads > 1:   # the multi-head ReLU-weighted indexer
        heads = wl.query_walk_heads(w, r, l, steps)
        scores = np.stack([indexer_scores_multihead(keys, heads[t], wl.step_idx_weights(w, r, l, t))
                           for t in range(steps)], axis=1)
    else:
        scores = indexer_scores_many(keys, wl.query_walk(w, r, l, steps))
    cache = oracle_cache(w, r, l, n_slots or w.hot_slots, replacement, seed)
    n0 = int(w.contexts()[r])
    out = []
    for t in range(steps):
        n = n0 + t + 1
        sel = topk_select(scores[:n, t], w.top_k)
        st = cache.step(sel, allocate=n - 1 if write_allocate else None)
        out.append((sel, st, cache.snapshot(n)))
    return out


def oracle_attention(w, r, l, t, sel):
    rows = wl.kv_rows_at(w, r, l, sel)
    return sparse_attention(wl.step_query(w, r, l, t), rows, h_kv=w.h_kv, d_qk=w.d_qk, d_v=w.d_v,
                            v_offset=w.v_offset)


def check_order(order, stamp):
    keys = sorted(range(len(stamp)), key=lambda s: (stamp[s], s))
    assert order.tolist() == keys


def full_parity(w, steps, hot_slots=None, fetch_mode=2, fused=False, replacement="lru", seed=0,
                write_allocate=False):
    cache = make_cache(w, steps, hot_slots, fetch_mode=fetch_mode, replacement=replacement, replacement_seed=seed,
                       write_allocate=write_allocate)
    prefill(cache, w)
    inp = StepInputs(w, steps)
    got = run_steps(cache, w, inp, steps, collect_meta=True, fused=fused)
    B = hot_slots or w.hot_slots
    worst = (0.0, 0.0)
    for l in range(w.n_layers):
        for r in range(w.n_requests):
            prev_h = prev_m = 0
            for t, (sel, st, snap) in enumerate(oracle_steps(w, r, l, steps, B, replacement, seed,
                                                             write_allocate)):
                k_eff = sel.size
                g_sel = got["sel"][l, t][r]
                assert np.array_equal(g_sel[:k_eff], sel), f"selection r{r} l{l} t{t}"
                assert (g_sel[k_eff:] == -1).all()
                page, rev, stamp, order, (length, step, hits, misses) = got["meta"][l, t][r]
                assert length == int(w.contexts()[r]) + t + 1 and step == t + 1
                assert (hits - prev_h, misses - prev_m) == (st["hits"], st["misses"]), f"hit/miss r{r} l{l} t{t}"
                prev_h, prev_m = hits, misses
                o_page, o_rev, o_stamp, _ = snap
                assert np.array_equal(page, o_page), f"page table r{r} l{l} t{t}"
                assert np.array_equal(rev, o_rev), f"reverse map r{r} l{l} t{t}"
                assert np.array_equal(stamp, o_stamp), f"stamps r{r} l{l} t{t}"
                check_order(order, stamp)
                ref = oracle_attention(w, r, l, t, sel)
                ma, rel = attention_error(got["out"][l, t][r], ref)
                assert ma <= MAX_ABS and rel <= REL_L2, f"attention r{r} l{l} t{t}: {ma} {rel}"
                worst = (max(worst[0], ma), max(worst[1], rel))
    st = cache.stats()
    assert st["device_error"] == 0
    cache.close()
    return got, worst


def test_tiny_workload_every_step():
    # 1 request x 1 layer, context 4096 (+32), d_idx 64, k 256, B 512, 32 steps
    full_parity(wl.WORKLOADS["tiny"], 32)


@pytest.mark.parametrize("fetch_mode", [0, 1, 2])
def test_gqa_batch_ragged_small(fetch_mode):
    # several requests and layers, contexts not multiples of any tile, GQA 32/8
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=5003, top_k=256,
                         hot_slots=512, steps=6)
    full_parity(w, 6, fetch_mode=fetch_mode)


def test_mixed_lengths_small():
    w = wl.make_workload("mixed_8k_200k", n_requests=5, context_range=(300, 9000), top_k=256,
                         hot_slots=384, steps=5)
    full_parity(w, 5)


@pytest.mark.parametrize("h_q,h_kv", [(8, 8), (16, 2), (64, 4), (16, 1)])
def test_gqa_head_groupings(h_q, h_kv):
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=1500, h_q=h_q, h_kv=h_kv,
                         top_k=200, hot_slots=300, steps=3, d_idx=32)
    full_parity(w, 3)


@pytest.mark.parametrize("h_q,top_k,context", [(16, 200, 3001), (128, 256, 2600)])
def test_latent_rows_mla(h_q, top_k, context):
    # one shared 576-dim latent row per position, read as K and (first 512) as V;
    # k_eff not a multiple of the 64-row unit, several requests and layers
    w = wl.make_workload("mla_128k", n_requests=3, n_layers=2, context=context, h_q=h_q, top_k=top_k,
                         hot_slots=384, steps=4)
    full_parity(w, 4)


def test_latent_rows_short_context_and_fused_append():
    # contexts shorter than k (dense), the new token appended by the decode call
    w = wl.make_workload("mla_128k", n_requests=2, n_layers=1, context=150, h_q=32, top_k=256,
                         hot_slots=256, steps=3)
    full_parity(w, 3, fused=True)


def test_latent_rows_bit_identical_across_B():
    w = wl.make_workload("mla_128k", n_requests=2, n_layers=1, context=3000, h_q=64, top_k=256,
                         hot_slots=256, steps=3, sigma=0.3)
    outs = []
    for B in (256, 1024):
        cache = make_cache(w, 3, B)
        prefill(cache, w)
        outs.append(run_steps(cache, w, StepInputs(w, 3), 3))
        cache.close()
    for t in range(3):
        assert np.array_equal(outs[0]["out"][0, t], outs[1]["out"][0, t])
        assert np.array_equal(outs[0]["sel"][0, t], outs[1]["sel"][0, t])


def test_k_equals_B_and_high_sigma():
    # every unhit slot is a victim each step; low locality
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=3000, top_k=256,
                         hot_slots=256, steps=5, sigma=0.3)
    full_parity(w, 5)


def test_fetch_in_attention_matches_the_oracle():
    # fetch_mode 0: the attention kernel copies the missed rows (overlapped with HBM reads)
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=4100, top_k=256,
                         hot_slots=512, steps=4, sigma=0.3)
    full_parity(w, 4, fetch_mode=0)


@pytest.mark.parametrize("fetch_mode", [0, 1])
def test_append_fused_into_decode_matches_the_oracle(fetch_mode):
    # the new token rides on hs_decode_layer; it is selectable in the same step
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=2900, top_k=256,
                         hot_slots=512, steps=5)
    full_parity(w, 5, fetch_mode=fetch_mode, fused=True)


def test_fused_and_separate_append_are_bit_identical():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=5000, top_k=384,
                         hot_slots=512, steps=4, sigma=0.3)
    runs = []
    for fused in (False, True):
        cache = make_cache(w, 4)
        prefill(cache, w)
        runs.append(run_steps(cache, w, StepInputs(w, 4), 4, collect_meta=True, fused=fused))
        cache.close()
    for key in runs[0]["out"]:
        assert np.array_equal(runs[0]["out"][key], runs[1]["out"][key])
        assert np.array_equal(runs[0]["sel"][key], runs[1]["sel"][key])
        for a, b in zip(runs[0]["meta"][key], runs[1]["meta"][key]):
            for x, y in zip(a[:4], b[:4]):
                assert np.array_equal(x, y)
            assert a[4] == b[4]


def test_fetch_modes_are_bit_identical():
    # mode 2 pulls in RESOLVE on the cold first step (768 misses x 2 requests) and
    # leaves the few misses of later steps to the attention kernel
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=6000, top_k=768,
                         hot_slots=1024, steps=4, sigma=0.3)
    runs = []
    for mode in (0, 1, 2):
        cache = make_cache(w, 4, fetch_mode=mode)
        prefill(cache, w)
        runs.append(run_steps(cache, w, StepInputs(w, 4), 4, collect_meta=True))
        cache.close()
    for other in runs[1:]:
        for key in runs[0]["out"]:
            assert np.array_equal(runs[0]["out"][key], other["out"][key])
            assert np.array_equal(runs[0]["sel"][key], other["sel"][key])
            for a, b in zip(runs[0]["meta"][key], other["meta"][key]):
                for x, y in zip(a[:4], b[:4]):
                    assert np.array_equal(x, y)
                assert a[4] == b[4]


def test_output_bit_identical_across_B():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=4000, top_k=256,
                         hot_slots=256, steps=4)
    outs = []
    for B in (256, 512, 1024):
        cache = make_cache(w, 4, B)
        prefill(cache, w)
        outs.append(run_steps(cache, w, StepInputs(w, 4), 4))
        cache.close()
    for t in range(4):
        assert np.array_equal(outs[0]["out"][0, t], outs[1]["out"][0, t])
        assert np.array_equal(outs[0]["out"][0, t], outs[2]["out"][0, t])
        assert np.array_equal(outs[0]["sel"][0, t], outs[2]["sel"][0, t])


def test_repeated_runs_are_bit_identical():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=2500, top_k=256,
                         hot_slots=512, steps=3)
    runs = []
    for _ in range(2):
        cache = make_cache(w, 3)
        prefill(cache, w)
        runs.append(run_steps(cache, w, StepInputs(w, 3), 3))
        cache.close()
    for key in runs[0]["out"]:
        assert np.array_equal(runs[0]["out"][key], runs[1]["out"][key])


def test_context_shorter_than_k_is_dense():
    # k >= N: every position is selected (k_eff = N); the tail of sel_out is -1
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=100, top_k=256,
                         hot_slots=256, steps=3)
    full_parity(w, 3)


def test_ties_take_the_lowest_positions():
    import torch
    from tiered_kv_cache_int8_gb300 import HiSparseCache
    dev = torch.device("cuda", 0)
    R, N, d, k = 2, 3000, 64, 128
    cache = HiSparseCache(n_layers=1, max_requests=R, max_context=N + 4, h_q=4, h_kv=1, d_qk=128, d_v=128,
                          d_idx=d, top_k=k, hot_slots=k)
    kv = torch.randn(R, N, 256, device=dev).to(torch.bfloat16)
    keys = torch.full((R, N, d), 3, dtype=torch.int8, device=dev)
    keys[1, 2000:2010] = 4            # ten strictly higher scores, then ties
    cache.append(0, kv, keys)
    q_idx = torch.ones(R, d, dtype=torch.int8, device=dev)
    q = torch.randn(R, 4, 128, device=dev).to(torch.bfloat16)
    sel = torch.empty(R, k, dtype=torch.int32, device=dev)
    cache.decode_layer(0, q_idx, q, sel_out=sel)
    s = sel.cpu().numpy()
    assert s[0].tolist() == list(range(k))
    assert s[1].tolist() == sorted(list(range(k - 10)) + list(range(2000, 2010)))
    assert cache.stats()["device_error"] == 0
    cache.close()


def test_ties_through_the_candidate_list():
    # repeated calls: from the second one on the top-k works from the keys the
    # score kernel listed above the previous call's threshold, here all ties
    import torch
    from tiered_kv_cache_int8_gb300 import HiSparseCache
    dev = torch.device("cuda", 0)
    R, N, d, k = 2, 200, 32, 128
    cache = HiSparseCache(n_layers=1, max_requests=R, max_context=N + 4, h_q=4, h_kv=1, d_qk=128, d_v=128,
                          d_idx=d, top_k=k, hot_slots=k)
    kv = torch.randn(R, N, 256, device=dev).to(torch.bfloat16)
    keys = torch.full((R, N, d), 3, dtype=torch.int8, device=dev)
    keys[1, 150:157] = 4              # seven strictly higher scores, then ties
    cache.append(0, kv, keys)
    q_idx = torch.ones(R, d, dtype=torch.int8, device=dev)
    q = torch.randn(R, 4, 128, device=dev).to(torch.bfloat16)
    for _ in range(3):
        sel = torch.empty(R, k, dtype=torch.int32, device=dev)
        cache.decode_layer(0, q_idx, q, sel_out=sel)
        s = sel.cpu().numpy()
        assert s[0].tolist() == list(range(k))
        assert s[1].tolist() == sorted(list(range(k - 7)) + list(range(150, 157)))
    assert cache.stats()["device_error"] == 0
    cache.close()


def test_context_above_the_one_pass_limit():
    # 300K positions: the top-k takes its rescan path (more than 256K positions)
    w = wl.make_workload("tiny", context=300_000, top_k=256, hot_slots=512, steps=3, d_idx=16)
    full_parity(w, 3)


def test_request_subset_and_order():
    import torch
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=1, context=2000, top_k=128,
                         hot_slots=256, steps=2)
    cache = make_cache(w, 2)
    prefill(cache, w)
    dev = torch.device("cuda", 0)
    ids = torch.tensor([2, 0], dtype=torch.int32, device=dev)
    kv = torch.from_numpy(np.stack([wl.step_kv_row(w, r, 0, 0) for r in (2, 0)])[:, None].view(np.int16)).to(dev)
    keys = torch.from_numpy(np.stack([wl.step_idx_key(w, r, 0, 0) for r in (2, 0)])[:, None]).to(dev)
    cache.append(0, kv, keys, req_ids=ids)
    q_idx = torch.from_numpy(np.stack([wl.query_walk(w, r, 0, 1)[0] for r in (2, 0)])).to(dev)
    q = torch.from_numpy(np.stack([wl.step_query(w, r, 0, 0) for r in (2, 0)]).view(np.int16)).to(dev)
    sel = torch.empty(2, w.top_k, dtype=torch.int32, device=dev)
    out = cache.decode_layer(0, q_idx, q, sel_out=sel, req_ids=ids)
    for i, r in enumerate((2, 0)):
        o_sel, o_st, _ = oracle_steps(w, r, 0, 1)[0]
        assert np.array_equal(sel[i].cpu().numpy(), o_sel)
        ref = oracle_attention(w, r, 0, 0, o_sel)
        ma, rel = attention_error(out[i].view(torch.int16).cpu().numpy().view(np.uint16), ref)
        assert ma <= MAX_ABS and rel <= REL_L2
    assert cache.snapshot(1, 0, 1)[4][:2] == (2000, 0)     # request 1 untouched
    assert cache.snapshot(2, 0, 1)[4][:2] == (2001, 1)
    cache.close()


def test_empty_request_and_bad_ids_set_error_bits():
    import torch
    from tiered_kv_cache_int8_gb300 import HiSparseCache, hs
    dev = torch.device("cuda", 0)
    cache = HiSparseCache(n_layers=1, max_requests=2, max_context=64, h_q=4, h_kv=1, d_qk=128, d_v=128,
                          d_idx=16, top_k=8, hot_slots=8)
    q_idx = torch.ones(1, 16, dtype=torch.int8, device=dev)
    q = torch.ones(1, 4, 128, device=dev).to(torch.bfloat16)
    out = torch.full((1, 4, 128), 7.0, device=dev).to(torch.bfloat16)
    cache.decode_layer(0, q_idx, q, out=out)                 # request 0 has no positions
    assert (out.float() == 0).all()
    assert cache.stats()["device_error"] == hs.HS_DEVERR_EMPTY
    cache.close()
    cache = HiSparseCache(n_layers=1, max_requests=2, max_context=64, h_q=4, h_kv=1, d_qk=128, d_v=128,
                          d_idx=16, top_k=8, hot_slots=8)
    bad = torch.tensor([5], dtype=torch.int32, device=dev)
    cache.append(0, torch.zeros(1, 1, 256, dtype=torch.bfloat16, device=dev),
                 torch.zeros(1, 1, 16, dtype=torch.int8, device=dev), req_ids=bad)
    cache.decode_layer(0, q_idx, q, req_ids=bad)
    assert cache.stats()["device_error"] & hs.HS_DEVERR_REQ_RANGE
    cache.close()


def test_append_past_capacity_is_rejected_whole():
    import torch
    from tiered_kv_cache_int8_gb300 import HiSparseCache, hs
    dev = torch.device("cuda", 0)
    cache = HiSparseCache(n_layers=1, max_requests=2, max_context=40, h_q=4, h_kv=1, d_qk=128, d_v=128,
                          d_idx=16, top_k=8, hot_slots=8)
    cache.append(0, torch.zeros(2, 30, 256, dtype=torch.bfloat16, device=dev),
                 torch.zeros(2, 30, 16, dtype=torch.int8, device=dev))
    cache.append(0, torch.zeros(1, 20, 256, dtype=torch.bfloat16, device=dev),
                 torch.zeros(1, 20, 16, dtype=torch.int8, device=dev))
    assert cache.stats()["device_error"] == hs.HS_DEVERR_CAPACITY
    assert cache.snapshot(0, 0, 1)[4][0] == 30 and cache.snapshot(1, 0, 1)[4][0] == 30
    with pytest.raises(hs.HsError):
        cache.append(0, torch.zeros(1, 41, 256, dtype=torch.bfloat16, device=dev),
                     torch.zeros(1, 41, 16, dtype=torch.int8, device=dev))
    cache.close()


def test_reset_request_recycles_the_id():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=2, context=1800, top_k=128,
                         hot_slots=256, steps=2)
    cache = make_cache(w, 2)
    prefill(cache, w)
    run_steps(cache, w, StepInputs(w, 2), 2, collect_out=False)
    cache.reset_request(1)
    page, rev, stamp, order, sc = cache.snapshot(1, 1, 1800)
    assert sc == (0, 0, 0, 0) and (page == -1).all() and (rev == -1).all() and (stamp == -1).all()
    assert order.tolist() == list(range(256))
    assert cache.snapshot(0, 1, 1)[4][1] == 2
    cache.close()


def test_graph_capture_replays_the_same_step():
    import torch
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=3000, top_k=256,
                         hot_slots=512, steps=3)
    inp = StepInputs(w, 3)
    eager = make_cache(w, 3)
    prefill(eager, w)
    ref = run_steps(eager, w, inp, 3)
    eager.close()

    cache = make_cache(w, 3)
    prefill(cache, w)
    dev = torch.device("cuda", 0)
    q_idx = inp.q_idx[0, 0].clone()
    q = inp.q[0, 0].clone()
    kv = inp.kv[0, 0].clone()
    keys = inp.keys[0, 0].clone()
    out = torch.empty(2, w.h_q, w.d_v, dtype=torch.bfloat16, device=dev)
    sel = torch.empty(2, w.top_k, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cache.append(0, kv, keys, stream=s)
            cache.decode_layer(0, q_idx, q, out=out, sel_out=sel, stream=s)
    torch.cuda.synchronize()
    # capture enqueues nothing: the cache is still at step 0
    assert cache.snapshot(0, 0, 1)[4][:2] == (3000, 0)
    for t in range(3):
        q_idx.copy_(inp.q_idx[0, t])
        q.copy_(inp.q[0, t])
        kv.copy_(inp.kv[0, t])
        keys.copy_(inp.keys[0, t])
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(sel.cpu().numpy(), ref["sel"][0, t])
        assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"][0, t])
    assert cache.stats()["device_error"] == 0
    cache.close()


@pytest.mark.parametrize("fetch_mode", [0, 1, 2])
def test_fifo_replacement_matches_the_oracle(fetch_mode):
    # the pages' comparison policy: only fills renew a slot's stamp; B close to k
    # and a fast-moving query so hits and evictions mix every step
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=4100, top_k=256,
                         hot_slots=320, steps=6, sigma=0.3)
    full_parity(w, 6, fetch_mode=fetch_mode, replacement="fifo")


def test_fifo_latent_rows_and_fused_append():
    w = wl.make_workload("mla_128k", n_requests=2, n_layers=1, context=2600, h_q=32, top_k=256,
                         hot_slots=320, steps=4, sigma=0.3)
    full_parity(w, 4, fused=True, replacement="fifo")


def test_replacement_policy_changes_placement_not_the_result():
    # LRU, FIFO and random put rows in different slots and miss differently; the
    # selection and the attention output are bit-identical
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=6000, top_k=512,
                         hot_slots=640, steps=6, sigma=0.3)
    runs = []
    for rep in ("lru", "fifo", "random"):
        cache = make_cache(w, 6, replacement=rep, replacement_seed=99)
        prefill(cache, w)
        runs.append(run_steps(cache, w, StepInputs(w, 6), 6, collect_meta=True))
        cache.close()
    for other in runs[1:]:
        differ = False
        for key in runs[0]["out"]:
            assert np.array_equal(runs[0]["out"][key], other["out"][key])
            assert np.array_equal(runs[0]["sel"][key], other["sel"][key])
            for a, b in zip(runs[0]["meta"][key], other["meta"][key]):
                differ |= not np.array_equal(a[1], b[1])   # reverse maps
        assert differ, "another policy should place rows differently on this trace"


@pytest.mark.parametrize("fetch_mode,seed", [(1, 0), (2, 0xC0FFEE)])
def test_random_replacement_matches_the_oracle(fetch_mode, seed):
    # the pages' other comparison policy: victims by a counter-based hash (same
    # generator on both sides); several requests and layers, so the counter's
    # request and layer fields matter
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=4100, top_k=256,
                         hot_slots=320, steps=6, sigma=0.3)
    full_parity(w, 6, fetch_mode=fetch_mode, replacement="random", seed=seed)


def test_random_replacement_large_cache_and_latent_rows():
    # B = 4 k (most victims are free slots at first, then random among filled ones)
    w = wl.make_workload("mla_128k", n_requests=2, n_layers=1, context=2600, h_q=32, top_k=128,
                         hot_slots=512, steps=6, sigma=0.3)
    full_parity(w, 6, fused=True, replacement="random", seed=5)


def test_widest_index_keys_and_largest_selection():
    # the largest shapes the kernels take: d_idx 256 (16 key chunks per position),
    # top_k 8192 with k = B (every unhit slot a victim), fused append of a 256-byte key
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=20000, d_idx=256, top_k=8192,
                         hot_slots=8192, steps=3, sigma=0.3)
    full_parity(w, 3, fused=True)


@pytest.mark.parametrize("replacement", ["lru", "random"])
def test_largest_hot_cache_keeps_the_reverse_map_in_global_memory(replacement):
    # B = 16384 leaves no room for the reverse map in RESOLVE's shared memory, so
    # eviction (and the random policy's never-filled test) read it from HBM
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=40000, top_k=2048,
                         hot_slots=16384, steps=4, sigma=0.3)
    full_parity(w, 4, replacement=replacement, seed=3)


@pytest.mark.parametrize("fetch_mode,replacement", [(0, "lru"), (1, "lru"), (2, "fifo"), (2, "random")])
def test_write_allocate_matches_the_oracle(fetch_mode, replacement):
    # the token each call appends counts as used by the call (the oracle's
    # write-allocate variant); page table, reverse map, stamps, order and
    # counters bit-exact after every step, attention within tolerance
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=3000, top_k=256, hot_slots=320,
                         steps=8, sigma=0.3)
    full_parity(w, 8, fetch_mode=fetch_mode, fused=True, replacement=replacement, write_allocate=True)


def test_write_allocate_changes_placement_not_the_result():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=2500, top_k=128, hot_slots=200,
                         steps=6, sigma=0.2)
    outs = []
    for wa in (False, True):
        cache = make_cache(w, 6, write_allocate=wa)
        prefill(cache, w)
        outs.append(run_steps(cache, w, StepInputs(w, 6), 6, fused=True))
        cache.close()
    for t in range(6):
        assert np.array_equal(outs[0]["sel"][0, t], outs[1]["sel"][0, t])
        assert np.array_equal(outs[0]["out"][0, t], outs[1]["out"][0, t])


def test_write_allocate_needs_a_free_slot():
    from tiered_kv_cache_int8_gb300 import hs
    w = wl.make_workload("batch16_32k", n_requests=1, n_layers=1, context=300, top_k=128, hot_slots=128, steps=1)
    with pytest.raises(hs.HsError) as e:
        make_cache(w, 1, write_allocate=True)
    assert e.value.status == hs.HS_ERR_CONFIG


@pytest.mark.parametrize("d_idx,heads", [(128, 4), (64, 8), (128, 2)])
def test_multihead_indexer_matches_the_oracle(d_idx, heads):
    # s[p] = sum_h w_h * max(0, q_h . K[p]) with 32-bit keys: selection, cache
    # state and attention against the oracle's multi-head scores
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=1, context=3001, top_k=256, hot_slots=512,
                         steps=5, d_idx=d_idx, idx_heads=heads, sigma=0.2)
    full_parity(w, 5, fused=True)


def test_multihead_indexer_ties_and_short_contexts():
    # all-zero weights: every score ties at 0, so the lowest positions win
    import torch
    from tiered_kv_cache_int8_gb300 import hs
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=700, top_k=256, hot_slots=512,
                         steps=1, d_idx=64, idx_heads=4)
    cache = make_cache(w, 1)
    prefill(cache, w)
    inp = StepInputs(w, 1)
    qi = inp.q_idx[0, 0].clone()
    qi[:, 4 * 64:4 * 64 + 4] = 0
    sel = torch.full((2, 256), -7, dtype=torch.int32, device="cuda")
    cache.decode_layer(0, qi, inp.q[0, 0], sel_out=sel, new_kv=inp.kv[0, 0], new_keys=inp.keys[0, 0])
    assert np.array_equal(sel.cpu().numpy(), np.tile(np.arange(256, dtype=np.int32), (2, 1)))
    assert cache.stats()["device_error"] == 0
    cache.close()


def _shared_selection_oracle(w, steps, share, write_allocate=False):
    """Per (request, layer, step): (sel, step result, snapshot) when every layer
    reuses its group lead's selection of the same step (lead = layer - layer % share)."""
    out = {}
    for r in range(w.n_requests):
        n0 = int(w.contexts()[r])
        leads = {}
        for lead in range(0, w.n_layers, share):
            keys = wl.idx_keys_upto(w, r, lead, steps)
            sc = indexer_scores_many(keys, wl.query_walk(w, r, lead, steps))
            leads[lead] = [topk_select(sc[:n0 + t + 1, t], w.top_k) for t in range(steps)]
        for l in range(w.n_layers):
            cache = LRUHotCache(w.hot_slots)
            for t in range(steps):
                sel = leads[l - l % share][t]
                st = cache.step(sel, allocate=n0 + t if write_allocate else None)
                out[r, l, t] = (sel, st, cache.snapshot(n0 + t + 1))
    return out


@pytest.mark.parametrize("share,prefetch,fetch_mode,wa", [(2, True, 2, False), (4, True, 0, True),
                                                           (2, False, 0, False), (4, False, 1, False)])
def test_shared_selection_matches_the_oracle(share, prefetch, fetch_mode, wa):
    # layers of a group reuse the lead's selection; with prefetch the lead's call
    # resolves the followers and pulls their rows ahead, without it each follower
    # resolves at its own call: same selections, cache state and outputs
    steps = 6
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=4, context=3000, top_k=256, hot_slots=384,
                         steps=steps, sigma=0.3)
    cache = make_cache(w, steps, fetch_mode=fetch_mode, write_allocate=wa, index_share=share,
                       share_prefetch=prefetch)
    prefill(cache, w)
    got = run_steps(cache, w, StepInputs(w, steps), steps, collect_meta=True, fused=True)
    ref = _shared_selection_oracle(w, steps, share, wa)
    for l in range(w.n_layers):
        for r in range(w.n_requests):
            prev_h = prev_m = 0
            for t in range(steps):
                sel, st, snap = ref[r, l, t]
                g_sel = got["sel"][l, t][r]
                assert np.array_equal(g_sel[:sel.size], sel), f"selection r{r} l{l} t{t}"
                page, rev, stamp, order, (length, step, hits, misses) = got["meta"][l, t][r]
                assert length == int(w.contexts()[r]) + t + 1 and step == t + 1
                assert (hits - prev_h, misses - prev_m) == (st["hits"], st["misses"]), f"hit/miss r{r} l{l} t{t}"
                prev_h, prev_m = hits, misses
                assert np.array_equal(page, snap[0]) and np.array_equal(rev, snap[1])
                assert np.array_equal(stamp, snap[2])
                check_order(order, stamp)
                o = oracle_attention(w, r, l, t, sel)
                ma, rel = attention_error(got["out"][l, t][r], o)
                assert ma <= MAX_ABS and rel <= REL_L2, f"attention r{r} l{l} t{t}: {ma} {rel}"
    assert cache.stats()["device_error"] == 0
    cache.close()


def test_follower_without_its_lead_is_reported():
    import torch
    from tiered_kv_cache_int8_gb300 import hs
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=2, context=1000, top_k=128, hot_slots=256,
                         steps=1)
    cache = make_cache(w, 1, index_share=2, share_prefetch=True)
    prefill(cache, w)
    inp = StepInputs(w, 1)
    out = cache.decode_layer(1, inp.q_idx[1, 0], inp.q[1, 0], new_kv=inp.kv[1, 0], new_keys=inp.keys[1, 0])
    torch.cuda.synchronize()
    assert cache.stats()["device_error"] & hs.HS_DEVERR_NO_LEAD
    assert not out.view(torch.int16).any()
    cache.close()


def test_attention_timeline_counters():
    # the GQA attention kernel's stage waits and CTA timeline (hs_stats): the first
    # step misses every selected row, so host stages are seen; latent rows record
    # nothing
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=2, context=5003, top_k=256, hot_slots=512,
                         steps=4)
    cache = make_cache(w, 4)
    prefill(cache, w)
    run_steps(cache, w, StepInputs(w, 4), 4)
    st = cache.stats()
    cache.close()
    assert st["device_error"] == 0
    assert st["att_host_stages"] > 0 and st["att_host_wait_ns"] > 0
    assert st["att_hbm_stages"] > 0
    # 3 requests x 256 rows in 16-row stages, 2 layers x 4 steps
    assert st["att_host_stages"] + st["att_hbm_stages"] == 3 * 256 // 16 * 2 * 4
    assert 0 < st["att_last_median_ns"] <= st["att_last_span_ns"] < 10**9
    w = wl.make_workload("mla_128k", n_requests=2, n_layers=1, context=3000, h_q=16, top_k=256, hot_slots=256,
                         steps=2)
    cache = make_cache(w, 2)
    prefill(cache, w)
    run_steps(cache, w, StepInputs(w, 2), 2)
    st = cache.stats()
    cache.close()
    assert st["att_host_stages"] + st["att_hbm_stages"] == 0 and st["att_last_span_ns"] == 0
