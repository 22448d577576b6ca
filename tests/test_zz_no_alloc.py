"""hs_indexer_topk_static: the selection entry point for callers that cannot
allocate device memory (code running inside another allocator, under a pool that
forbids side allocations, or in a plugin handed only raw buffers).  Its scratch
is a static device array inside the library.

Checked here: its output equals the selection hs_decode_layer reports for the
same keys and queries, and the oracle's full-sort top-k, on two calls in a row
(the second call reuses the array the first one left behind); mixed lengths
(0, < k, = k, > k), all-equal keys (every score ties), and the narrowest and
widest index keys; free device memory does not change across calls; its error
word reads 0 after good calls.  Collected last on purpose: a run that stops at
the first failure has run every other test by then."""
import numpy as np
import pytest

import workload as wl
from oracle import indexer_scores, topk_select
from tests.harness import StepInputs, make_cache, prefill

pytestmark = pytest.mark.gpu


def _oracle_selection(keys: np.ndarray, q: np.ndarray, lengths, k: int) -> np.ndarray:
    out = np.full((len(lengths), k), -1, np.int32)
    for r, n in enumerate(lengths):
        sel = topk_select(indexer_scores(keys[r, :n], q[r]), k)
        out[r, :sel.size] = sel
    return out


def test_static_selection_matches_decode_on_two_calls():
    import torch
    from tiered_kv_cache_int8_gb300.build import build
    build()
    from tiered_kv_cache_int8_gb300 import hs
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=1, context=5003, top_k=256,
                         hot_slots=512, steps=2)
    cache = make_cache(w, 2)
    prefill(cache, w)
    inp = StepInputs(w, 2)
    n0 = int(w.contexts()[0])
    n_max = n0 + 2
    keys = np.zeros((w.n_requests, n_max, w.d_idx), np.int8)
    for r in range(w.n_requests):
        keys[r] = wl.idx_keys_upto(w, r, 0, 2)
    keys_d = torch.from_numpy(keys).to(dev)
    for t in range(2):
        cache.append(0, inp.kv[0, t], inp.keys[0, t])
        sel_ref = torch.empty((w.n_requests, w.top_k), dtype=torch.int32, device=dev)
        cache.decode_layer(0, inp.q_idx[0, t], inp.q[0, t], sel_out=sel_ref)
        lengths = [n0 + t + 1] * w.n_requests
        sel = hs.indexer_topk_static(keys_d, lengths, inp.q_idx[0, t], w.top_k)
        torch.cuda.synchronize()
        got = sel.cpu().numpy()
        assert np.array_equal(got, sel_ref.cpu().numpy()), f"call {t}"
        assert np.array_equal(got, _oracle_selection(keys, inp.walk[0][:, t], lengths, w.top_k)), f"call {t}"
    assert hs.indexer_topk_static_error(0) == 0
    cache.close()


@pytest.mark.parametrize("d_idx", [16, 128, 256])
def test_static_selection_matches_the_oracle_on_mixed_lengths_and_ties(d_idx):
    import torch
    from tiered_kv_cache_int8_gb300.build import build
    build()
    from tiered_kv_cache_int8_gb300 import hs
    dev = torch.device("cuda", 0)
    k = 256
    n_max = 5003
    rng = np.random.default_rng(1000 + d_idx)
    # lengths: empty, shorter than k, exactly k, longer than k (one of them with
    # all-zero keys: every score ties, so the selection is positions 0..k-1)
    lengths = [0, 100, k, 5003, 4001, 2999]
    zero_req = 4
    keys = rng.integers(-127, 128, size=(len(lengths), n_max, d_idx), dtype=np.int8)
    keys[zero_req] = 0
    keys_d = torch.from_numpy(keys).to(dev)
    sel = torch.full((len(lengths), k), -7, dtype=torch.int32, device=dev)
    for call in range(3):
        q = rng.integers(-127, 128, size=(len(lengths), d_idx), dtype=np.int8)
        q_d = torch.from_numpy(q).to(dev)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        hs.indexer_topk_static(keys_d, lengths, q_d, k, sel_out=sel)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info(dev)[0]
        # the first call on a device may load the library's device module (and with
        # it the static array); every call after that leaves free memory unchanged
        if call > 0:
            assert free_after == free_before, f"call {call}: free device memory changed"
        got = sel.cpu().numpy()
        assert np.array_equal(got, _oracle_selection(keys, q, lengths, k)), f"call {call}"
        assert np.array_equal(got[zero_req], np.arange(k)), "ties must take the lowest positions"
        assert (got[0] == -1).all() and np.array_equal(got[2], np.arange(k))
        assert hs.indexer_topk_static_error(0) == 0


def test_static_selection_rejects_sizes_beyond_its_array():
    import torch
    from tiered_kv_cache_int8_gb300 import hs
    dev = torch.device("cuda", 0)
    q = torch.zeros((65, 16), dtype=torch.int8, device=dev)
    keys = torch.zeros((65, 4, 16), dtype=torch.int8, device=dev)
    with pytest.raises(hs.HsError) as e:
        hs.indexer_topk_static(keys, [4] * 65, q, 2)
    assert e.value.status == hs.HS_ERR_CAPACITY and "64" in str(e.value)
    keys = torch.zeros((2, (1 << 20) + 8, 16), dtype=torch.int8, device=dev)
    with pytest.raises(hs.HsError) as e:
        hs.indexer_topk_static(keys, [4, 4], q[:2], 2)
    assert e.value.status == hs.HS_ERR_CAPACITY
