"""hs_indexer_topk_static: the selection entry point for callers that cannot
allocate device memory (its scratch is a static device array inside the
library).  Its output must equal the selection hs_decode_layer reports for the
same keys and queries, on two calls in a row (the second call reuses the array
the first one left behind).  Collected last on purpose."""
import numpy as np
import pytest

import workload as wl
from tests.harness import StepInputs, make_cache, prefill

pytestmark = pytest.mark.gpu


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
        assert np.array_equal(sel.cpu().numpy(), sel_ref.cpu().numpy()), f"call {t}"
    cache.close()


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
