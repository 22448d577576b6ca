"""Failure paths, injected on the host (no GPU fault is ever provoked): an
allocation that fails inside hs_create must come back as HS_ERR_OOM with every
earlier allocation released, and the next hs_create must succeed and decode."""
import numpy as np
import pytest

import workload as wl
from tests.harness import StepInputs, bf16_bits_to_f64, make_cache, prefill, run_steps

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("what", ["hostalloc", "devalloc"])
def test_injected_allocation_failure_is_reported_and_released(what, monkeypatch):
    import torch
    from tiered_kv_cache_int8_gb300.build import build
    build()
    from tiered_kv_cache_int8_gb300 import hs
    dev = torch.device("cuda", 0)
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=3000, top_k=256,
                         hot_slots=512, steps=2)
    torch.cuda.synchronize(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    monkeypatch.setenv("HS_FAULT_INJECT", what)
    with pytest.raises(hs.HsError) as e:
        make_cache(w, 2)
    assert e.value.status == hs.HS_ERR_OOM, str(e.value)
    assert "injected" in str(e.value) or "failed" in str(e.value)
    torch.cuda.synchronize(dev)
    # everything hs_create had allocated before the failure is released again
    # (within one allocation granule of the driver's own bookkeeping)
    assert torch.cuda.mem_get_info(dev)[0] >= free0 - (2 << 20)
    monkeypatch.delenv("HS_FAULT_INJECT")
    cache = make_cache(w, 2)
    prefill(cache, w)
    got = run_steps(cache, w, StepInputs(w, 2), 2, collect_out=True)
    assert all(np.isfinite(bf16_bits_to_f64(got["out"][0, t])).all() for t in range(2))
    assert cache.stats()["device_error"] == 0
    cache.close()


def test_a_wait_that_runs_out_sets_the_timeout_bit_and_the_gpu_stays_usable(monkeypatch):
    # HS_FAULT_INJECT=noready makes the select kernel withhold request 0's
    # publication: the attention kernel's bounded wait for it gives up after
    # about a second, the call completes with HS_DEVERR_TIMEOUT, the other
    # requests are still exact, and a fresh handle afterwards works normally
    import torch
    from tiered_kv_cache_int8_gb300.build import build
    build()
    from oracle import indexer_scores_many, sparse_attention, topk_select
    from tests.harness import MAX_ABS, REL_L2, attention_error
    from tiered_kv_cache_int8_gb300 import hs
    w = wl.make_workload("batch16_32k", n_requests=3, n_layers=1, context=3000, top_k=256,
                         hot_slots=512, steps=1)
    monkeypatch.setenv("HS_FAULT_INJECT", "noready")
    cache = make_cache(w, 1)
    monkeypatch.delenv("HS_FAULT_INJECT")
    prefill(cache, w)
    got = run_steps(cache, w, StepInputs(w, 1), 1, collect_out=True, fused=True)
    st = cache.stats()
    assert st["device_error"] & hs.HS_DEVERR_TIMEOUT
    for r in (1, 2):
        keys = wl.idx_keys_upto(w, r, 0, 1)
        sel = topk_select(indexer_scores_many(keys, wl.query_walk(w, r, 0, 1))[:, 0], w.top_k)
        assert np.array_equal(got["sel"][0, 0][r][:sel.size], sel)
        ref = sparse_attention(wl.step_query(w, r, 0, 0), wl.kv_rows_at(w, r, 0, sel), h_kv=w.h_kv,
                               d_qk=w.d_qk, d_v=w.d_v, v_offset=w.v_offset)
        ma, rel = attention_error(got["out"][0, 0][r], ref)
        assert ma <= MAX_ABS and rel <= REL_L2
    cache.close()
    torch.cuda.synchronize()
    cache = make_cache(w, 2)
    prefill(cache, w)
    run_steps(cache, w, StepInputs(w, 2), 2, collect_out=True, fused=True)
    assert cache.stats()["device_error"] == 0
    cache.close()
