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
