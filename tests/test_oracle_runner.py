"""The oracle's replay of a workload: per-step bookkeeping and bounds."""
import numpy as np

import workload as wl
from oracle import bf16_to_f64, belady_misses
from oracle.runner import replay_request_layer


def test_tiny_replay_bookkeeping():
    w = wl.WORKLOADS["tiny"]
    r = replay_request_layer(w, 0, 0, steps=12, attention_steps=[0, 11])
    for t in range(12):
        assert r["hits"][t] + r["misses"][t] == w.top_k
        assert r["sel"][t].size == w.top_k and (np.diff(r["sel"][t]) > 0).all()
        assert r["sel"][t].max() < 4096 + t + 1
    assert r["misses"][0] == w.top_k                       # cold first step
    assert sum(r["misses"]) >= belady_misses(r["sel"], w.hot_slots)
    assert r["out"][0].shape == (8, 128) and np.isfinite(r["out"][11]).all()
    # locality of the walk: later steps mostly hit
    assert np.mean(r["hits"][1:]) > 0.5 * w.top_k


def test_k_at_least_context_is_dense_attention():
    # k >= N selects every position; with a zero attention query the output is
    # the plain mean of all V rows of the kv head (dense attention closed form)
    w = wl.make_workload("tiny", context=40, top_k=64, hot_slots=64, steps=3)
    r = replay_request_layer(w, 0, 0, attention_steps=None)
    for t in range(3):
        assert r["sel"][t].tolist() == list(range(40 + t + 1))
    rows = wl.kv_rows_at(w, 0, 0, np.arange(43))
    from oracle import sparse_attention
    o = sparse_attention(np.zeros((8, 128), np.uint16), rows, h_kv=1, d_qk=128, d_v=128, v_offset=128)
    assert np.allclose(o, bf16_to_f64(rows)[:, 128:].mean(0), atol=1e-14)
