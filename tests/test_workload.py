"""The seeded generators: deterministic, independent of threading, right
shapes, ranges and distributions, and consistent random access."""
import numpy as np

import workload as wl


def test_tiny_shapes_and_ranges():
    w = wl.WORKLOADS["tiny"]
    kv = wl.prefill_kv(w, 0, 0)
    assert kv.shape == (4096, w.row_elems) and kv.dtype == np.uint16 and w.row_bytes == 512
    keys = wl.prefill_idx_keys(w, 0, 0)
    assert keys.shape == (4096, 64) and keys.min() >= -127 and keys.max() <= 127
    walk = wl.query_walk(w, 0, 0)
    assert walk.shape == (32, 64) and np.abs(walk).max() == 127
    x = (kv.astype(np.uint32) << 16).view(np.float32)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_deterministic_and_thread_independent():
    w = wl.make_workload("batch16_32k", context=9000, n_requests=2)
    a = wl.prefill_kv(w, 1, 2, parallel=True)
    b = wl.prefill_kv(w, 1, 2, parallel=False)
    assert np.array_equal(a, b)
    c = wl.prefill_kv(w, 0, 2)
    assert not np.array_equal(a[:100], c[:100])


def test_random_access_matches_bulk():
    w = wl.make_workload("batch16_32k", context=9000, n_requests=2)
    bulk = wl.prefill_kv(w, 1, 0)
    pos = np.array([0, 4095, 4096, 8999, 9000, 9003])
    got = wl.kv_rows_at(w, 1, 0, pos)
    assert np.array_equal(got[:4], bulk[pos[:4]])
    assert np.array_equal(got[4], wl.step_kv_row(w, 1, 0, 0))
    assert np.array_equal(got[5], wl.step_kv_row(w, 1, 0, 3))
    keys = wl.idx_keys_upto(w, 1, 0, 3)
    assert keys.shape == (9003, 128) and np.array_equal(keys[9001], wl.step_idx_key(w, 1, 0, 1))


def test_walk_locality_grows_with_smaller_sigma():
    base = wl.make_workload("batch16_32k", n_requests=1, steps=40)
    cos = {}
    for s in (0.05, 0.1, 0.3):
        q = wl.query_walk(wl.make_workload("batch16_32k", n_requests=1, steps=40, sigma=s), 0, 0).astype(float)
        c = (q[1:] * q[:-1]).sum(1) / np.linalg.norm(q[1:], axis=1) / np.linalg.norm(q[:-1], axis=1)
        cos[s] = c.mean()
    assert cos[0.05] > cos[0.1] > cos[0.3] > 0.8
    del base


def test_mixed_lengths_in_range():
    w = wl.WORKLOADS["mixed_8k_200k"]
    n = w.contexts()
    assert n.shape == (64,) and n.min() >= 8192 and n.max() <= 204800
    assert np.array_equal(n, wl.WORKLOADS["mixed_8k_200k"].contexts())


def test_sizes_of_the_full_workloads():
    w2 = wl.WORKLOADS["batch16_32k"]
    assert abs(w2.host_bytes() / 1e9 - 8.6) < 0.1 and abs(w2.hot_bytes() / 1e9 - 1.07) < 0.01
    w5 = wl.WORKLOADS["stress_128k"]
    assert abs(w5.host_bytes() / 2 ** 30 - 64) < 0.1


def test_multihead_queries_and_weights():
    w = wl.make_workload("batch16_32k", n_requests=2, n_layers=1, context=100, steps=6, idx_heads=4)
    h = wl.query_walk_heads(w, 1, 0, 6)
    assert h.shape == (6, 4, w.d_idx) and h.dtype == np.int8
    assert np.array_equal(h[:, 0], wl.query_walk(w, 1, 0, 6))        # head 0 is the single-head walk
    assert not np.array_equal(h[:, 1], h[:, 2])                        # independent heads
    assert np.array_equal(h, wl.query_walk_heads(w, 1, 0, 6))          # deterministic
    wt = wl.step_idx_weights(w, 1, 0, 3)
    assert wt.shape == (4,) and wt.dtype == np.int8 and (wt >= 0).all()
