"""Pins of the oracle's fp64 sparse attention: closed forms that a dropped term,
a wrong head mapping, a wrong V offset or a wrong scale would break."""
import math
import os

import numpy as np

from oracle import bf16_to_f64, hot_cache_bytes, hot_over_full, sparse_attention
from tests.conftest import GOLDEN
from workload import f32_to_bf16_bits


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_bf16_decode_known_patterns():
    assert bf16_to_f64(np.array([0x3F80, 0xC000, 0x0000, 0x3E80], dtype=np.uint16)).tolist() == [1.0, -2.0, 0.0, 0.25]
    # round to nearest even on the way in: 1 + 2^-8 is a tie between 1 and 1+2^-7
    assert bf16_to_f64(bf([1.0 + 2.0 ** -8]))[0] == 1.0
    assert bf16_to_f64(bf([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


def _rows(rng, n, elems):
    return bf(rng.standard_normal((n, elems)))


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(0)
    h_q, h_kv, d = 8, 2, 16
    rows = _rows(rng, 11, h_kv * 2 * d)
    q = bf(np.zeros((h_q, d)))
    o = sparse_attention(q, rows, h_kv=h_kv, d_qk=d, d_v=d, v_offset=h_kv * d)
    vals = bf16_to_f64(rows)
    for h in range(h_q):
        g = h // (h_q // h_kv)
        assert np.allclose(o[h], vals[:, h_kv * d + g * d: h_kv * d + (g + 1) * d].mean(0), atol=1e-15)


def test_gqa_head_mapping_with_constant_values():
    # V of kv head g is the constant g+1; with any query the output of q head h is
    # the constant of the kv head it reads: floor(h * H_kv / H_q) + 1
    rng = np.random.default_rng(1)
    h_q, h_kv, d = 12, 4, 8
    n = 9
    k_part = rng.standard_normal((n, h_kv * d))
    v_part = np.repeat(np.arange(1, h_kv + 1, dtype=np.float64), d)[None, :].repeat(n, 0)
    rows = bf(np.concatenate([k_part, v_part], 1))
    q = bf(rng.standard_normal((h_q, d)))
    o = sparse_attention(q, rows, h_kv=h_kv, d_qk=d, d_v=d, v_offset=h_kv * d)
    for h in range(h_q):
        assert np.allclose(o[h], (h * h_kv) // h_q + 1, atol=1e-12)


def test_dominant_logit_returns_its_value_row():
    h_q, d = 4, 32
    n = 6
    rows = np.zeros((n, 2 * d), dtype=np.float32)
    rows[:, d:] = np.arange(n)[:, None] * 0.5 - 1.0      # V row i = 0.5 i - 1
    rows[3, :d] = 8.0                                    # K row 3 aligned with q
    q = np.full((h_q, d), 8.0, dtype=np.float32)         # logit of row 3 = 2048/sqrt(32) = 362
    o = sparse_attention(bf(q), bf(rows), h_kv=1, d_qk=d, d_v=d, v_offset=d)
    assert np.allclose(o, 0.5 * 3 - 1.0, atol=1e-12)


def test_two_row_softmax_pins_the_scale():
    # logits differ by scale * q.(K0 - K1); p0 = 1 / (1 + exp(-(l0 - l1)))
    d = 64
    rows = np.zeros((2, 2 * d), dtype=np.float32)
    rows[0, 0] = 1.0
    rows[0, d:] = 1.0          # V0 = 1
    rows[1, d:] = -1.0         # V1 = -1
    q = np.zeros((1, d), dtype=np.float32)
    q[0, 0] = 2.0
    o = sparse_attention(bf(q), bf(rows), h_kv=1, d_qk=d, d_v=d, v_offset=d)
    l_diff = 2.0 / math.sqrt(d)
    p0 = 1.0 / (1.0 + math.exp(-l_diff))
    assert np.allclose(o, p0 * 1 + (1 - p0) * -1, atol=1e-14)
    # explicit scale overrides the default
    o2 = sparse_attention(bf(q), bf(rows), h_kv=1, d_qk=d, d_v=d, v_offset=d, scale=1.0)
    p0 = 1.0 / (1.0 + math.exp(-2.0))
    assert np.allclose(o2, 2 * p0 - 1, atol=1e-14)


def test_latent_row_values_are_its_first_columns():
    # one shared 576-wide latent row read as K (all 576) and V (first 512)
    rng = np.random.default_rng(2)
    rows = _rows(rng, 7, 576)
    q = bf(np.zeros((16, 576)))
    o = sparse_attention(q, rows, h_kv=1, d_qk=576, d_v=512, v_offset=0)
    assert np.allclose(o, bf16_to_f64(rows)[:, :512].mean(0)[None, :], atol=1e-15)


def test_selection_order_does_not_matter_and_empty_is_zero():
    rng = np.random.default_rng(3)
    rows = _rows(rng, 20, 2 * 2 * 16)
    q = bf(rng.standard_normal((4, 16)))
    kw = dict(h_kv=2, d_qk=16, d_v=16, v_offset=32)
    a = sparse_attention(q, rows, **kw)
    b = sparse_attention(q, rows[::-1].copy(), **kw)
    assert np.allclose(a, b, atol=1e-14)
    assert (sparse_attention(q, rows[:0], **kw) == 0).all()
    # convex combination: each output lies inside the range of its value column
    vals = bf16_to_f64(rows)[:, 32:]
    assert (a <= vals.max(0).max() + 1e-12).all() and (a >= vals.min(0).min() - 1e-12).all()


def _read_capacity():
    d = {}
    for line in open(os.path.join(GOLDEN, "capacity_glm51_128k.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            d[k] = float(v)
    return d


def test_capacity_matches_the_printed_figures():
    c = _read_capacity()
    hot = hot_cache_bytes(c["full_kv_gb"], int(c["positions"]), int(c["hot_slots"]))
    assert round(hot, 1) == c["printed_hot_gb"]                 # 0.409 GB -> "about 0.4 GB"
    ratio = 1.0 / hot_over_full(int(c["hot_slots"]), int(c["positions"]))
    assert abs(ratio - c["printed_reduction"]) / c["printed_reduction"] < 0.1   # 32x -> "about 30x"
