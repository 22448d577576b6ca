"""Pins of the oracle's multi-head ReLU-weighted indexer, s[p] = sum_h w_h *
max(0, q_h . K[p]) (exact int64):

* a pure-Python triple loop on small random inputs;
* closed forms: one head with weight 1 is the single-head score through a
  ReLU; two opposite heads with equal weight a give a * |q . K|;
* linearity in the weights, and all-zero weights give all-zero scores (so the
  top-k is positions 0..k-1);
* the largest magnitude the variant admits (8 heads, weights 127, d_idx 256,
  entries -128) stays below 2^32, the width the library's keys have."""
import numpy as np

from oracle import indexer_scores, indexer_scores_multihead, topk_select


def _loop(keys, q, w):
    out = []
    for p in range(keys.shape[0]):
        s = 0
        for h in range(q.shape[0]):
            d = sum(int(keys[p, j]) * int(q[h, j]) for j in range(keys.shape[1]))
            s += int(w[h]) * max(0, d)
        out.append(s)
    return np.array(out, dtype=np.int64)


def test_equals_a_plain_loop():
    rng = np.random.default_rng(8)
    for H in (1, 2, 4, 8):
        keys = rng.integers(-128, 128, size=(37, 16), dtype=np.int8)
        q = rng.integers(-128, 128, size=(H, 16), dtype=np.int8)
        w = rng.integers(0, 128, size=H, dtype=np.int8)
        assert np.array_equal(indexer_scores_multihead(keys, q, w), _loop(keys, q, w))


def test_closed_forms():
    rng = np.random.default_rng(9)
    keys = rng.integers(-127, 128, size=(200, 64), dtype=np.int8)
    q = rng.integers(-127, 128, size=64, dtype=np.int8)
    single = indexer_scores(keys, q)
    one = indexer_scores_multihead(keys, q[None, :], np.array([1], np.int8))
    assert np.array_equal(one, np.maximum(single, 0))
    both = indexer_scores_multihead(keys, np.stack([q, -q]), np.array([5, 5], np.int8))
    assert np.array_equal(both, 5 * np.abs(single))


def test_linear_in_the_weights_and_zero_weights():
    rng = np.random.default_rng(10)
    keys = rng.integers(-127, 128, size=(300, 32), dtype=np.int8)
    q = rng.integers(-127, 128, size=(4, 32), dtype=np.int8)
    w1 = rng.integers(0, 64, size=4, dtype=np.int8)
    w2 = rng.integers(0, 64, size=4, dtype=np.int8)
    s1, s2 = indexer_scores_multihead(keys, q, w1), indexer_scores_multihead(keys, q, w2)
    assert np.array_equal(indexer_scores_multihead(keys, q, (w1 + w2).astype(np.int8)), s1 + s2)
    z = indexer_scores_multihead(keys, q, np.zeros(4, np.int8))
    assert not z.any()
    assert np.array_equal(topk_select(z, 20), np.arange(20))


def test_largest_magnitude_fits_32_bits():
    keys = np.full((1, 256), -128, np.int8)
    q = np.full((8, 256), -128, np.int8)
    s = indexer_scores_multihead(keys, q, np.full(8, 127, np.int8))
    assert s[0] == 8 * 127 * 128 * 128 * 256 and s[0] < 2 ** 32
