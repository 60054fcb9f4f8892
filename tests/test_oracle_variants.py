"""Pins of the differential-attention oracle ("Attention Variants", differential attention):
checked against the independent attend oracle, closed forms and a case worked by hand."""
import math

import numpy as np

from oracle import attend, attention_weights, diff_attend


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_diff_reduces_to_plain_attention():
    """lambda = 0 gives attend(Q1, K1, V); Q2, K2 = Q1, K1 gives (1 - lambda) attend."""
    B, H, n_kv, T, d = 2, 4, 2, 37, 8
    q1, k1, q2, k2, v = (_rand(s, 200 + i) for i, s in enumerate(
        [(B, H, T, d), (B, n_kv, T, d), (B, H, T, d), (B, n_kv, T, d), (B, n_kv, T, d)]))
    ref, _ = attend(q1, k1, v, causal=True)
    assert np.max(np.abs(diff_attend(q1, k1, q2, k2, v, 0.0) - ref)) <= 1e-13
    assert np.max(np.abs(diff_attend(q1, k1, q1, k1, v, 0.7) - 0.3 * ref)) <= 1e-13
    lens = [30, 37]
    ref, _ = attend(q1[:, :, :25], k1, v, k_lens=lens, causal=True, window=9)
    got = diff_attend(q1[:, :, :25], k1, q2[:, :, :25], k2, v, 0.0, k_lens=lens, window=9)
    assert np.max(np.abs(got - ref)) <= 1e-13


def test_diff_rows_and_constant_values():
    """Each softmax row sums to 1 over the allowed keys, so the rows of A1 - lambda A2 sum to
    1 - lambda and constant values c give (1 - lambda) c; masked keys get weight 0."""
    B, H, T, d, lam = 1, 2, 11, 4, 0.6
    q1, k1, q2, k2 = (_rand(s, 210 + i) for i, s in enumerate([(B, H, T, d), (B, 1, T, d)] * 2))
    w = attention_weights(q1, k1, causal=True)
    assert np.allclose(w.sum(axis=3), 1.0, atol=1e-14)
    assert np.all(np.triu(w[0, 0], 1) == 0.0)
    v = np.full((B, 1, T, d), 2.5)
    assert np.allclose(diff_attend(q1, k1, q2, k2, v, lam), (1 - lam) * 2.5, atol=1e-13)


def test_diff_by_hand():
    """T = 2, d = 1, causal: row 0 sees only key 0 (weights 1 in both maps, out = (1 - lam) v0);
    row 1 weights softmax([q k0, q k1]) per map, written out."""
    q1 = np.array([[[[1.0], [2.0]]]])
    k1 = np.array([[[[0.5], [1.0]]]])
    q2 = np.array([[[[-1.0], [0.5]]]])
    k2 = np.array([[[[1.0], [3.0]]]])
    v = np.array([[[[10.0], [20.0]]]])
    lam = 0.5
    out = diff_attend(q1, k1, q2, k2, v, lam)
    assert abs(out[0, 0, 0, 0] - (1 - lam) * 10.0) < 1e-13
    a = np.exp([2.0 * 0.5, 2.0 * 1.0]); a /= a.sum()
    b = np.exp([0.5 * 1.0, 0.5 * 3.0]); b /= b.sum()
    expect = (a[0] - lam * b[0]) * 10.0 + (a[1] - lam * b[1]) * 20.0
    assert abs(out[0, 0, 1, 0] - expect) < 1e-13


def test_diff_rows_subset_is_the_same_rows_of_the_full_result():
    """Evaluating only some query rows (as the full-size parity tests do) gives exactly those
    rows of the full computation, with per-sequence lengths and a window."""
    B, H, n_kv, T, d = 2, 4, 2, 41, 8
    q1, k1, q2, k2, v = (_rand(s, 240 + i) for i, s in enumerate(
        [(B, H, T, d), (B, n_kv, T, d), (B, H, T, d), (B, n_kv, T, d), (B, n_kv, T, d)]))
    rows = np.array([0, 5, 17, 40, 23])
    for kw in ({}, {"k_lens": [41, 36], "window": 7}):
        full = diff_attend(q1, k1, q2, k2, v, 0.8, **kw)
        part = diff_attend(q1, k1, q2, k2, v, 0.8, rows=rows, **kw)
        assert np.array_equal(part, full[:, :, rows])
