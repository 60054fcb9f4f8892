"""Pins of the token top-k sparse attention oracle ("Attention in Code", section 5)."""
import math

import numpy as np

from oracle import attend
from oracle.dsa import dsa_decode, indexer_scores, sparse_attend, topk_indices


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_indexer_scores_by_loops():
    """score[t, s] = sum_j w[j, t] relu(qi[j, t] . ki[s]), written as plain loops."""
    Hi, T, L, di = 3, 4, 6, 5
    qi, ki, wi = _rand((Hi, T, di), 401), _rand((L, di), 402), _rand((Hi, T), 403)
    got = indexer_scores(qi, ki, wi)
    for t in range(T):
        for s in range(L):
            ref = 0.0
            for j in range(Hi):
                dot = sum(qi[j, t, e] * ki[s, e] for e in range(di))
                ref += wi[j, t] * max(dot, 0.0)
            assert abs(got[t, s] - ref) < 1e-12


def test_topk_at_least_length_is_full_attention_and_read_counts():
    """k >= L reproduces full causal attention (the page: difference 0); with 60 tokens and
    k = 16 every row reads min(16, t + 1) tokens, the last one 16."""
    H, n_kv, T, d, Hi, di = 4, 2, 60, 8, 2, 4
    q, k, v = _rand((H, T, d), 404), _rand((n_kv, T, d), 405), _rand((n_kv, T, d), 406)
    sc = indexer_scores(_rand((Hi, T, di), 407), _rand((T, di), 408), np.abs(_rand((Hi, T), 409)))
    full, _ = attend(q[None], k[None], v[None], causal=True)
    out, reads = sparse_attend(q, k, v, sc, topk=T)
    assert np.max(np.abs(out - full[0])) <= 1e-13
    assert np.array_equal(reads, np.arange(1, T + 1))
    out16, reads16 = sparse_attend(q, k, v, sc, topk=16)
    assert np.array_equal(reads16, np.minimum(np.arange(1, T + 1), 16)) and reads16[-1] == 16
    assert np.max(np.abs(out16[:, :16] - full[0, :, :16])) <= 1e-13      # rows that see <= 16 keys
    assert np.max(np.abs(out16 - full[0])) > 1e-3                          # no longer equal after


def test_topk_indices_by_sorting_and_ties():
    s = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 3.0, 0.5])
    assert topk_indices(s, np.ones(7, bool), 3).tolist() == [1, 3, 5]
    assert topk_indices(s, np.ones(7, bool), 4).tolist() == [0, 1, 3, 5]   # tie at 0.5: lowest index
    assert topk_indices(s, np.arange(7) <= 2, 5).tolist() == [0, 1, 2]     # only the allowed ones
    rng = np.random.default_rng(410)
    for _ in range(20):
        x = rng.standard_normal(50)
        kk = int(rng.integers(1, 60))
        ref = np.sort(np.argsort(-x, kind="stable")[:min(kk, 50)])
        assert np.array_equal(topk_indices(x, np.ones(50, bool), kk), ref)


def test_dsa_decode_is_the_last_row():
    """The batch decode form equals the last row of the prefill form for each sequence."""
    B, H, n_kv, Lm, d, Hi, di, kk = 2, 4, 2, 30, 8, 3, 4, 7
    q = _rand((B, H, 1, d), 411)
    k, v = _rand((B, n_kv, Lm, d), 412), _rand((B, n_kv, Lm, d), 413)
    qi, ki, wi = _rand((B, Hi, di), 414), _rand((B, Lm, di), 415), _rand((B, Hi), 416)
    lens = [30, 19]
    out, chosen = dsa_decode(q, k, v, qi, ki, wi, lens, kk)
    for b in range(B):
        L = lens[b]
        sc = indexer_scores(qi[b][:, None], ki[b, :L], wi[b][:, None])
        ref, _ = sparse_attend(q[b], k[b, :, :L], v[b, :, :L], sc, kk)
        assert np.max(np.abs(out[b] - ref)) <= 1e-14
        assert chosen[b].size == min(kk, L)


def test_empty_cache_gives_a_zero_row_like_attend():
    """A sequence with no cached token reads nothing: its row is 0 with or without a sink, the
    convention attend follows for a row with no allowed key (checked here against attend with
    an all-zero block mask); the other sequence is unaffected."""
    B, H, n_kv, Lm, d, Hi, di, kk = 2, 4, 2, 30, 8, 3, 4, 7
    q = _rand((B, H, 1, d), 421)
    k, v = _rand((B, n_kv, Lm, d), 422), _rand((B, n_kv, Lm, d), 423)
    qi, ki, wi = _rand((B, Hi, di), 424), _rand((B, Lm, di), 425), _rand((B, Hi), 426)
    sink = np.array([0.5, -1.0, 0.25, 2.0])
    for sk in (None, sink):
        out, chosen = dsa_decode(q, k, v, qi, ki, wi, [30, 0], kk, sink=sk)
        assert chosen[1].size == 0 and np.all(out[1] == 0.0)
        none, _ = attend(q[1:2], k[1:2], v[1:2], causal=False, sink=sk,
                         block_mask=np.zeros((1, H, 1, 1), dtype=bool), q_block=1, k_block=Lm)
        assert np.array_equal(out[1:2], none)
        ref, _ = dsa_decode(q[:1], k[:1], v[:1], qi[:1], ki[:1], wi[:1], [30], kk, sink=sk)
        assert np.array_equal(out[:1], ref)


def test_sparse_attend_with_sink_equals_attend_on_the_chosen_tokens():
    """"Attention in Code" s.3 and s.5 together: with a sink, top-k sparse attention equals the
    pinned attend with a key-level mask (q_block = k_block = 1) that admits exactly each row's
    chosen tokens, the same sink in the normaliser; so the sink branch of sparse_attend is
    checked against attend's, which the SDPA and closed-form pins fix.  Also for the decode form."""
    H, n_kv, T, d, Hi, di, kk = 4, 2, 40, 8, 2, 4, 9
    q, k, v = _rand((H, T, d), 431), _rand((n_kv, T, d), 432), _rand((n_kv, T, d), 433)
    sc = indexer_scores(_rand((Hi, T, di), 434), _rand((T, di), 435), np.abs(_rand((Hi, T), 436)))
    for sink in (_rand((H,), 437), np.array([5.0, 8.0, -3.0, 12.0])):
        out, reads = sparse_attend(q, k, v, sc, kk, sink=sink)
        mask = np.zeros((1, H, T, T), dtype=bool)
        for t in range(T):
            mask[0, :, t, topk_indices(sc[t], np.arange(T) <= t, kk)] = True
        ref, _ = attend(q[None], k[None], v[None], causal=True, sink=sink, block_mask=mask,
                        q_block=1, k_block=1)
        assert np.max(np.abs(out - ref[0])) <= 1e-13
        assert np.array_equal(reads, mask[0, 0].sum(axis=1))
    # decode form with a sink: the last row of each sequence
    B, Lm = 2, 30
    qd = _rand((B, H, 1, d), 438)
    kd, vd = _rand((B, n_kv, Lm, d), 439), _rand((B, n_kv, Lm, d), 440)
    qi, ki, wi = _rand((B, Hi, di), 441), _rand((B, Lm, di), 442), _rand((B, Hi), 443)
    sink = _rand((H,), 444)
    lens = [30, 17]
    out, chosen = dsa_decode(qd, kd, vd, qi, ki, wi, lens, kk, sink=sink)
    for b in range(B):
        L = lens[b]
        m = np.zeros((1, H, 1, L), dtype=bool)
        m[0, :, 0, chosen[b]] = True
        ref, _ = attend(qd[b:b + 1], kd[b:b + 1, :, :L], vd[b:b + 1, :, :L], causal=True, sink=sink,
                        block_mask=m, q_block=1, k_block=1)
        assert np.max(np.abs(out[b] - ref[0])) <= 1e-13
