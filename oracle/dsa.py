"""Oracle for token top-k sparse attention with a lightning-style indexer.  Float64 (the
indexer scores in float32 where noted); test infrastructure only (see the package header).

Source: "Attention in Code", section 5 (sparse attention: store everything, read a little).
A small scorer -- a few small query heads, one small key per token, a ReLU and a weighted
sum -- rates every earlier token for the current query; attention then runs over the top k
tokens only, under the causal rule.  The whole cache stays; what shrinks is what attention
reads.

Readings: ties at the k-th score are broken toward the lower token index; the decode form
(one query per sequence, at position L_b - 1, which may see every cached token) is the one
built on the GPU.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["indexer_scores", "topk_indices", "sparse_attend", "dsa_decode"]


def indexer_scores(qi, ki, wi):
    """score[t, s] = sum_j wi[j, t] * relu(qi[j, t] . ki[s]); qi [Hi, T, di], ki [L, di],
    wi [Hi, T].  Returns [T, L] float64."""
    qi = np.asarray(qi, dtype=np.float64)
    ki = np.asarray(ki, dtype=np.float64)
    wi = np.asarray(wi, dtype=np.float64)
    dots = np.einsum("jtd,sd->jts", qi, ki)                 # [Hi, T, L]
    return (wi[:, :, None] * np.maximum(dots, 0.0)).sum(axis=0)


def topk_indices(scores_row, allowed, topk: int):
    """Indices of the min(topk, #allowed) largest scores among the allowed positions of one
    row, in increasing index order; ties at the boundary go to the lower index."""
    s = np.asarray(scores_row)
    cand = np.flatnonzero(np.asarray(allowed, dtype=bool))
    if cand.size == 0:
        return cand
    order = sorted(cand.tolist(), key=lambda j: (-float(s[j]), j))   # score down, index up
    return np.array(sorted(order[:min(topk, cand.size)]), dtype=np.int64)


def sparse_attend(q, k, v, scores, topk: int, sink=None):
    """Each query row attends only to its top-k tokens by indexer score, causally.
    q [H, T, d]; k, v [n_kv, L, d]; scores [T, L] (one score per query row and token, shared by
    the heads).  Returns (out [H, T, d], reads [T]: tokens each row attended to)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H, T, d = q.shape
    n_kv, L = k.shape[0], k.shape[1]
    g = H // n_kv
    out = np.zeros((H, T, v.shape[-1]))
    reads = np.zeros(T, dtype=np.int64)
    for t in range(T):
        i = L - T + t                                       # absolute position of row t
        keep = topk_indices(scores[t], np.arange(L) <= i, topk)
        reads[t] = keep.size
        if keep.size == 0:            # no token to read (an empty cache): the row stays 0, as
            continue                  # attend leaves a row with no allowed key
        for h in range(H):
            s = k[h // g, keep] @ q[h, t] / math.sqrt(d)
            m = s.max() if sink is None else max(s.max(), float(sink[h]))
            w = np.exp(s - m)
            z = w.sum() + (0.0 if sink is None else math.exp(float(sink[h]) - m))
            out[h, t] = w @ v[h // g, keep] / z
    return out, reads


def dsa_decode(q, k, v, qi, ki, wi, lens, topk: int, sink=None, scores=None):
    """Decode form for a batch: q [B, H, 1, d]; k, v [B, n_kv, L_max, d]; qi [B, Hi, di];
    ki [B, L_max, di]; wi [B, Hi]; lens [B] tokens cached per sequence.  The query of
    sequence b sits at position lens[b] - 1 and may see every cached token.  ``scores``
    [B, L_max] replaces the indexer's scores when given (to attend over a set chosen
    elsewhere).  Returns (out [B, H, 1, d], list of the selected index arrays)."""
    B = q.shape[0]
    out = np.zeros(q.shape[:3] + (v.shape[-1],))
    chosen = []
    for b in range(B):
        L = int(lens[b])
        if scores is None:
            sc = indexer_scores(np.asarray(qi)[b][:, None, :], np.asarray(ki)[b, :L], np.asarray(wi)[b][:, None])
        else:
            sc = np.asarray(scores)[b:b + 1, :L]
        o, _ = sparse_attend(np.asarray(q)[b], np.asarray(k)[b, :, :L], np.asarray(v)[b, :, :L], sc, topk, sink)
        out[b] = o
        chosen.append(topk_indices(sc[0], np.ones(L, dtype=bool), topk))
    return out, chosen
