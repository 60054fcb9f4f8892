"""Oracle for the attention variants built beside the main path.  Float64; test
infrastructure only (see the package header).

Differential attention ("Attention Variants" lesson, differential attention; its step 4):
two attention maps from two query/key pairs over the same values, the second scaled by a
mixing coefficient lambda and subtracted:
    A1 = softmax(Q1 K1^T / sqrt(d)),  A2 = softmax(Q2 K2^T / sqrt(d)),  out = (A1 - lambda A2) V
with the causal rule applied to both maps.  Written out with explicit weight matrices.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import positions, visible

__all__ = ["attention_weights", "diff_attend"]


def attention_weights(q, k, *, k_lens=None, causal: bool = True, window: int = 0, rows=None):
    """Explicit softmax weights [B, H, Tq, Tk_max]: row t of sequence b puts weight
    e^(s_j) / sum_A e^(s_j) on every allowed key j (positions and visibility as in attend)
    and 0 elsewhere; a row with no allowed key is all zero.  rows: optional subset of the
    query rows t (the result then has len(rows) rows, in that order)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, H, Tq, d = q.shape
    n_kv, Tk_max = k.shape[1], k.shape[2]
    g = H // n_kv
    rows = np.arange(Tq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    w = np.zeros((B, H, rows.shape[0], Tk_max))
    for b in range(B):
        Tk = Tk_max if k_lens is None else int(k_lens[b])
        allow = visible(positions(Tq, Tk)[rows], Tk, causal, window)            # [R, Tk]
        for h in range(H):
            s = q[b, h, rows] @ k[b, h // g, :Tk].T / math.sqrt(d)              # [R, Tk]
            s = np.where(allow, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            e = np.where(allow, np.exp(s - m), 0.0)
            z = e.sum(axis=1, keepdims=True)
            w[b, h, :, :Tk] = np.divide(e, z, out=np.zeros_like(e), where=z > 0)
    return w


def diff_attend(q1, k1, q2, k2, v, lam: float, *, k_lens=None, causal: bool = True, window: int = 0,
                rows=None):
    """(A1 - lam A2) V for every (batch, query head, query row): q1, q2 [B, H, Tq, d];
    k1, k2, v [B, n_kv, Tk_max, d]; query head h uses kv head h // (H / n_kv); rows: optional
    subset of the query rows, as in attention_weights."""
    v = np.asarray(v, dtype=np.float64)
    a1 = attention_weights(q1, k1, k_lens=k_lens, causal=causal, window=window, rows=rows)
    a2 = attention_weights(q2, k2, k_lens=k_lens, causal=causal, window=window, rows=rows)
    B, H = a1.shape[:2]
    g = H // v.shape[1]
    out = np.zeros((B, H, a1.shape[2], v.shape[-1]))
    for b in range(B):
        for h in range(H):
            out[b, h] = (a1[b, h] - lam * a2[b, h]) @ v[b, h // g]
    return out
