"""Oracle for softmax(QK^T / sqrt(d) + mask) V with grouped-query heads, an absolute-position
causal mask, an optional sliding window, an optional per-head sink and an optional
block-level mask.  Float64 throughout; test infrastructure only (see the package header).

Definitions followed:
  * "Attention in Code", "one function all designs use": scores are q.k / sqrt(d) with d the
    query's last dimension; positions a query may not see get a score of minus infinity
    before the softmax; a sink is one more logit per head that takes part in the softmax
    normaliser but has no value vector, so its weight is dropped before the weighted sum of
    values.  The causal rule puts the Tq new queries at absolute positions Tk-Tq .. Tk-1
    and lets position i see key j when j <= i, and, with a window W, also j > i - W.
  * "Attention in Code", section 1 (MHA, MQA, GQA): query head h reads key/value head
    h // (n_heads / n_kv); the number of query heads must be a multiple of n_kv.
  * "Express note" (tilnote.io), "causal attention is a position problem": under a KV cache
    the causal rule must use the absolute position, not the index inside the query block.
  * "Attention Masking" guide, Example 6: keys at or beyond a sequence's length are masked.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["positions", "visible", "attend"]


def positions(Tq: int, Tk: int) -> np.ndarray:
    """Absolute positions of Tq new queries appended to a cache holding Tk keys in total."""
    return np.arange(Tk - Tq, Tk, dtype=np.int64)


def visible(i: np.ndarray, Tk: int, causal: bool = True, window: int = 0) -> np.ndarray:
    """bool [len(i), Tk]: True where the query at absolute position i[r] may look at key j.

    j <= i under the causal rule and, with a window W >= 1, j > i - W as well: the W most
    recent keys including the query's own position.
    """
    i = np.asarray(i, dtype=np.int64)
    j = np.arange(Tk, dtype=np.int64)
    ok = np.ones((i.shape[0], Tk), dtype=bool)
    if causal:
        ok &= j[None, :] <= i[:, None]
    if window:
        ok &= j[None, :] > i[:, None] - window
    return ok


def attend(q, k, v, *, k_lens=None, causal: bool = True, window: int = 0, sink=None,
           block_mask=None, q_block: int = 128, k_block: int = 64, rows=None):
    """Attention for every (batch, query head, query row); returns (out, lse).

    q: [B, H, Tq, d]; k, v: [B, n_kv, Tk_max, d]; k_lens: [B] keys present per sequence
    (default Tk_max); sink: [H] logits or None; block_mask: [B, H, ceil(Tq/q_block),
    ceil(Tk_max/k_block)] nonzero where the (query block, key block) pair may be used;
    rows: optional subset of query rows t (the output then has len(rows) rows).

    For row t of sequence b the absolute position is i = Tk_b - Tq + t and the allowed set
    is A = {j < Tk_b : visible(i, j) and block_mask[b, h, t // q_block, j // k_block]}.
    With m = max({s_j : j in A} + {sink_h}) and Z = sum_A e^(s_j - m) + e^(sink_h - m):
        out = sum_A e^(s_j - m) v_j / Z,   lse = m + ln Z   (natural log).
    A row whose allowed set is empty and which has no sink gets out = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Tq, d = q.shape
    n_kv, Tk_max = k.shape[1], k.shape[2]
    if H % n_kv != 0:
        raise ValueError("n_heads must be a multiple of n_kv")
    if window and not causal:
        raise ValueError("a window is defined only together with the causal rule")
    g = H // n_kv
    rows = np.arange(Tq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.zeros((B, H, R, v.shape[-1]), dtype=np.float64)
    lse = np.full((B, H, R), -np.inf, dtype=np.float64)
    scale = 1.0 / math.sqrt(d)
    for b in range(B):
        Tk = Tk_max if k_lens is None else int(k_lens[b])
        if Tq > Tk:
            raise ValueError("Tq must not exceed the number of keys present")
        base = visible(positions(Tq, Tk)[rows], Tk, causal, window)
        for h in range(H):
            kvh = h // g
            allowed = base
            if block_mask is not None:
                bm = np.asarray(block_mask[b, h]).astype(bool)
                allowed = base & bm[rows // q_block][:, np.arange(Tk) // k_block]
            s = (q[b, h, rows] @ k[b, kvh, :Tk].T) * scale
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1) if Tk > 0 else np.full(R, -np.inf)
            if sink is not None:
                m = np.maximum(m, float(sink[h]))
            live = np.isfinite(m)
            ms = np.where(live, m, 0.0)
            w = np.where(allowed, np.exp(s - ms[:, None]), 0.0)
            Z = w.sum(axis=1)
            if sink is not None:
                Z = Z + np.exp(float(sink[h]) - ms)
            num = w @ v[b, kvh, :Tk]
            ok = live & (Z > 0)
            out[b, h] = np.where(ok[:, None], num / np.where(ok, Z, 1.0)[:, None], 0.0)
            lse[b, h] = np.where(ok, ms + np.log(np.where(ok, Z, 1.0)), -np.inf)
    return out, lse
