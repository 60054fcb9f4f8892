"""Oracle for decoding through a W-slot ring-buffer key/value cache.  Float64; test
infrastructure only (see the package header).

Source: "Attention in Code", section 2 (sliding window: ring buffer).  A sliding-window
layer only ever looks at the latest W tokens, so its cache keeps W slots and token n is
written into slot n mod W, overwriting the oldest one.  Once the buffer has wrapped the
slots are out of order, which does not matter: a softmax over a set of keys does not depend
on the order of the keys.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["ring_contents", "ring_decode"]


def ring_decode(q, k, v, window: int, sink=None):
    """Feed T tokens one at a time through a W-slot ring cache; return [H, T, d] outputs.

    q: [H, T, d] query rows; k, v: [n_kv, T, d] the key/value row each token writes into
    the cache; query head h reads ring head h // (H / n_kv).  Token t writes slot t mod W,
    then its query attends over the min(t + 1, W) slots filled so far, with an optional
    per-head sink logit taking part in the normaliser.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H, T, d = q.shape
    n_kv = k.shape[0]
    g = H // n_kv
    ring_k = np.zeros((n_kv, window, d))
    ring_v = np.zeros((n_kv, window, v.shape[-1]))
    out = np.zeros((H, T, v.shape[-1]))
    for t in range(T):
        ring_k[:, t % window] = k[:, t]
        ring_v[:, t % window] = v[:, t]
        filled = min(t + 1, window)
        for h in range(H):
            s = ring_k[h // g, :filled] @ q[h, t] / math.sqrt(d)
            m = s.max() if sink is None else max(s.max(), float(sink[h]))
            w = np.exp(s - m)
            Z = w.sum() + (0.0 if sink is None else math.exp(float(sink[h]) - m))
            out[h, t] = (w @ ring_v[h // g, :filled]) / Z
    return out


def ring_contents(k, v, window: int, n_tokens: int | None = None):
    """The ring caches after tokens 0 .. n_tokens-1 of k, v [n_kv, T, d] were written, token t
    into slot t mod W ("Attention in Code", section 2).  Slots never written stay zero.
    Returns (ring_k, ring_v), each [n_kv, W, d]."""
    k = np.asarray(k)
    v = np.asarray(v)
    n = k.shape[1] if n_tokens is None else n_tokens
    ring_k = np.zeros((k.shape[0], window, k.shape[2]), dtype=k.dtype)
    ring_v = np.zeros((v.shape[0], window, v.shape[2]), dtype=v.dtype)
    for t in range(n):
        ring_k[:, t % window] = k[:, t]
        ring_v[:, t % window] = v[:, t]
    return ring_k, ring_v
