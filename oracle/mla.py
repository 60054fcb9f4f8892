"""Oracle for multi-head latent attention (MLA).  Float64; test infrastructure only (see the
package header).

Source: "Attention in Code", section 4 (store only the latent vectors, move the weights to the
query side).  Each cached token holds a compressed vector c_kv (r numbers) and one small key
k_rope (dr numbers) shared by every head; head h's key and value are c_kv @ w_uk[h] (plus
k_rope) and c_kv @ w_uv[h].
  naive:    rebuild every head's keys and values from the latents, then attend as usual;
  absorbed: q_lat = q_nope @ w_uk[h]^T moves the query into latent space, the scores are
            (q_lat . c_kv + q_rope . k_rope) / sqrt(dn + dr), the softmax weights average the
            latents, and w_uv expands the result once per head.
The two agree for any weights: q_nope . (c_kv w_uk) = (q_nope w_uk^T) . c_kv, and the weighted
average commutes with the linear map w_uv.  The scale is that of the head's full query,
1 / sqrt(dn + dr).
"""
from __future__ import annotations

import math

import numpy as np

from .attention import attend

__all__ = ["mla_naive", "mla_absorbed"]


def _causal(T: int, L: int) -> np.ndarray:
    """bool [T, L]: query t (absolute position L - T + t) may see token j <= L - T + t."""
    return np.arange(L)[None, :] <= (L - T + np.arange(T))[:, None]


def mla_naive(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv):
    """q_nope [H, T, dn], q_rope [H, T, dr], c_kv [L, r], k_rope [L, dr], w_uk [H, r, dn],
    w_uv [H, r, dv]: per-head keys [c_kv w_uk | k_rope] and values c_kv w_uv, causal attention.
    Returns [H, T, dv]."""
    q_nope, q_rope, c_kv, k_rope, w_uk, w_uv = (np.asarray(x, dtype=np.float64)
                                                for x in (q_nope, q_rope, c_kv, k_rope, w_uk, w_uv))
    H, L = q_nope.shape[0], c_kv.shape[0]
    k = np.concatenate([c_kv @ w_uk, np.broadcast_to(k_rope, (H,) + k_rope.shape)], axis=-1)
    v = c_kv @ w_uv
    q = np.concatenate([q_nope, q_rope], axis=-1)
    out, _ = attend(q[None], k[None], v[None], causal=True)
    return out[0]


def mla_absorbed(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv):
    """Same result without per-head keys or values; returns [H, T, dv]."""
    q_nope, q_rope, c_kv, k_rope, w_uk, w_uv = (np.asarray(x, dtype=np.float64)
                                                for x in (q_nope, q_rope, c_kv, k_rope, w_uk, w_uv))
    T, L = q_nope.shape[1], c_kv.shape[0]
    scale = 1.0 / math.sqrt(q_nope.shape[-1] + q_rope.shape[-1])
    q_lat = q_nope @ np.swapaxes(w_uk, -1, -2)                    # [H, T, r]
    s = (q_lat @ c_kv.T + q_rope @ k_rope.T) * scale               # [H, T, L]
    s = np.where(_causal(T, L)[None], s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    w = np.exp(s - m)
    w /= w.sum(axis=-1, keepdims=True)
    return (w @ c_kv) @ w_uv                                        # [H, T, dv]
