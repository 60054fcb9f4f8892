"""Oracle for the block statistics and the block selection of radius-bounded sparse prefill.
Float64 throughout; test infrastructure only (see the package header).

Source: "RBS-Attention review" (patty.io), a prose review with no formulas.  The steps,
in the review's order:
  * "attention computed less" section: keys are grouped into blocks, each block is
    represented by one centroid, and a block's score is the query's inner product with it;
  * "when one average swallows an important token": one sharp key among many ordinary
    ones is averaged away, so the mean score alone drops the block (mean dilution);
  * "why bring in an unfamiliar ruler called the radius": the maximum key-block radius is
    the distance from the centroid to the farthest key of the block; it is judged against
    the distribution of radii of that prompt, layer and head, and blocks whose radius is
    unusually large in that context are rescued;
  * "what remains when two sieves are stacked": each branch thresholds on its own and the
    two block masks are joined by a union;
  * "how regular sparsity persuades the GPU": the union mask is block-level and drives a
    block-sparse FlashAttention pass.

The review prints neither threshold formula.  The readings taken here (each is also a
documented reading of the library):
  * mean score of a (query block, key block) pair: the mean of the block's query rows dotted
    with the centroid, over sqrt(d) -- by linearity equal to the mean of the rows' scores;
  * mean branch: keep a key block when its mean score is >= (largest mean score among the
    key blocks the query block may see) - tau_mean, in logit units;
  * radius branch: per (sequence, kv head), z = (r - mean(r)) / std(r) over all key blocks of
    the prompt (population std); rescue when z >= lambda_radius; nothing when std is 0;
    the rescue is shared by the query heads of the kv head and applies to every query
    block that may see the key block;
  * the key blocks overlapping the query block's own positions are always kept, so no query
    row is left with an empty set (a boundary convention; the review says nothing on it).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["block_stats", "allowed_blocks", "radius_zscores", "select_blocks"]


def block_stats(k, k_lens=None, k_block: int = 64):
    """Centroid and maximum radius of every key block.

    k: [B, n_kv, Tk_max, d].  Block beta of sequence b covers keys beta*k_block ..
    min((beta+1)*k_block, Tk_b) - 1 and holds n of them.  centroid = (1/n) sum_j k_j and
    radius = max_j ||k_j - centroid||_2.  Blocks with no key present (n = 0) get a zero
    centroid and a zero radius.  Returns (centroid [B, n_kv, nKb, d], radius [B, n_kv, nKb])
    with nKb = ceil(Tk_max / k_block).
    """
    k = np.asarray(k, dtype=np.float64)
    B, n_kv, Tk_max, d = k.shape
    nKb = -(-Tk_max // k_block)
    centroid = np.zeros((B, n_kv, nKb, d), dtype=np.float64)
    radius = np.zeros((B, n_kv, nKb), dtype=np.float64)
    for b in range(B):
        Tk = Tk_max if k_lens is None else int(k_lens[b])
        for kvh in range(n_kv):
            for beta in range(-(-Tk // k_block)):
                blk = k[b, kvh, beta * k_block:min((beta + 1) * k_block, Tk)]
                c = blk.mean(axis=0)
                centroid[b, kvh, beta] = c
                radius[b, kvh, beta] = np.sqrt(((blk - c) ** 2).sum(axis=1)).max()
    return centroid, radius


def allowed_blocks(alpha: int, Tq: int, Tk: int, q_block: int, k_block: int,
                   causal: bool = True, window: int = 0) -> np.ndarray:
    """bool [ceil(Tk/k_block)]: key blocks holding at least one key that some row of query
    block alpha may see.

    The rows of query block alpha sit at absolute positions i_first .. i_last.  Row i sees
    keys in (i - W, i] (causal, window W) or [0, i] (causal, no window); the union over the
    block's rows is (i_first - W, i_last] or [0, i_last].  A key block meets it when its
    first key is <= i_last and, with a window, its last key is > i_first - W.
    """
    t0, t1 = alpha * q_block, min(Tq, (alpha + 1) * q_block)
    i_first, i_last = Tk - Tq + t0, Tk - Tq + t1 - 1
    nKb = -(-Tk // k_block)
    j_lo = np.arange(nKb, dtype=np.int64) * k_block
    j_hi = np.minimum(j_lo + k_block, Tk) - 1
    ok = np.ones(nKb, dtype=bool)
    if causal:
        ok &= j_lo <= i_last
        if window:
            ok &= j_hi > i_first - window
    return ok


# Consistency factor of the median absolute deviation for normally distributed data:
# 1 / (the 0.75 quantile of the standard normal), so that 1.4826 * MAD estimates sigma.
MAD_NORMAL = 1.4826


def radius_zscores(radius_row: np.ndarray, rule: str = "z"):
    """How unusual each radius of one (sequence, kv head) row is, judged against the row's
    own distribution ("RBS-Attention review": a radius is large relative to the prompt,
    layer and head).

    rule "z":   (r - mean) / population std.
    rule "mad": (r - median) / (1.4826 * median(|r - median|)), the robust form: a few very
                large radii cannot inflate the scale and hide themselves.
    Returns None when the scale is zero (nothing stands out).
    """
    r = np.asarray(radius_row, dtype=np.float64)
    if rule == "z":
        mu = r.mean()
        sigma = math.sqrt(((r - mu) ** 2).mean())
        if sigma == 0.0:
            return None
        return (r - mu) / sigma
    if rule == "mad":
        med = float(np.median(r))
        mad = float(np.median(np.abs(r - med)))
        if mad == 0.0:
            return None
        return (r - med) / (MAD_NORMAL * mad)
    raise ValueError(f"unknown radius rule {rule!r}")


def select_blocks(q, centroid, radius, *, Tk: int, q_block: int = 128, k_block: int = 64,
                  causal: bool = True, window: int = 0, tau_mean: float = math.inf,
                  lambda_radius: float = 3.0, return_margins: bool = False,
                  radius_rule: str = "z", tau_bound: float | None = None, group_shared: bool = False):
    """Union of the mean-score branch and the radius-rescue branch, plus the diagonal.

    radius_rule: "z" or "mad" (see radius_zscores).  tau_bound: when given, a third branch
    keeps block beta if the Cauchy-Schwarz bound on the pooled query's score over the
    block's keys, (q_mean . c + |q_mean| r) / sqrt(d) >= max_j q_mean . k_j / sqrt(d), is at
    least the best visible mean score minus tau_bound: a block whose keys could score that
    high is kept however low its mean.  With return_margins the bound branch's margins are
    returned as a fifth array.

    group_shared: one selection per kv head, from the query rows of all its g query heads pooled
    together (the mean over heads and rows); every head of the group gets that mask.

    q: [B, H, Tq, d]; centroid: [B, n_kv, >=nKb, d]; radius: [B, n_kv, >=nKb] with
    nKb = ceil(Tk / k_block).  Returns (mask uint8 [B, H, nQb, nKb], n_selected int32
    [B, H, nQb]) and, with return_margins, also (mean_margin, z_margin) float64 arrays of
    the mask's shape: the signed distance of each block's mean score from its keep
    threshold and of its radius z-score from lambda_radius (NaN where not defined).
    """
    q = np.asarray(q, dtype=np.float64)
    centroid = np.asarray(centroid, dtype=np.float64)
    radius = np.asarray(radius, dtype=np.float64)
    B, H, Tq, d = q.shape
    n_kv = centroid.shape[1]
    g = H // n_kv
    nQb, nKb = -(-Tq // q_block), -(-Tk // k_block)
    scale = 1.0 / math.sqrt(d)
    mask = np.zeros((B, H, nQb, nKb), dtype=np.uint8)
    mean_margin = np.full((B, H, nQb, nKb), np.nan)
    z_margin = np.full((B, H, nQb, nKb), np.nan)
    bound_margin = np.full((B, H, nQb, nKb), np.nan)
    for b in range(B):
        for kvh in range(n_kv):
            z = radius_zscores(radius[b, kvh, :nKb], radius_rule)
            rescue = np.zeros(nKb, dtype=bool) if z is None else z >= lambda_radius
            c = centroid[b, kvh, :nKb]
            for h in range(kvh * g, (kvh + 1) * g):
                for alpha in range(nQb):
                    t0, t1 = alpha * q_block, min(Tq, (alpha + 1) * q_block)
                    i_first, i_last = Tk - Tq + t0, Tk - Tq + t1 - 1
                    allowed = allowed_blocks(alpha, Tq, Tk, q_block, k_block, causal, window)
                    if group_shared:
                        q_mean = q[b, kvh * g:(kvh + 1) * g, t0:t1].reshape(-1, d).mean(axis=0)
                    else:
                        q_mean = q[b, h, t0:t1].mean(axis=0)
                    s = (c @ q_mean) * scale
                    top = s[allowed].max()
                    keep_mean = s >= top - tau_mean
                    keep_bound = np.zeros(nKb, dtype=bool)
                    if tau_bound is not None:
                        ub = (c @ q_mean + np.linalg.norm(q_mean) * radius[b, kvh, :nKb]) * scale
                        keep_bound = ub >= top - tau_bound
                        bound_margin[b, h, alpha] = ub - (top - tau_bound)
                    j_lo = np.arange(nKb, dtype=np.int64) * k_block
                    j_hi = np.minimum(j_lo + k_block, Tk) - 1
                    diagonal = (j_lo <= i_last) & (j_hi >= i_first)
                    sel = allowed & (keep_mean | keep_bound | rescue | diagonal)
                    mask[b, h, alpha] = sel
                    mean_margin[b, h, alpha] = s - (top - tau_mean)
                    if z is not None:
                        z_margin[b, h, alpha] = z - lambda_radius
    n_selected = mask.sum(axis=3, dtype=np.int32)
    if return_margins:
        if tau_bound is not None:
            return mask, n_selected, mean_margin, z_margin, bound_margin
        return mask, n_selected, mean_margin, z_margin
    return mask, n_selected
