"""Pins for the block-statistics and block-selection oracle.  CPU only."""
import math

import numpy as np
import pytest
from scipy.spatial.distance import cdist

from oracle import allowed_blocks, attend, block_stats, radius_zscores, select_blocks
from workloads import planted_outliers


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_block_stats_by_direct_distances():
    """Centroids as explicit sums and radii as the largest pairwise distance from scipy's
    cdist, with a ragged last block and a shorter second sequence."""
    k = _rand((2, 3, 45, 7), 101)
    lens = np.array([45, 30])
    kb = 8
    c, r = block_stats(k, lens, kb)
    assert c.shape == (2, 3, 6, 7) and r.shape == (2, 3, 6)
    for b in range(2):
        for h in range(3):
            for beta in range(6):
                lo, hi = beta * kb, min((beta + 1) * kb, int(lens[b]))
                if lo >= hi:
                    assert np.all(c[b, h, beta] == 0) and r[b, h, beta] == 0
                    continue
                keys = k[b, h, lo:hi]
                cen = sum(keys[j] for j in range(hi - lo)) / (hi - lo)
                assert np.max(np.abs(c[b, h, beta] - cen)) <= 1e-14
                far = cdist(keys, cen[None, :]).max()
                assert abs(r[b, h, beta] - far) <= 1e-13


def test_block_stats_degenerate_blocks():
    """A block of identical keys has radius 0; a one-key block has centroid = that key."""
    k = np.tile(_rand((1, 1, 1, 5), 111), (1, 1, 9, 1))
    k[0, 0, 8] = _rand((5,), 112)
    c, r = block_stats(k, None, 4)
    assert r[0, 0, 0] == 0 and r[0, 0, 1] == 0
    assert np.array_equal(c[0, 0, 2], k[0, 0, 8]) and r[0, 0, 2] == 0


def test_radius_bounds_every_score_in_the_block():
    """Cauchy-Schwarz: for any q, max_j q.k_j <= q.c + ||q|| r over the block's keys, with
    equality at q = k_far - c (k_far the key farthest from the centroid)."""
    k = _rand((1, 1, 64 * 6, 16), 121)
    c, r = block_stats(k, None, 64)
    rng = np.random.default_rng(122)
    for beta in range(6):
        keys = k[0, 0, beta * 64:(beta + 1) * 64]
        for _ in range(20):
            qv = rng.standard_normal(16) * rng.uniform(0.1, 5)
            bound = qv @ c[0, 0, beta] + np.linalg.norm(qv) * r[0, 0, beta]
            assert (keys @ qv).max() <= bound + 1e-12
        far = keys[np.argmax(np.linalg.norm(keys - c[0, 0, beta], axis=1))]
        qv = far - c[0, 0, beta]
        bound = qv @ c[0, 0, beta] + np.linalg.norm(qv) * r[0, 0, beta]
        assert abs((keys @ qv).max() - bound) <= 1e-11


@pytest.mark.parametrize("Tq,Tk,qb,kb,W", [(40, 40, 8, 5, 0), (23, 61, 8, 4, 0), (30, 30, 7, 3, 6),
                                           (16, 50, 4, 8, 13), (1, 33, 128, 4, 9)])
def test_allowed_blocks_by_enumerating_pairs(Tq, Tk, qb, kb, W):
    """Closed-form block visibility against enumerating every (row, key) pair."""
    for alpha in range(-(-Tq // qb)):
        brute = np.zeros(-(-Tk // kb), dtype=bool)
        for t in range(alpha * qb, min(Tq, (alpha + 1) * qb)):
            i = Tk - Tq + t
            for j in range(Tk):
                if j <= i and (W == 0 or j > i - W):
                    brute[j // kb] = True
        assert np.array_equal(allowed_blocks(alpha, Tq, Tk, qb, kb, True, W), brute)
    assert np.all(allowed_blocks(0, Tq, Tk, qb, kb, causal=False))


def _brute_select(q, c, r, Tk, qb, kb, W, tau, lam):
    """Pure-Python selection: enumerated visibility, explicit means and z-scores."""
    B, H, Tq, d = q.shape
    n_kv = c.shape[1]
    g = H // n_kv
    nQb, nKb = -(-Tq // qb), -(-Tk // kb)
    out = np.zeros((B, H, nQb, nKb), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            kvh = h // g
            rr = [float(r[b, kvh, x]) for x in range(nKb)]
            mu = sum(rr) / nKb
            sd = math.sqrt(sum((x - mu) ** 2 for x in rr) / nKb)
            for alpha in range(nQb):
                rows = range(alpha * qb, min(Tq, (alpha + 1) * qb))
                vis = set()
                own = set()
                for t in rows:
                    i = Tk - Tq + t
                    own.add(i // kb)
                    for j in range(Tk):
                        if j <= i and (W == 0 or j > i - W):
                            vis.add(j // kb)
                qm = [sum(q[b, h, t, e] for t in rows) / len(rows) for e in range(d)]
                score = {x: sum(qm[e] * c[b, kvh, x, e] for e in range(d)) / math.sqrt(d) for x in vis}
                top = max(score.values())
                for x in vis:
                    keep = score[x] >= top - tau
                    keep |= sd > 0 and (rr[x] - mu) / sd >= lam
                    keep |= x in own
                    out[b, h, alpha, x] = keep
    return out


@pytest.mark.parametrize("tau,lam,W", [(0.02, 1.5, 0), (0.0, 2.0, 0), (0.05, 1.0, 40), (math.inf, 3.0, 0)])
def test_select_matches_brute_force(tau, lam, W):
    """Tiny case (T = 256, query block 32, key block 16) against the pure-Python selection."""
    B, H, n_kv, T, d, qb, kb = 1, 4, 2, 256, 8, 32, 16
    q = _rand((B, H, T, d), 131)
    k = _rand((B, n_kv, T, d), 132)
    k[0, 0, 37] *= 6.0
    k[0, 1, 200] *= 6.0
    c, r = block_stats(k, None, kb)
    mask, nsel = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, window=W, tau_mean=tau,
                               lambda_radius=lam)
    brute = _brute_select(q, c, r, T, qb, kb, W, tau, lam)
    assert np.array_equal(mask, brute)
    assert np.array_equal(nsel, brute.sum(axis=3))


def test_select_dense_limit_and_chunked_queries():
    """tau_mean = inf keeps every visible block; the block-sparse attention over that mask is
    the dense result.  Works with Tq < Tk (a chunk at an offset) and a window."""
    B, H, n_kv, Tq, Tk, d, qb, kb, W = 1, 4, 2, 40, 100, 8, 16, 8, 30
    q = _rand((B, H, Tq, d), 141)
    k = _rand((B, n_kv, Tk, d), 142)
    v = _rand((B, n_kv, Tk, d), 143)
    c, r = block_stats(k, None, kb)
    mask, _ = select_blocks(q, c, r, Tk=Tk, q_block=qb, k_block=kb, window=W)
    for alpha in range(mask.shape[2]):
        vis = allowed_blocks(alpha, Tq, Tk, qb, kb, True, W)
        assert np.array_equal(mask[0, :, alpha].astype(bool), np.tile(vis, (H, 1)))
    dense, _ = attend(q, k, v, causal=True, window=W)
    sparse, _ = attend(q, k, v, causal=True, window=W, block_mask=mask, q_block=qb, k_block=kb)
    assert np.array_equal(sparse, dense)


def test_select_keeps_diagonal_and_argmax():
    """With tau_mean = 0 and no rescue, each query block keeps exactly its best-scoring
    visible key block plus the blocks over its own positions, so no row is empty."""
    B, H, n_kv, T, d, qb, kb = 1, 2, 1, 96, 8, 16, 8
    q = _rand((B, H, T, d), 151)
    k = _rand((B, n_kv, T, d), 152)
    c, r = block_stats(k, None, kb)
    mask, nsel, mm, zm = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.0,
                                       lambda_radius=math.inf, return_margins=True)
    for h in range(H):
        for alpha in range(T // qb):
            own = set(range(alpha * qb // kb, ((alpha + 1) * qb - 1) // kb + 1))
            sel = set(np.nonzero(mask[0, h, alpha])[0])
            assert own <= sel and len(sel - own) <= 1
            vis = allowed_blocks(alpha, T, T, qb, kb)
            best = np.nanargmax(np.where(vis, mm[0, h, alpha], -np.inf))
            assert best in sel
    # Every row keeps a key: dense attention over the mask has no empty rows.
    v = _rand((B, n_kv, T, d), 153)
    _, lse = attend(q, k, v, block_mask=mask, q_block=qb, k_block=kb)
    assert np.all(np.isfinite(lse))


def test_radius_branch_rescues_planted_outliers_that_the_mean_misses():
    """"RBS-Attention review", mean dilution: one planted key of norm 8 sqrt(d) in a block of
    64 ordinary keys barely moves the centroid's score, but its radius stands far out of the
    head's radius distribution.  The radius branch finds every planted block; the mean
    branch alone, at a budget of ~10% of blocks, finds few of them."""
    n_kv, H, T, d, kb, qb = 2, 4, 64 * 160, 32, 64, 128
    k = _rand((1, n_kv, T, d), 161).astype(np.float32).astype(np.float64)
    planted = planted_outliers(162, n_kv, T, d, kb, fraction=0.05)
    for kvh, blk, tok, vec in planted:
        k[0, kvh, tok] = vec
    q = _rand((1, H, T, d), 163)
    c, r = block_stats(k, None, kb)
    for kvh in range(n_kv):
        z = radius_zscores(r[0, kvh])
        hit = {blk for kh, blk, _, _ in planted if kh == kvh}
        found = set(np.nonzero(z >= 3.0)[0])
        assert found == hit
    mask_r, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=-math.inf,
                              lambda_radius=3.0)
    _, _, mm, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.0,
                                lambda_radius=math.inf, return_margins=True)
    last = mask_r.shape[2] - 1  # the last query block sees every key block
    for h in range(H):
        hit = sorted({blk for kh, blk, _, _ in planted if kh == h // (H // n_kv)})
        rescued = set(np.nonzero(mask_r[0, h, last])[0])
        assert set(hit) <= rescued
        # mean branch with the top 10% of blocks by mean score
        s = mm[0, h, last]
        top = set(np.argsort(-s)[:len(s) // 10])
        assert len(top & set(hit)) <= len(hit) // 2


def test_mad_rule_by_hand_and_its_robustness():
    """Robust radius rule: median and median absolute deviation worked by hand on small rows
    (odd and even counts), and the reason for the rule: when one block in ten is an outlier,
    the outliers inflate the population std until none reaches z >= 3, while the median and
    MAD still place every outlier far out."""
    z = radius_zscores(np.array([1.0, 2.0, 3.0, 4.0, 100.0]), "mad")
    # median 3, deviations 2 1 0 1 97 -> MAD 1
    assert np.allclose(z, (np.array([1, 2, 3, 4, 100]) - 3.0) / 1.4826)
    z = radius_zscores(np.array([1.0, 2.0, 4.0, 10.0]), "mad")
    # median (2 + 4) / 2 = 3, deviations 2 1 1 7 -> MAD (1 + 2) / 2 = 1.5
    assert np.allclose(z, (np.array([1, 2, 4, 10]) - 3.0) / (1.4826 * 1.5))
    assert radius_zscores(np.array([5.0, 5.0, 5.0, 9.0]), "mad") is None   # MAD 0: nothing stands out
    r = 13.0 + 0.5 * _rand(200, 151)
    r[::10] = 20.0                                                         # 20 planted outliers
    assert np.sum(radius_zscores(r, "z")[::10] >= 3.0) == 0
    assert np.all(radius_zscores(r, "mad")[::10] >= 3.0)


def test_bound_branch_bounds_the_block_scores_and_contains_the_mean_branch():
    """The bound branch's score (q_mean . c + |q_mean| r) / sqrt(d) is at least the pooled
    query's score against every key of the block (checked key by key); so at equal
    thresholds the bound branch keeps every block the mean branch keeps, infinite tau_bound
    keeps every visible block, and a brute-force union matches."""
    B, H, n_kv, T, d, qb, kb = 1, 4, 2, 256, 8, 32, 16
    q = _rand((B, H, T, d), 161)
    k = _rand((B, n_kv, T, d), 162)
    k[0, 1, 90] *= 7.0
    c, r = block_stats(k, None, kb)
    nKb = T // kb
    for h in range(H):
        kvh = h // (H // n_kv)
        for alpha in range(T // qb):
            qm = q[0, h, alpha * qb:(alpha + 1) * qb].mean(axis=0)
            ub = (c[0, kvh] @ qm + np.linalg.norm(qm) * r[0, kvh]) / math.sqrt(d)
            best = (k[0, kvh].reshape(nKb, kb, d) @ qm).max(axis=1) / math.sqrt(d)
            assert np.all(ub >= best - 1e-12)
    for tau in (0.0, 0.3, 1.0):
        m_mean, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=tau, lambda_radius=math.inf)
        m_both, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=-math.inf,
                                  lambda_radius=math.inf, tau_bound=tau)
        m_mean_only = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=-math.inf,
                                    lambda_radius=math.inf)[0]                   # diagonal only
        assert np.all(m_both >= m_mean)
        assert np.all(m_both >= m_mean_only)
    dense, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=-math.inf,
                             lambda_radius=math.inf, tau_bound=math.inf)
    for alpha in range(T // qb):
        assert np.array_equal(dense[0, :, alpha], np.repeat(allowed_blocks(alpha, T, T, qb, kb, True, 0)[None], H, 0))
    # brute force of the three-branch union with the robust rule
    tau, tb, lam = 0.05, 0.2, 2.0
    mask, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=tau, lambda_radius=lam,
                            radius_rule="mad", tau_bound=tb)
    for h in range(H):
        kvh = h // (H // n_kv)
        rr = r[0, kvh]
        med = sorted(rr)[nKb // 2 - 1: nKb // 2 + 1]
        med = (med[0] + med[1]) / 2
        dev = sorted(abs(x - med) for x in rr)
        mad = (dev[nKb // 2 - 1] + dev[nKb // 2]) / 2
        for alpha in range(T // qb):
            qm = q[0, h, alpha * qb:(alpha + 1) * qb].mean(axis=0)
            vis = allowed_blocks(alpha, T, T, qb, kb, True, 0)
            s = c[0, kvh] @ qm / math.sqrt(d)
            top = s[vis].max()
            for x in range(nKb):
                ub = s[x] + np.linalg.norm(qm) * rr[x] / math.sqrt(d)
                own = alpha * qb // kb <= x <= ((alpha + 1) * qb - 1) // kb
                keep = vis[x] and (s[x] >= top - tau or ub >= top - tb or
                                   (rr[x] - med) / (1.4826 * mad) >= lam or own)
                assert mask[0, h, alpha, x] == keep


def test_group_shared_selection():
    """One mask per kv head from the group-pooled query: with one query head per kv head it is
    the per-head selection; otherwise every head of a group carries the same mask, equal to the
    per-head selection of the pooled query (the mean of the group's rows), checked by brute force."""
    B, n_kv, T, d, qb, kb = 1, 2, 256, 8, 32, 16
    k = _rand((B, n_kv, T, d), 171)
    k[0, 1, 77] *= 6.0
    c, r = block_stats(k, None, kb)
    q1 = _rand((B, n_kv, T, d), 172)
    a, _ = select_blocks(q1, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.05, lambda_radius=2.0)
    s, _ = select_blocks(q1, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.05, lambda_radius=2.0, group_shared=True)
    assert np.array_equal(a, s)
    g = 4
    q = _rand((B, n_kv * g, T, d), 173)
    m, _ = select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.05, lambda_radius=2.0, group_shared=True)
    pooled = q.reshape(B, n_kv, g, T, d).mean(axis=2)          # same block means as pooling g x rows
    ref = _brute_select(pooled, c, r, T, qb, kb, 0, 0.05, 2.0)
    for h in range(n_kv * g):
        assert np.array_equal(m[0, h], ref[0, h // g])


def test_planted_key_scale_reading():
    """The 128K workload's planted key, two readings of "8x a random unit direction": the literal
    8 u has norm 8, under an ordinary N(0, I) key's norm of about sqrt(d), so it sits inside its
    block's radius and the radius branch (z >= 3) rescues none of the planted blocks; the reading
    taken, 8 sqrt(d) u, lifts every planted block's radius out of the distribution, and the
    blocks at z >= 3 are then exactly the planted ones (the outliers themselves widen sigma, so
    their z stays near 4.5 at 5 % of blocks)."""
    from workloads import planted_outliers
    n_kv, T, d, kb = 1, 8192, 128, 64
    base = np.random.default_rng(181).standard_normal((1, n_kv, T, d))
    rescued = {}
    for name, scale in (("literal", 8.0), ("taken", None)):
        k = base.copy()
        planted = planted_outliers(182, n_kv, T, d, kb, 0.05, scale=scale)
        for kvh, blk, tok, vec in planted:
            k[0, kvh, tok] = vec
        _, radius = block_stats(k, k_block=kb)
        z = radius_zscores(radius[0, 0], "z")
        blocks = [blk for _, blk, _, _ in planted]
        rescued[name] = float(np.mean(z[blocks] >= 3.0))
        if name == "literal":
            assert np.max(z[blocks]) < 3.0
        else:
            assert np.min(z[blocks]) > 4.0
            assert set(np.flatnonzero(z >= 3.0).tolist()) == set(blocks)
    assert rescued == {"literal": 0.0, "taken": 1.0}
