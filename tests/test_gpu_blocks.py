"""GPU parity of ga_block_stats and ga_select_blocks against the float64 oracle, and of the
whole sparse prefill (stats -> selection -> block-sparse attention)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from tests.helpers import assert_close, host_tensor, to_f64
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, planted_outliers, randn_bhtd

pytestmark = pytest.mark.gpu

BAND = 1e-6   # selection decisions may differ only within this distance of a threshold


def planted_keys(seed, B, n_kv, T, d, k_block, fraction=0.05):
    bits = randn_bhtd(seed, "k", (B, n_kv, T, d), "bf16")
    for b in range(B):
        for kvh, blk, tok, vec in planted_outliers(seed + b, n_kv, T, d, k_block, fraction):
            bits[b, kvh, tok] = f32_to_bf16_bits(vec)
    ref = bf16_bits_to_f32(bits).astype(np.float64)
    dev = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return dev, ref


def compare_masks(gpu_mask, ref_mask, mean_margin, z_margin, what):
    diff = gpu_mask != ref_mask
    if not diff.any():
        return 0
    near = (np.abs(np.nan_to_num(mean_margin, nan=np.inf)) < BAND) | \
           (np.abs(np.nan_to_num(z_margin, nan=np.inf)) < BAND)
    bad = diff & ~near
    assert not bad.any(), f"{what}: {int(bad.sum())} block decisions differ outside the band"
    return int(diff.sum())


@pytest.mark.parametrize("dtype,B,n_kv,T,d,kb,lens", [
    ("bf16", 2, 2, 1000, 128, 64, [1000, 613]),
    ("bf16", 1, 3, 777, 256, 64, None),
    ("f32", 1, 2, 300, 40, 17, [250]),
    ("bf16", 1, 1, 4096, 128, 128, None),
    ("bf16", 2, 2, 700, 64, 64, [700, 333]),      # register-resident kernel, d = 64
    ("bf16", 1, 2, 517, 32, 48, [517]),           # d = 32, blocks of 48 keys, partial last block
])
def test_block_stats(dtype, B, n_kv, T, d, kb, lens):
    k, kr = host_tensor(51, "k", (B, n_kv, T, d), dtype)
    k_lens = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    c, r = ga.ga_block_stats(k, kb, k_lens=k_lens)
    cr, rr = oracle.block_stats(kr, lens, kb)
    assert np.max(np.abs(to_f64(c) - cr)) <= 1e-5
    assert np.max(np.abs(to_f64(r) - rr) / np.maximum(rr, 1.0)) <= 1e-5


@pytest.mark.parametrize("B,H,n_kv,Tq,Tk,d,qb,kb,W,tau,lam", [
    (1, 8, 2, 4096, 4096, 128, 128, 64, 0, 0.02, 3.0),
    (2, 4, 2, 2048, 2048, 128, 128, 64, 0, math.inf, 3.0),
    (1, 4, 1, 1000, 3000, 128, 128, 64, 0, 0.01, 2.0),        # chunk at an offset
    (1, 4, 2, 3000, 3000, 128, 256, 128, 700, 0.015, 2.5),    # window
    (1, 2, 2, 900, 900, 64, 100, 30, 0, 0.03, 1.5),           # odd sizes
    (1, 4, 2, 2048, 2048, 128, 128, 64, 0, -math.inf, 3.0),   # radius branch only
])
def test_select_blocks(B, H, n_kv, Tq, Tk, d, qb, kb, W, tau, lam):
    q, qr = host_tensor(61, "q", (B, H, Tq, d), "bf16")
    k, kr = planted_keys(62, B, n_kv, Tk, d, kb)
    c, r = ga.ga_block_stats(k, kb)
    mask, nsel = ga.ga_select_blocks(q, c, r, Tk=Tk, q_block=qb, k_block=kb, window=W, tau_mean=tau,
                                     lambda_radius=lam)
    cr, rr = oracle.block_stats(kr, None, kb)
    mref, nref, mm, zm = oracle.select_blocks(qr, cr, rr, Tk=Tk, q_block=qb, k_block=kb, window=W,
                                              tau_mean=tau, lambda_radius=lam, return_margins=True)
    gm = mask.cpu().numpy()
    n_diff = compare_masks(gm, mref, mm, zm, "select")
    if n_diff == 0:
        assert np.array_equal(nsel.cpu().numpy(), nref)
    assert np.array_equal(nsel.cpu().numpy(), gm.sum(axis=3))


def test_sparse_prefill_end_to_end():
    """Planted outliers: stats -> selection -> block-sparse attention.  The attention output
    equals the oracle run with the GPU's own mask; the radius branch keeps every planted
    block for the last query block; tau = inf reproduces dense attention bit for bit."""
    B, H, n_kv, T, d, qb, kb = 1, 8, 2, 4096, 128, 128, 64
    q, qr = host_tensor(71, "q", (B, H, T, d), "bf16")
    k, kr = planted_keys(72, B, n_kv, T, d, kb)
    v, vr = host_tensor(71, "v", (B, n_kv, T, d), "bf16")
    c, r = ga.ga_block_stats(k, kb)
    mask, nsel = ga.ga_select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=0.01,
                                     lambda_radius=3.0)
    out = ga.ga_attend(q, k, v, block_mask=mask, q_block=qb, k_block=kb)
    gm = mask.cpu().numpy()
    ref, _ = oracle.attend(qr, kr, vr, block_mask=gm, q_block=qb, k_block=kb)
    assert_close(to_f64(out), ref, "bf16", "sparse attention")
    planted = planted_outliers(72, n_kv, T, d, kb)
    for h in range(H):
        blocks = [blk for kvh, blk, _, _ in planted if kvh == h // (H // n_kv)]
        assert gm[0, h, -1, blocks].all()
    density = gm.sum() / sum(oracle.allowed_blocks(a, T, T, qb, kb).sum() for a in range(T // qb)) / H
    assert 0.0 < density < 0.9
    dense_mask, _ = ga.ga_select_blocks(q, c, r, Tk=T, q_block=qb, k_block=kb, tau_mean=math.inf)
    a = ga.ga_attend(q, k, v, block_mask=dense_mask, q_block=qb, k_block=kb)
    ones = torch.ones_like(dense_mask)
    b = ga.ga_attend(q, k, v, block_mask=ones, q_block=qb, k_block=kb)
    # tau = inf selects every visible block: the same tiles as an all-ones mask, same bits
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # and dense attention (another kernel at d = 128) within the bf16 tolerance
    assert_close(to_f64(a), to_f64(ga.ga_attend(q, k, v)), "bf16", "tau = inf vs dense")


@pytest.mark.parametrize("B,H,n_kv,Tq,Tk,d,qb,kb,W,tau,lam,rule,tb", [
    (1, 8, 2, 4096, 4096, 128, 128, 64, 0, 0.02, 3.0, "mad", None),             # robust rule
    (1, 4, 2, 2048, 2048, 128, 128, 64, 0, -math.inf, math.inf, "z", 0.5),      # bound branch alone
    (1, 4, 2, 3000, 3000, 128, 256, 128, 700, 0.015, 2.5, "mad", 0.3),          # all, with a window
    (2, 4, 1, 1000, 3000, 128, 128, 64, 0, 0.01, 2.0, "mad", 0.2),              # chunk at an offset
])
def test_select_blocks_variants(B, H, n_kv, Tq, Tk, d, qb, kb, W, tau, lam, rule, tb):
    """Robust (median / MAD) radius rule and the Cauchy-Schwarz bound branch.  The oracle gets
    the GPU's own centroids and radii (fp32, widened exactly), so the radius decisions of the
    two sides are the same fp64 arithmetic on the same inputs; score decisions may differ only
    within the band."""
    q, qr = host_tensor(63, "q", (B, H, Tq, d), "bf16")
    k, _ = planted_keys(64, B, n_kv, Tk, d, kb)
    c, r = ga.ga_block_stats(k, kb)
    mask, nsel = ga.ga_select_blocks(q, c, r, Tk=Tk, q_block=qb, k_block=kb, window=W, tau_mean=tau,
                                     lambda_radius=lam, radius_rule=rule, tau_bound=tb)
    out = oracle.select_blocks(qr, to_f64(c), to_f64(r), Tk=Tk, q_block=qb, k_block=kb, window=W,
                               tau_mean=tau, lambda_radius=lam, return_margins=True,
                               radius_rule=rule, tau_bound=tb)
    mref, nref, mm, zm = out[:4]
    bm = out[4] if tb is not None else np.full_like(mm, np.nan)
    gm = mask.cpu().numpy()
    diff = gm != mref
    near = (np.abs(np.nan_to_num(mm, nan=np.inf)) < BAND) | (np.abs(np.nan_to_num(bm, nan=np.inf)) < BAND)
    # radius decisions are not in the band: the two sides compute them identically
    assert not (diff & ~near).any(), f"{int((diff & ~near).sum())} decisions differ outside the band"
    if tb is not None:   # the bound (>= the mean score) keeps every block the mean branch keeps at tau_bound
        m_mean, _ = ga.ga_select_blocks(q, c, r, Tk=Tk, q_block=qb, k_block=kb, window=W, tau_mean=tb,
                                        lambda_radius=math.inf)
        assert np.all(gm >= m_mean.cpu().numpy())
    assert np.array_equal(nsel.cpu().numpy(), gm.sum(axis=3))
    if not diff.any():
        assert np.array_equal(nsel.cpu().numpy(), nref)


@pytest.mark.parametrize("B,H,n_kv,Tq,Tk,d,qb,kb,W,tau,lam", [
    (1, 8, 2, 4096, 4096, 128, 128, 64, 0, 0.02, 3.0),
    (1, 4, 1, 1000, 3000, 128, 128, 64, 0, 0.01, 2.0),        # chunk at an offset, MQA
])
def test_select_blocks_group_shared(B, H, n_kv, Tq, Tk, d, qb, kb, W, tau, lam):
    """One selection per kv head from its heads' pooled query rows; every head of the group
    carries the same mask."""
    q, qr = host_tensor(65, "q", (B, H, Tq, d), "bf16")
    k, _ = planted_keys(66, B, n_kv, Tk, d, kb)
    c, r = ga.ga_block_stats(k, kb)
    mask, nsel = ga.ga_select_blocks(q, c, r, Tk=Tk, q_block=qb, k_block=kb, window=W, tau_mean=tau,
                                     lambda_radius=lam, group_shared=True)
    mref, nref, mm, zm = oracle.select_blocks(qr, to_f64(c), to_f64(r), Tk=Tk, q_block=qb, k_block=kb, window=W,
                                              tau_mean=tau, lambda_radius=lam, return_margins=True,
                                              group_shared=True)
    gm = mask.cpu().numpy()
    g = H // n_kv
    for h in range(H):                       # the group's heads carry one mask
        assert np.array_equal(gm[:, h], gm[:, (h // g) * g])
    n_diff = compare_masks(gm, mref, mm, zm, "group-shared select")
    if n_diff == 0:
        assert np.array_equal(nsel.cpu().numpy(), nref)
    assert np.array_equal(nsel.cpu().numpy(), gm.sum(axis=3))
