"""GPU parity of token top-k sparse attention for decode ("Attention in Code", section 5):
indexer scores against the float64 oracle; the top-k selection exactly when the oracle selects
from the GPU's own fp32 scores (same tie rule), and against the oracle's float64 scores up to a
stated band around the k-th score; the gathered decode against the oracle
over the same token sets; k >= L against full attention; and the bench's full-size workload on
sampled sequences."""
import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from oracle.dsa import indexer_scores, topk_indices
from tests.helpers import assert_close, host_tensor, to_f64

pytestmark = pytest.mark.gpu


def _indexer_inputs(B, Hi, di, L, seed):
    qi, qir = host_tensor(seed, "qi", (B, 1, Hi, di), "bf16")
    ki, kir = host_tensor(seed, "ki", (B, 1, L, di), "bf16")
    wr = np.abs(np.random.default_rng(seed).standard_normal((B, Hi))).astype(np.float32)
    return qi[:, 0].contiguous(), qir[:, 0], ki[:, 0].contiguous(), kir[:, 0], torch.from_numpy(wr).cuda(), wr


@pytest.mark.parametrize("B,Hi,di,L,lens", [
    (2, 8, 128, 1000, [1000, 611]),
    (1, 4, 64, 777, None),
    (1, 16, 128, 1300, None),
    (2, 1, 64, 64, [64, 1]),
    (3, 8, 128, 530, [0, 17, 530]),    # an empty cache scores -inf everywhere
])
def test_indexer_scores(B, Hi, di, L, lens):
    qi, qir, ki, kir, wi, wr = _indexer_inputs(B, Hi, di, L, seed=501 + Hi)
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    sc = to_f64(ga.ga_dsa_indexer(qi, wi, ki, ln))
    for b in range(B):
        n = L if lens is None else lens[b]
        if n:
            ref = indexer_scores(qir[b][:, None], kir[b, :n], wr[b][:, None].astype(np.float64))[0]
            assert np.max(np.abs(sc[b, :n] - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
        assert np.all(np.isneginf(sc[b, n:]))


@pytest.mark.parametrize("B,L,topk,kind", [
    (3, 5000, 512, "normal"),
    (2, 3000, 2048, "ties"),       # integer-valued scores: many ties at the boundary
    (2, 1000, 1500, "normal"),     # topk > L: every token
    (2, 32768, 2048, "abs"),       # non-negative, concentrated: the top digits fall in one or two bins
    (1, 50000, 2048, "abs"),       # a row too long to stage in shared memory
    (2, 30000, 2048, "binary"),    # two values: the chosen bin never shrinks to a candidate list
])
def test_topk_indices_exact(B, L, topk, kind):
    rng = np.random.default_rng(511)
    s = rng.standard_normal((B, L)).astype(np.float32)
    if kind == "ties":
        s = np.floor(s * 3.0).astype(np.float32)
    elif kind == "abs":
        s = np.abs(s)
    elif kind == "binary":
        s = (s > 0).astype(np.float32)
    lens = [L, L // 2, L - 7][:B]
    scores = torch.from_numpy(s).cuda()
    idx, n_sel = ga.ga_topk_indices(scores, topk, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    idx, n_sel = idx.cpu().numpy(), n_sel.cpu().numpy()
    for b in range(B):
        ref = topk_indices(s[b, :lens[b]], np.ones(lens[b], bool), topk)
        assert n_sel[b] == ref.size
        assert np.array_equal(idx[b, :ref.size], ref)
        assert np.all(idx[b, ref.size:] == -1)


def _decode_inputs(B, H, n_kv, Lm, d, Hi, di, seed):
    q, qr = host_tensor(seed, "q", (B, H, 1, d), "bf16")
    k, kr = host_tensor(seed, "k", (B, n_kv, Lm, d), "bf16")
    v, vr = host_tensor(seed, "v", (B, n_kv, Lm, d), "bf16")
    qi, qir, ki, kir, wi, wr = _indexer_inputs(B, Hi, di, Lm, seed + 1)
    return (q, k, v, qi, wi, ki), (qr, kr, vr, qir, kir, wr)


@pytest.mark.parametrize("B,H,n_kv,Lm,d,Hi,di,topk,lens,use_sink", [
    (2, 8, 2, 3000, 128, 8, 128, 512, [3000, 1234], False),
    (2, 4, 1, 2000, 256, 4, 64, 300, [2000, 150], True),     # d = 256; a sequence shorter than k
    (1, 4, 4, 900, 64, 2, 64, 200, [600], False),            # d = 64; cache rows past the length hold NaN
])
def test_dsa_decode_matches_oracle(B, H, n_kv, Lm, d, Hi, di, topk, lens, use_sink):
    dev, ref = _decode_inputs(B, H, n_kv, Lm, d, Hi, di, seed=521)
    q, k, v, qi, wi, ki = dev
    qr, kr, vr, qir, kir, wr = ref
    sink = skr = None
    if use_sink:
        skr = np.random.default_rng(7).standard_normal(H).astype(np.float32)
        sink = torch.from_numpy(skr).cuda()
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for b, n in enumerate(lens):               # rows no selection may read
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    out, idx, n_sel, scores = ga.dsa_decode(q, k, v, qi, wi, ki, topk, ln, sink=sink)
    assert ga.ga_read_device_status() == ga.GA_OK
    # the oracle attends over the tokens its own top-k picks from the GPU's scores
    expect, chosen = oracle.dsa_decode(qr, kr, vr, qir, kir, wr, lens, topk, sink=skr, scores=to_f64(scores))
    idx, n_sel = idx.cpu().numpy(), n_sel.cpu().numpy()
    for b in range(B):
        assert np.array_equal(idx[b, :n_sel[b]], chosen[b])
    assert_close(to_f64(out), expect, "bf16", "dsa decode")


def test_dsa_topk_at_least_length_is_full_attention():
    """k >= L: every cached token is read, and the result is full decode attention."""
    B, H, n_kv, Lm, d = 2, 8, 2, 700, 128
    dev, ref = _decode_inputs(B, H, n_kv, Lm, d, 8, 128, seed=531)
    q, k, v, qi, wi, ki = dev
    qr, kr, vr = ref[:3]
    out, idx, n_sel, _ = ga.dsa_decode(q, k, v, qi, wi, ki, 1024)
    assert n_sel.cpu().tolist() == [Lm, Lm]
    full, _ = oracle.attend(qr, kr, vr, causal=True)
    assert_close(to_f64(out), full, "bf16", "dsa k >= L")


def test_dsa_full_size_sampled():
    """The bench's workload (B64 H32 Hkv8 d128, lengths U[16384, 32768], indexer 8 heads x 128,
    k = 2048): scores, selection and output checked on sampled sequences."""
    from workloads import bf16_bits_to_f32, randn_bhtd, uniform_lengths
    B, H, n_kv, Lm, d, Hi, di, topk = 64, 32, 8, 32768, 128, 8, 128, 2048
    lens = uniform_lengths(541, B, 16384, 32768)
    q, qr = host_tensor(541, "q", (B, H, 1, d), "bf16")
    kb = randn_bhtd(541, "k", (B, n_kv, Lm, d), "bf16")      # bf16 bits; float64 only where sampled
    vb = randn_bhtd(541, "v", (B, n_kv, Lm, d), "bf16")
    k = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).cuda()
    qi, qir = host_tensor(542, "qi", (B, 1, Hi, di), "bf16")
    qi, qir = qi[:, 0].contiguous(), qir[:, 0]
    kib = randn_bhtd(542, "ki", (B, 1, Lm, di), "bf16")[:, 0]
    ki = torch.from_numpy(np.ascontiguousarray(kib).view(np.int16)).view(torch.bfloat16).cuda()
    wr = np.abs(np.random.default_rng(542).standard_normal((B, Hi))).astype(np.float32)
    wi = torch.from_numpy(wr).cuda()
    out, idx, n_sel, scores = ga.dsa_decode(q, k, v, qi, wi, ki, topk, torch.from_numpy(lens).cuda())
    assert ga.ga_read_device_status() == ga.GA_OK
    sc, idx, n_sel = to_f64(scores), idx.cpu().numpy(), n_sel.cpu().numpy()
    f64 = lambda x: bf16_bits_to_f32(x).astype(np.float64)
    for b in np.random.default_rng(543).choice(B, size=3, replace=False):
        n = int(lens[b])
        ref_sc = indexer_scores(qir[b][:, None], f64(kib[b, :n]), wr[b][:, None].astype(np.float64))[0]
        tol = 1e-5 * max(1.0, np.max(np.abs(ref_sc)))
        assert np.max(np.abs(sc[b, :n] - ref_sc)) <= tol
        chosen = topk_indices(sc[b, :n], np.ones(n, bool), topk)
        assert np.array_equal(idx[b, :n_sel[b]], chosen)
        _topk_against_f64(idx[b], int(n_sel[b]), ref_sc, topk, tol)
        expect, _ = oracle.attend(qr[b:b + 1], f64(kb[b:b + 1, :, chosen]), f64(vb[b:b + 1, :, chosen]),
                                  causal=False)
        assert_close(to_f64(out[b:b + 1]), expect, "bf16", f"dsa full size b={b}")


def _topk_against_f64(idx_row, n_sel, ref_sc, topk, tol):
    """The GPU's selection for one sequence against the oracle's top-k of the oracle's own
    float64 indexer scores.  Both scores agree within tol (asserted by the caller), so a token
    can be decided differently only when its float64 score lies within 2 tol of the k-th largest
    float64 score; every other decision must match.  Returns the number of tokens decided
    differently (all of them inside that band)."""
    n = ref_sc.shape[0]
    want = topk_indices(ref_sc, np.ones(n, bool), topk)
    got = idx_row[:n_sel]
    assert n_sel == want.size
    assert np.all(np.diff(got) > 0)                       # increasing positions, no repeats
    if want.size == n:
        assert np.array_equal(got, want)
        return 0
    kth = np.sort(ref_sc)[::-1][topk - 1]
    differ = np.setxor1d(got, want)
    near = np.abs(ref_sc[differ] - kth) <= 2 * tol
    assert near.all(), f"{int((~near).sum())} tokens outside the band of the k-th score decided differently"
    return int(differ.size)


@pytest.mark.parametrize("B,Hi,di,L,topk,lens", [
    (4, 8, 128, 20000, 2048, [20000, 15000, 9001, 2048]),
    (2, 4, 64, 6000, 500, [6000, 4999]),
])
def test_topk_against_float64_indexer_scores(B, Hi, di, L, topk, lens):
    """Top-k parity decided on the oracle's float64 scores, not on the GPU's fp32 ones: the
    indexer runs on the GPU, its selection is compared with the float64 oracle's indexer and
    top-k, and tokens may differ only inside the band that the score tolerance allows."""
    qi, qir, ki, kir, wi, wr = _indexer_inputs(B, Hi, di, L, seed=561 + di)
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scores = ga.ga_dsa_indexer(qi, wi, ki, ln)
    idx, n_sel = ga.ga_topk_indices(scores, topk, ln)
    sc, idx, n_sel = to_f64(scores), idx.cpu().numpy(), n_sel.cpu().numpy()
    differ = 0
    for b in range(B):
        n = lens[b]
        ref_sc = indexer_scores(qir[b][:, None], kir[b, :n], wr[b][:, None].astype(np.float64))[0]
        tol = 1e-5 * max(1.0, np.max(np.abs(ref_sc)))
        assert np.max(np.abs(sc[b, :n] - ref_sc)) <= tol
        differ += _topk_against_f64(idx[b], int(n_sel[b]), ref_sc, topk, tol)
    print(f"top-k vs float64 scores: {differ} token decisions differ, all within the band")


@pytest.mark.parametrize("Lm,topk", [(500, 64), (6000, 5000)])   # one key chunk; ten chunks + combine
def test_dsa_decode_empty_cache_row_is_zero(Lm, topk):
    """A sequence with no cached token: the indexer scores -inf, top-k selects nothing, and the
    gathered decode writes a zero row (the sink carries no value); the other sequence is exact."""
    B, H, n_kv, d = 2, 8, 2, 128
    dev, ref = _decode_inputs(B, H, n_kv, Lm, d, 8, 128, seed=551)
    q, k, v, qi, wi, ki = dev
    qr, kr, vr, qir, kir, wr = ref
    lens = [Lm, 0]
    skr = np.linspace(-1.0, 1.0, H).astype(np.float32)
    out, idx, n_sel, scores = ga.dsa_decode(q, k, v, qi, wi, ki, topk,
                                            torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                            sink=torch.from_numpy(skr).cuda())
    assert ga.ga_read_device_status() == ga.GA_OK
    assert n_sel.cpu().tolist() == [min(topk, Lm), 0]
    assert torch.all(out[1] == 0)
    expect, _ = oracle.dsa_decode(qr, kr, vr, qir, kir, wr, lens, topk, sink=skr, scores=to_f64(scores))
    assert_close(to_f64(out), expect, "bf16", "dsa empty cache")
