"""Pins for the attention oracle: each check ties the oracle to something other than itself
(scalar brute force, a library routine, a closed form, or a worked example printed on the
pages).  CPU only."""
import math
import os
import zlib

import numpy as np
from scipy.special import logsumexp
import pytest
import torch

from oracle import attend, positions, ring_contents, ring_decode, visible

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _brute_attend(q, k, v, causal, window, sink, block_mask, q_block, k_block, k_lens):
    """Scalar triple loop in pure Python: every score, every exponential, one at a time."""
    B, H, Tq, d = q.shape
    n_kv = k.shape[1]
    out = np.zeros((B, H, Tq, v.shape[-1]))
    lse = np.full((B, H, Tq), -math.inf)
    for b in range(B):
        Tk = k.shape[2] if k_lens is None else int(k_lens[b])
        for h in range(H):
            kvh = h // (H // n_kv)
            for t in range(Tq):
                i = Tk - Tq + t
                scores = []
                for j in range(Tk):
                    if causal and j > i:
                        continue
                    if window and j <= i - window:
                        continue
                    if block_mask is not None and not block_mask[b, h, t // q_block, j // k_block]:
                        continue
                    dot = 0.0
                    for c in range(d):
                        dot += q[b, h, t, c] * k[b, kvh, j, c]
                    scores.append((j, dot / math.sqrt(d)))
                logits = [s for _, s in scores] + ([float(sink[h])] if sink is not None else [])
                if not logits:
                    continue
                m = max(logits)
                Z = sum(math.exp(x - m) for x in logits)
                for j, s in scores:
                    out[b, h, t] += math.exp(s - m) / Z * v[b, kvh, j]
                lse[b, h, t] = m + math.log(Z)
    return out, lse


@pytest.mark.parametrize("case", [
    dict(B=1, H=4, n_kv=2, Tq=9, Tk=9, d=5, causal=True, window=0, sink=False, bm=False),
    dict(B=2, H=6, n_kv=3, Tq=5, Tk=13, d=4, causal=True, window=3, sink=True, bm=False),
    dict(B=1, H=2, n_kv=1, Tq=7, Tk=7, d=3, causal=False, window=0, sink=True, bm=False),
    dict(B=2, H=4, n_kv=4, Tq=11, Tk=20, d=6, causal=True, window=0, sink=False, bm=True),
    dict(B=2, H=4, n_kv=1, Tq=3, Tk=17, d=2, causal=True, window=5, sink=True, bm=True, lens=True),
])
def test_attend_matches_scalar_brute_force(case):
    rng_seed = zlib.crc32(repr(sorted(case.items())).encode()) & 0xFFFF
    B, H, n_kv, Tq, Tk, d = (case[x] for x in ("B", "H", "n_kv", "Tq", "Tk", "d"))
    q = _rand((B, H, Tq, d), rng_seed)
    k = _rand((B, n_kv, Tk, d), rng_seed + 1)
    v = _rand((B, n_kv, Tk, d), rng_seed + 2)
    sink = _rand((H,), rng_seed + 3) if case["sink"] else None
    qb, kb = 4, 3
    bm = None
    if case["bm"]:
        bm = (np.random.default_rng(rng_seed + 4).random((B, H, -(-Tq // qb), -(-Tk // kb))) < 0.6)
        bm = bm.astype(np.uint8)
    k_lens = None
    if case.get("lens"):
        k_lens = np.array([Tk, Tk - 4])
    o1, l1 = attend(q, k, v, causal=case["causal"], window=case["window"], sink=sink,
                    block_mask=bm, q_block=qb, k_block=kb, k_lens=k_lens)
    o2, l2 = _brute_attend(q, k, v, case["causal"], case["window"], sink, bm, qb, kb, k_lens)
    assert np.max(np.abs(o1 - o2)) <= 1e-13
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    assert np.max(np.abs(l1[fin] - l2[fin]), initial=0.0) <= 1e-13


@pytest.mark.parametrize("n_kv,window,sink", [(8, 0, False), (2, 0, True), (1, 6, False), (2, 11, True)])
def test_attend_matches_torch_sdpa(n_kv, window, sink):
    """torch SDPA in float64 with K/V expanded per query head and a boolean mask built from
    torch.tril / torch.triu offsets; the sink case appends the sink logit as an extra column."""
    B, H, Tq, Tk, d = 2, 8, 24, 40, 16
    q = _rand((B, H, Tq, d), 11)
    k = _rand((B, n_kv, Tk, d), 12)
    v = _rand((B, n_kv, Tk, d), 13)
    sk = _rand((H,), 14) * 2 if sink else None
    o, lse = attend(q, k, v, causal=True, window=window, sink=sk)

    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    g = H // n_kv
    K = tk.repeat_interleave(g, dim=1)
    V = tv.repeat_interleave(g, dim=1)
    ones = torch.ones(Tq, Tk, dtype=torch.bool)
    m = ones.tril(diagonal=Tk - Tq)
    if window:
        m &= ones.triu(diagonal=Tk - Tq - window + 1)
    if sink:
        s = tq @ K.transpose(-1, -2) / math.sqrt(d)
        s = s.masked_fill(~m, -math.inf)
        col = torch.from_numpy(sk).view(1, H, 1, 1).expand(B, H, Tq, 1)
        p = torch.cat([s, col], dim=-1).softmax(-1)[..., :-1]
        ref = p @ V
        ref_lse = torch.logsumexp(torch.cat([s, col], dim=-1), dim=-1)
    else:
        ref = torch.nn.functional.scaled_dot_product_attention(tq, K, V, attn_mask=m)
        s = (tq @ K.transpose(-1, -2) / math.sqrt(d)).masked_fill(~m, -math.inf)
        ref_lse = torch.logsumexp(s, dim=-1)
        # the normaliser once more from scipy over numpy scores (an independent library)
        sn = np.einsum("bhtd,bhsd->bhts", q, K.numpy()) / math.sqrt(d)
        assert np.max(np.abs(lse - logsumexp(np.where(m.numpy(), sn, -np.inf), axis=-1))) <= 1e-12
    assert np.max(np.abs(o - ref.numpy())) <= 1e-12
    assert np.max(np.abs(lse - ref_lse.numpy())) <= 1e-12


@pytest.mark.parametrize("n_kv", [8, 2, 1])
def test_token_by_token_equals_all_at_once(n_kv):
    """"Attention in Code" s.1: feeding a 40-token sequence one token at a time through the
    cache gives the all-at-once result (MHA, GQA and MQA).  Each decode step is a call with
    Tq = 1 and Tk = t + 1, so the query's absolute position must be Tk - 1."""
    H, T, d = 8, 40, 16
    q = _rand((1, H, T, d), 21)
    k = _rand((1, n_kv, T, d), 22)
    v = _rand((1, n_kv, T, d), 23)
    full, full_lse = attend(q, k, v, causal=True)
    for t in range(T):
        step, step_lse = attend(q[:, :, t:t + 1], k[:, :, :t + 1], v[:, :, :t + 1], causal=True)
        assert np.max(np.abs(step[:, :, 0] - full[:, :, t])) <= 1e-13
        assert np.max(np.abs(step_lse[:, :, 0] - full_lse[:, :, t])) <= 1e-13
    # The same steps expressed with a cache allocated at T and per-sequence lengths.
    for t in range(T):
        step, _ = attend(q[:, :, t:t + 1], k, v, causal=True, k_lens=np.array([t + 1]))
        assert np.max(np.abs(step[:, :, 0] - full[:, :, t])) <= 1e-13


def test_chunked_prefill_uses_absolute_positions():
    """"Express note": a chunk of new queries after a cache offset must be masked by absolute
    position.  Chunks of 7 rows over a 30-token prompt reproduce the all-at-once rows; using
    the in-chunk index instead (a block starting at position 0) does not."""
    H, n_kv, T, d = 4, 2, 30, 8
    q = _rand((1, H, T, d), 31)
    k = _rand((1, n_kv, T, d), 32)
    v = _rand((1, n_kv, T, d), 33)
    full, _ = attend(q, k, v, causal=True, window=9)
    for s in range(0, T, 7):
        e = min(T, s + 7)
        part, _ = attend(q[:, :, s:e], k[:, :, :e], v[:, :, :e], causal=True, window=9)
        assert np.max(np.abs(part - full[:, :, s:e])) <= 1e-13
    wrong = visible(np.arange(7), 14)  # in-block index for a chunk at offset 7
    right = visible(positions(7, 14), 14)
    assert not np.array_equal(wrong, right)


def test_gqa_equals_mha_with_replicated_kv_weights():
    """"Attention in Code" s.1: n_kv = 2 GQA equals 8-head MHA whose K/V projection weights
    are copied across the 4 heads of each group."""
    rng = np.random.default_rng(41)
    T, dim, H, n_kv, d = 20, 32, 8, 2, 16
    g = H // n_kv
    x = rng.standard_normal((T, dim))
    wq = rng.standard_normal((dim, H * d)) / math.sqrt(dim)
    wk = rng.standard_normal((dim, n_kv * d)) / math.sqrt(dim)
    wv = rng.standard_normal((dim, n_kv * d)) / math.sqrt(dim)
    q = (x @ wq).reshape(T, H, d).transpose(1, 0, 2)[None]
    k = (x @ wk).reshape(T, n_kv, d).transpose(1, 0, 2)[None]
    v = (x @ wv).reshape(T, n_kv, d).transpose(1, 0, 2)[None]
    gqa, _ = attend(q, k, v, causal=True)
    wk_mha = np.concatenate([wk[:, (h // g) * d:(h // g + 1) * d] for h in range(H)], axis=1)
    wv_mha = np.concatenate([wv[:, (h // g) * d:(h // g + 1) * d] for h in range(H)], axis=1)
    k8 = (x @ wk_mha).reshape(T, H, d).transpose(1, 0, 2)[None]
    v8 = (x @ wv_mha).reshape(T, H, d).transpose(1, 0, 2)[None]
    mha, _ = attend(q, k8, v8, causal=True)
    assert np.max(np.abs(gqa - mha)) <= 1e-13
    # A head-to-group mapping of h % n_kv would not match.
    k_mod = np.stack([k[0, h % n_kv] for h in range(H)])[None]
    v_mod = np.stack([v[0, h % n_kv] for h in range(H)])[None]
    other, _ = attend(q, k_mod, v_mod, causal=True)
    assert np.max(np.abs(other - gqa)) > 1e-3


def _golden_masks():
    sets, cur = {}, None
    with open(os.path.join(GOLDEN, "swa_n8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line[1:-1]
                sets[cur] = []
            else:
                sets[cur].append([c == "1" for c in line])
    return {k_: np.array(v_) for k_, v_ in sets.items()}


def test_visible_sets_match_window_diagram():
    """"Attention Variants", sliding-window diagram: n = 8 positions, full causal and W = 4."""
    g = _golden_masks()
    i = positions(8, 8)
    assert np.array_equal(visible(i, 8, causal=True, window=0), g["full_causal"])
    assert np.array_equal(visible(i, 8, causal=True, window=4), g["window_4"])


def test_window_edge_cases():
    """"Attention Variants", exercise 1 and step 2: window >= n reproduces full causal
    attention bit for bit, and window = 1 lets every token see only itself."""
    q = _rand((1, 4, 12, 8), 51)
    k = _rand((1, 2, 12, 8), 52)
    v = _rand((1, 2, 12, 8), 53)
    full, _ = attend(q, k, v, causal=True)
    for w in (12, 13, 1000):
        wo, _ = attend(q, k, v, causal=True, window=w)
        assert np.array_equal(wo, full)
    one, _ = attend(q, k, v, causal=True, window=1)
    expect = np.repeat(v, 2, axis=1)
    assert np.array_equal(one, expect)


def test_ring_cache_equals_window_mask_and_forgets_token_zero():
    """"Attention in Code" s.2: a W = 8 ring cache over 50 tokens gives the window-masked
    all-at-once result at every step, and changing token 0's value by 100 leaves every
    output from step 8 on exactly unchanged."""
    H, n_kv, T, d, W = 4, 2, 50, 16, 8
    q = _rand((H, T, d), 61)
    k = _rand((n_kv, T, d), 62)
    v = _rand((n_kv, T, d), 63)
    ring = ring_decode(q, k, v, W)
    masked, _ = attend(q[None], k[None], v[None], causal=True, window=W)
    assert np.max(np.abs(ring - masked[0])) <= 1e-13
    v2 = v.copy()
    v2[:, 0] += 100.0
    masked2, _ = attend(q[None], k[None], v2[None], causal=True, window=W)
    assert np.array_equal(masked2[0, :, W:], masked[0, :, W:])
    assert np.max(np.abs(masked2[0, :, :W] - masked[0, :, :W])) > 1.0
    ring2 = ring_decode(q, k, v2, W)
    assert np.array_equal(ring2[:, W:], ring[:, W:])


def test_ring_contents_slot_rule_and_decode_consistency():
    """"Attention in Code" s.2: after n tokens slot s holds the newest token t < n with
    t mod W = s (checked by enumerating the tokens), never-written slots stay zero, and the
    last ring_decode output is plain attention over the min(n, W) filled slots in slot order."""
    n_kv, T, d, W = 2, 23, 4, 8
    k = _rand((n_kv, T, d), 64)
    v = _rand((n_kv, T, d), 65)
    for n in (0, 3, 8, 9, 23):
        rk, rv = ring_contents(k, v, W, n)
        for slot in range(W):
            owners = [t for t in range(n) if t % W == slot]
            if owners:
                assert np.array_equal(rk[:, slot], k[:, max(owners)])
                assert np.array_equal(rv[:, slot], v[:, max(owners)])
            else:
                assert not rk[:, slot].any() and not rv[:, slot].any()
    H = 4
    q = _rand((H, T, d), 66)
    ring = ring_decode(q, k, v, W)
    rk, rv = ring_contents(k, v, W)
    last, _ = attend(q[None, :, T - 1:], rk[None], rv[None], causal=False)
    assert np.max(np.abs(ring[:, T - 1] - last[0, :, 0])) <= 1e-13


def test_sink_closed_forms():
    """"Attention in Code" s.3: a sink of -inf gives plain attention exactly; with a sink the
    weights on the keys sum to 1 / (1 + e^(sink - lse_plain)) < 1; a large sink drives the
    output towards zero (about e^-sink relative)."""
    H, T, d = 4, 16, 8
    q = _rand((1, H, T, d), 71)
    k = _rand((1, 2, T, d), 72)
    v = _rand((1, 2, T, d), 73)
    plain, lse = attend(q, k, v, causal=True)
    neg, neg_lse = attend(q, k, v, causal=True, sink=np.full(H, -np.inf))
    assert np.array_equal(neg, plain)
    assert np.array_equal(neg_lse, lse)
    sink = _rand((H,), 74)
    ones = np.ones_like(v)
    wsum, lse_s = attend(q, k, ones, causal=True, sink=sink)
    expect = 1.0 / (1.0 + np.exp(sink[None, :, None] - lse))
    assert np.max(np.abs(wsum[..., 0] - expect)) <= 1e-13
    assert np.all(wsum < 1.0)
    assert np.max(np.abs(lse_s - np.logaddexp(lse, sink[None, :, None]))) <= 1e-13
    with_sink, _ = attend(q, k, v, causal=True, sink=sink)
    scale = np.exp(lse - lse_s)[..., None]
    assert np.max(np.abs(with_sink - plain * scale)) <= 1e-13
    big, _ = attend(q, k, v, causal=True, sink=np.full(H, 20.0))
    ratio = np.linalg.norm(big) / np.linalg.norm(plain)
    assert 1e-11 < ratio < 1e-6


def test_uniform_keys_give_mean_of_visible_values():
    """Closed form: when every key is the same vector all visible scores are equal, so each
    output is the plain mean of the values the row may see."""
    T, d, W = 20, 4, 6
    k = np.tile(_rand((1, 1, 1, d), 81), (1, 1, T, 1))
    q = _rand((1, 2, T, d), 82)
    v = _rand((1, 1, T, d), 83)
    o, _ = attend(q, k, v, causal=True, window=W)
    for t in range(T):
        lo = max(0, t - W + 1)
        assert np.max(np.abs(o[0, :, t] - v[0, 0, lo:t + 1].mean(axis=0))) <= 1e-14


def test_empty_rows_and_block_mask_expansion():
    """A row left with no key and no sink returns 0 with lse = -inf; with a sink it returns 0
    with lse = sink.  A block mask equals the same mask expanded to single keys."""
    q = _rand((1, 2, 8, 4), 91)
    k = _rand((1, 1, 8, 4), 92)
    v = _rand((1, 1, 8, 4), 93)
    bm = np.zeros((1, 2, 2, 2), dtype=np.uint8)
    bm[0, 0, 1, 0] = 1
    o, lse = attend(q, k, v, causal=True, block_mask=bm, q_block=4, k_block=4)
    assert np.all(o[0, 1] == 0) and np.all(np.isneginf(lse[0, 1]))
    assert np.all(o[0, 0, :4] == 0) and np.all(np.isfinite(lse[0, 0, 4:]))
    o2, lse2 = attend(q, k, v, causal=True, block_mask=bm, q_block=4, k_block=4,
                      sink=np.array([0.5, -0.25]))
    assert np.all(o2[0, 1] == 0) and np.allclose(lse2[0, 1], -0.25)
    # Key-level expansion of the block mask through a per-key mask of size 1.
    fine = np.repeat(np.repeat(bm, 4, axis=2), 4, axis=3)
    o3, _ = attend(q, k, v, causal=True, block_mask=fine, q_block=1, k_block=1)
    assert np.array_equal(o3, o)


def test_padding_mask_example_is_the_key_length_mask():
    """"Attention Masking" Example 1: the batch [[1, 2, 3, 0], [4, 5, 0, 0]] (id 0 = padding) has
    the padding pattern of key lengths 3 and 2, and attention with those lengths equals the guide's
    form -- -1e9 added to the padded keys' scores before the softmax -- written out with NumPy
    (e^-1e9 underflows to exactly 0 in float64)."""
    sec, cur = {}, None
    for line in open(os.path.join(GOLDEN, "padding_mask_example1.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = line[1:-1]
            sec[cur] = []
        else:
            sec[cur].append(line)
    ids = np.array([[int(x) for x in row.split()] for row in sec["input_ids"]])
    keys = np.array([[c == "1" for c in row] for row in sec["keys"]])
    assert np.array_equal(ids != 0, keys)
    lens = keys.sum(axis=1)
    assert lens.tolist() == [3, 2]
    B, H, T, d = 2, 4, 4, 8
    # two query rows (the boundary keeps Tq <= each sequence's key count) over the padded keys
    q, k, v = _rand((B, H, 2, d), 191), _rand((B, 2, T, d), 192), _rand((B, 2, T, d), 193)
    ours, _ = attend(q, k, v, k_lens=lens, causal=False)
    kk, vv = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)             # GQA: head h reads kv h // 2
    s = q @ np.swapaxes(kk, -1, -2) / math.sqrt(d) + np.where(keys, 0.0, -1e9)[:, None, None, :]
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    guide = (p / p.sum(axis=-1, keepdims=True)) @ vv
    assert np.max(np.abs(ours - guide)) <= 1e-14


@pytest.mark.parametrize("sink_kind", ["random", "large", "minus_inf"])
def test_ring_decode_with_sink_equals_window_mask_with_sink(sink_kind):
    """"Attention in Code" s.2 and s.3 together: a W = 8 ring over 50 tokens with a per-head sink
    gives, at every step, what the pinned attend gives under the window mask with the same sink
    (the sink joins the normaliser of every row and carries no value), so a wrong sink term in
    the ring's own softmax (scaled by 1/sqrt(d), given a value, or taken against the wrong row
    maximum) shows up here."""
    H, n_kv, T, d, W = 4, 2, 50, 16, 8
    q = _rand((H, T, d), 81)
    k = _rand((n_kv, T, d), 82)
    v = _rand((n_kv, T, d), 83)
    sink = {"random": _rand((H,), 84), "large": np.array([6.0, 9.0, 12.0, 15.0]),
            "minus_inf": np.full(H, -np.inf)}[sink_kind]
    ring = ring_decode(q, k, v, W, sink=sink)
    masked, _ = attend(q[None], k[None], v[None], causal=True, window=W, sink=sink)
    assert np.max(np.abs(ring - masked[0])) <= 1e-13
    if sink_kind == "minus_inf":
        assert np.array_equal(ring, ring_decode(q, k, v, W))
    else:
        plain = ring_decode(q, k, v, W)
        assert np.all(np.linalg.norm(ring, axis=-1) < np.linalg.norm(plain, axis=-1))
