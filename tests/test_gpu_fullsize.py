"""Parity at the benchmark's full sizes, in the launch configuration bench.py times.

The GPU runs each workload whole; the oracle recomputes 256 sampled query rows per
(sequence, head) -- always including the first and last rows, query-block edges and window
edges -- and, for the 128K sparse workload, the block statistics and the selection of every
block exactly."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from tests.helpers import assert_close, to_f64
from workloads import (bf16_bits_to_f32, f32_to_bf16_bits, get_config, planted_outliers, randn_bhtd,
                       sample_rows, uniform_lengths)

pytestmark = pytest.mark.gpu


def upload(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def check_rows(out, qbits, kbits, vbits, rows, heads, *, lens=None, window=0, sink=None, mask=None,
               what=""):
    """Oracle on the sampled rows of the listed (b, h) pairs."""
    B, H, Tq, d = qbits.shape
    g = H // kbits.shape[1]
    o = out[:, :, rows].float().cpu().numpy()
    for b, h in heads:
        kvh = h // g
        sel_mask = None if mask is None else mask[b:b + 1, h:h + 1]
        ref, _ = oracle.attend(f64(qbits[b:b + 1, h:h + 1]), f64(kbits[b:b + 1, kvh:kvh + 1]),
                               f64(vbits[b:b + 1, kvh:kvh + 1]), rows=rows,
                               k_lens=None if lens is None else [int(lens[b])], window=window,
                               sink=None if sink is None else sink[h:h + 1], block_mask=sel_mask)
        assert_close(o[b, h][None, None].astype(np.float64), ref, "bf16", f"{what} b={b} h={h}")


def test_dense_causal_prefill_8k():
    c = get_config(2)
    shape_q = (c.batch, c.n_heads, c.Tq, c.d)
    shape_k = (c.batch, c.n_kv, c.Tk, c.d)
    qb, kb, vb = (randn_bhtd(c.seed, t, s) for t, s in (("q", shape_q), ("k", shape_k), ("v", shape_k)))
    out = ga.ga_attend(upload(qb), upload(kb), upload(vb))
    assert ga.ga_read_device_status() == ga.GA_OK
    rows = sample_rows(c.Tq, 256, seed=c.seed)
    heads = [(b, h) for b in range(c.batch) for h in (0, 5, 13, 31)]
    check_rows(out, qb, kb, vb, rows, heads, what="config 2")


def test_decode_and_chunk_32k():
    c = get_config(3)
    lens = uniform_lengths(c.seed, c.batch, *c.k_len_range)
    shape_k = (c.batch, c.n_kv, c.Tk, c.d)
    kb = randn_bhtd(c.seed, "k", shape_k, lengths=lens)
    vb = randn_bhtd(c.seed, "v", shape_k, lengths=lens)
    k, v = upload(kb), upload(vb)
    k_lens = torch.from_numpy(lens).cuda()
    # decode, Tq = 1: every (b, h) row is cheap for the oracle -- check a third of them
    qb = randn_bhtd(c.seed, "q", (c.batch, c.n_heads, 1, c.d))
    out = ga.ga_attend(upload(qb), k, v, k_lens=k_lens)
    assert ga.ga_read_device_status() == ga.GA_OK
    heads = [(b, h) for b in range(0, c.batch, 3) for h in range(c.n_heads)]
    check_rows(out, qb, kb, vb, np.array([0]), heads, lens=lens, what="decode")
    # chunk, Tq = 512 at absolute positions Tk_b - 512 + t
    Tq = c.extra["chunk_Tq"]
    qb = randn_bhtd(c.seed, "q512", (c.batch, c.n_heads, Tq, c.d))
    out = ga.ga_attend(upload(qb), k, v, k_lens=k_lens)
    assert ga.ga_read_device_status() == ga.GA_OK
    rows = sample_rows(Tq, 64, seed=c.seed, q_block=128)
    heads = [(b, h) for b in (0, 17, 63) for h in (0, 9, 31)]
    check_rows(out, qb, kb, vb, rows, heads, lens=lens, what="chunk")


@pytest.mark.parametrize("B,H,n_kv,Tq,d,Tk,lens", [
    (1, 8, 4, 640, 128, 98304, [98299]),
    (1, 4, 2, 384, 256, 98304, [98299]),
    (3, 4, 2, 384, 128, 65536, [65536, 40000, 500]),
])
def test_item_order_for_kv_beyond_l2(B, H, n_kv, Tq, d, Tk, lens):
    """A chunk of Tq rows at the end of caches whose K/V (201 MB) exceed L2: the prefill then
    numbers its items in blocks of four query tiles grouped by kv head.  Tq = 640 is one full
    block and a last block of one tile (d = 128); Tq = 384 a single block of three (d = 256,
    whose item decode divides by multiply-shifts; and d = 128 over three sequences of different
    lengths).  Every query tile of every head is checked on sampled rows, so an item the order
    skipped or repeated shows."""
    seed = 1101
    lens = np.array(lens, dtype=np.int32)              # absolute positions Tk_b - Tq + t
    qb = randn_bhtd(seed, "q", (B, H, Tq, d))
    kb = randn_bhtd(seed, "k", (B, n_kv, Tk, d), lengths=lens)
    vb = randn_bhtd(seed, "v", (B, n_kv, Tk, d), lengths=lens)
    out = ga.ga_attend(upload(qb), upload(kb), upload(vb), k_lens=torch.from_numpy(lens).cuda())
    assert ga.ga_read_device_status() == ga.GA_OK
    rows = sample_rows(Tq, 48, seed=seed, q_block=128)
    check_rows(out, qb, kb, vb, rows, [(b, h) for b in range(B) for h in range(H)], lens=lens,
               what=f"order d={d}")


def test_window_sink_and_full_causal_32k_d256():
    c = get_config(4)
    shape_q = (c.batch, c.n_heads, c.Tq, c.d)
    shape_k = (c.batch, c.n_kv, c.Tk, c.d)
    qb, kb, vb = (randn_bhtd(c.seed, t, s) for t, s in (("q", shape_q), ("k", shape_k), ("v", shape_k)))
    sink = np.random.Generator(np.random.PCG64(c.seed)).standard_normal(c.n_heads).astype(np.float32)
    q, k, v = upload(qb), upload(kb), upload(vb)
    rows = sample_rows(c.Tq, 256, seed=c.seed, window=c.window)
    heads = [(0, h) for h in (0, 7, 15)]
    out = ga.ga_attend(q, k, v, window=c.window, sink=torch.from_numpy(sink).cuda())
    assert ga.ga_read_device_status() == ga.GA_OK
    check_rows(out, qb, kb, vb, rows, heads, window=c.window, sink=sink, what="window+sink")
    out = ga.ga_attend(q, k, v, sink=torch.from_numpy(sink).cuda())
    check_rows(out, qb, kb, vb, rows, heads, sink=sink, what="full causal+sink")


def test_diff_attention_full_size_sampled():
    """Differential attention at the size the bench times it (B2 H32 Hkv8 d128 T8192 causal,
    lambda 0.8, the bench's inputs): 256 sampled rows of four (sequence, head) pairs against
    the float64 oracle ("Attention Variants", differential attention)."""
    c = get_config(2)
    B, H, n_kv, d, T = c.batch, c.n_heads, c.n_kv, c.d, c.Tq
    shp_q, shp_k = (B, H, T, d), (B, n_kv, T, d)
    bits = {t: randn_bhtd(c.seed, "diff_" + t, shp_q if t[0] == "q" else shp_k)
            for t in ("q1", "q2", "k1", "k2", "v")}
    dev = {t: upload(x) for t, x in bits.items()}
    out = ga.ga_attend_diff(dev["q1"], dev["k1"], dev["q2"], dev["k2"], dev["v"], 0.8)
    assert ga.ga_read_device_status() == ga.GA_OK
    rows = sample_rows(T, 256, seed=c.seed)
    o = out[:, :, rows].float().cpu().numpy().astype(np.float64)
    for b, h in ((0, 0), (0, 13), (1, 6), (1, 31)):
        kvh = h // c.g
        ref = oracle.diff_attend(f64(bits["q1"][b:b + 1, h:h + 1]), f64(bits["k1"][b:b + 1, kvh:kvh + 1]),
                                 f64(bits["q2"][b:b + 1, h:h + 1]), f64(bits["k2"][b:b + 1, kvh:kvh + 1]),
                                 f64(bits["v"][b:b + 1, kvh:kvh + 1]), 0.8, rows=rows)
        assert_close(o[b, h][None, None], ref, "bf16", f"diff attention b={b} h={h}")


@pytest.fixture(scope="module")
def sparse_128k():
    """The 128K block-sparse workload (planted outliers), on the device, with the oracle's block
    statistics of every block."""
    c = get_config(5)
    B, H, n_kv, d, T = c.batch, c.n_heads, c.n_kv, c.d, c.Tq
    qb = randn_bhtd(c.seed, "q", (B, H, T, d))
    kb = randn_bhtd(c.seed, "k", (B, n_kv, T, d))
    planted = planted_outliers(c.seed, n_kv, T, d, c.k_block, c.planted_fraction)
    for kvh, blk, tok, vec in planted:
        kb[0, kvh, tok] = f32_to_bf16_bits(vec)
    vb = randn_bhtd(c.seed, "v", (B, n_kv, T, d))
    q, k, v = upload(qb), upload(kb), upload(vb)
    cen, rad = ga.ga_block_stats(k, c.k_block)
    cr, rr = oracle.block_stats(f64(kb), None, c.k_block)
    return dict(c=c, qb=qb, kb=kb, vb=vb, q=q, k=k, v=v, cen=cen, rad=rad, cr=cr, rr=rr, planted=planted)


def _near(*margins):
    """Blocks whose oracle score lies within 1e-6 of one of its thresholds."""
    out = None
    for m in margins:
        x = np.abs(np.nan_to_num(m, nan=np.inf)) < 1e-6
        out = x if out is None else out | x
    return out


def test_block_sparse_prefill_128k(sparse_128k):
    s = sparse_128k
    c = s["c"]
    T, qbk, kbk = c.Tq, c.q_block, c.k_block
    cen, rad, cr, rr, planted = s["cen"], s["rad"], s["cr"], s["rr"], s["planted"]
    mask, nsel = ga.ga_select_blocks(s["q"], cen, rad, Tk=T, q_block=qbk, k_block=kbk, tau_mean=0.03,
                                     lambda_radius=c.extra["lambda_radius"])
    out = ga.ga_attend(s["q"], s["k"], s["v"], block_mask=mask, q_block=qbk, k_block=kbk)
    assert ga.ga_read_device_status() == ga.GA_OK
    # block statistics, every block
    assert np.max(np.abs(cen.cpu().numpy() - cr)) <= 1e-5
    assert np.max(np.abs(rad.cpu().numpy() - rr) / np.maximum(rr, 1.0)) <= 1e-5
    # selection, every block, four query heads
    gm = mask.cpu().numpy()
    for h in (0, 3, 12, 31):
        kvh = h // c.g
        qh = f64(s["qb"][:, h:h + 1])
        mref, nref, mm, zm = oracle.select_blocks(qh, cr[:, kvh:kvh + 1], rr[:, kvh:kvh + 1], Tk=T,
                                                  q_block=qbk, k_block=kbk, tau_mean=0.03,
                                                  lambda_radius=c.extra["lambda_radius"],
                                                  return_margins=True)
        diff = gm[:, h:h + 1] != mref
        assert not (diff & ~_near(mm, zm)).any(), f"head {h}: {(diff & ~_near(mm, zm)).sum()} decisions differ"
        # every planted block of this kv head is rescued for the last query block
        blocks = [blk for kh, blk, _, _ in planted if kh == kvh]
        assert gm[0, h, -1, blocks].all()
    # sparse attention on sampled rows, with the GPU's own mask
    rows = sample_rows(T, 128, seed=c.seed, extra=[tok + 1 for _, _, tok, _ in planted[:20]])
    check_rows(out, s["qb"], s["kb"], s["vb"], rows, [(0, 0), (0, 21)], mask=gm, what="sparse 128K")


@pytest.mark.parametrize("variant", ["mad", "bound", "group_shared"])
def test_selection_variants_128k(sparse_128k, variant):
    """The selection variants at the size the bench times them (the 128K workload, tau_mean 0.02,
    lambda 3): the robust MAD radius rule, the Cauchy-Schwarz bound branch as the rescue (no
    radius branch, tau_bound -3), and group-shared selection; every decision of the heads of two
    kv groups against the float64 oracle, mismatches allowed only within 1e-6 of a threshold
    ("RBS-Attention review": the two sieves, radius against its own distribution)."""
    s = sparse_128k
    c = s["c"]
    T, qbk, kbk, g = c.Tq, c.q_block, c.k_block, c.g
    lam = c.extra["lambda_radius"]
    kw = {"mad": dict(radius_rule="mad", lambda_radius=lam),
          "bound": dict(tau_bound=-3.0, lambda_radius=math.inf),
          "group_shared": dict(group_shared=True, lambda_radius=lam)}[variant]
    tau = 0.01 if variant == "group_shared" else 0.02
    mask, _ = ga.ga_select_blocks(s["q"], s["cen"], s["rad"], Tk=T, q_block=qbk, k_block=kbk, tau_mean=tau, **kw)
    assert ga.ga_read_device_status() == ga.GA_OK
    gm = mask.cpu().numpy()
    kvhs = (0, 5)
    heads = [h for kvh in kvhs for h in range(kvh * g, (kvh + 1) * g)] if variant == "group_shared" else [1, 22]
    okw = {"radius_rule": kw.get("radius_rule", "z"), "tau_bound": kw.get("tau_bound"),
           "group_shared": kw.get("group_shared", False), "lambda_radius": kw["lambda_radius"]}
    for kvh in sorted({h // g for h in heads}):
        hs = [h for h in heads if h // g == kvh]
        h0 = kvh * g
        # the oracle gets the whole group's rows when the group is pooled, else one head's
        qh = f64(s["qb"][:, h0:h0 + g]) if okw["group_shared"] else None
        for h in hs:
            q_in = qh if okw["group_shared"] else f64(s["qb"][:, h:h + 1])
            res = oracle.select_blocks(q_in, s["cr"][:, kvh:kvh + 1], s["rr"][:, kvh:kvh + 1], Tk=T, q_block=qbk,
                                       k_block=kbk, tau_mean=tau, return_margins=True, **okw)
            mref = res[0][:, (h - h0):(h - h0) + 1] if okw["group_shared"] else res[0]
            margins = [m[:, (h - h0):(h - h0) + 1] if okw["group_shared"] else m for m in res[2:]]
            diff = gm[:, h:h + 1] != mref
            bad = diff & ~_near(*margins)
            assert not bad.any(), f"{variant} head {h}: {int(bad.sum())} decisions differ outside the band"
            if okw["group_shared"]:
                break                          # every head of the group holds the same mask
        if okw["group_shared"]:
            assert all(np.array_equal(gm[:, h], gm[:, h0]) for h in range(h0, h0 + g))
