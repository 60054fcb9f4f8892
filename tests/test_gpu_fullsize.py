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


def test_block_sparse_prefill_128k():
    c = get_config(5)
    B, H, n_kv, d, T, qbk, kbk = c.batch, c.n_heads, c.n_kv, c.d, c.Tq, c.q_block, c.k_block
    qb = randn_bhtd(c.seed, "q", (B, H, T, d))
    kb = randn_bhtd(c.seed, "k", (B, n_kv, T, d))
    planted = planted_outliers(c.seed, n_kv, T, d, kbk, c.planted_fraction)
    for kvh, blk, tok, vec in planted:
        kb[0, kvh, tok] = f32_to_bf16_bits(vec)
    vb = randn_bhtd(c.seed, "v", (B, n_kv, T, d))
    q, k, v = upload(qb), upload(kb), upload(vb)
    cen, rad = ga.ga_block_stats(k, kbk)
    mask, nsel = ga.ga_select_blocks(q, cen, rad, Tk=T, q_block=qbk, k_block=kbk, tau_mean=0.03,
                                     lambda_radius=c.extra["lambda_radius"])
    out = ga.ga_attend(q, k, v, block_mask=mask, q_block=qbk, k_block=kbk)
    assert ga.ga_read_device_status() == ga.GA_OK
    # block statistics, every block
    kr = f64(kb)
    cr, rr = oracle.block_stats(kr, None, kbk)
    assert np.max(np.abs(cen.cpu().numpy() - cr)) <= 1e-5
    assert np.max(np.abs(rad.cpu().numpy() - rr) / np.maximum(rr, 1.0)) <= 1e-5
    # selection, every block, two query heads per kv head
    gm = mask.cpu().numpy()
    qr = None
    for h in (0, 3, 12, 31):
        kvh = h // c.g
        qh = f64(qb[:, h:h + 1])
        mref, nref, mm, zm = oracle.select_blocks(qh, cr[:, kvh:kvh + 1], rr[:, kvh:kvh + 1], Tk=T,
                                                  q_block=qbk, k_block=kbk, tau_mean=0.03,
                                                  lambda_radius=c.extra["lambda_radius"],
                                                  return_margins=True)
        diff = gm[:, h:h + 1] != mref
        near = (np.abs(np.nan_to_num(mm, nan=np.inf)) < 1e-6) | (np.abs(np.nan_to_num(zm, nan=np.inf)) < 1e-6)
        assert not (diff & ~near).any(), f"head {h}: {(diff & ~near).sum()} decisions differ"
        # every planted block of this kv head is rescued for the last query block
        blocks = [blk for kh, blk, _, _ in planted if kh == kvh]
        assert gm[0, h, -1, blocks].all()
    # sparse attention on sampled rows, with the GPU's own mask
    rows = sample_rows(T, 128, seed=c.seed, extra=[tok + 1 for _, _, tok, _ in planted[:20]])
    check_rows(out, qb, kb, vb, rows, [(0, 0), (0, 21)], mask=gm, what="sparse 128K")
