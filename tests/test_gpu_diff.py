"""GPU parity of differential attention ("Attention Variants": (A1 - lambda A2) V) against the
float64 oracle, and its two reductions: lambda = 0 is plain attention (bit for bit: the second
pass adds exactly -0 * x), and equal query/key pairs give (1 - lambda) times attention."""
import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from tests.helpers import assert_close, host_tensor, to_f64

pytestmark = pytest.mark.gpu


def _inputs(B, H, n_kv, Tq, Tk, d, seed):
    q1, q1r = host_tensor(seed, "q1", (B, H, Tq, d), "bf16")
    q2, q2r = host_tensor(seed, "q2", (B, H, Tq, d), "bf16")
    k1, k1r = host_tensor(seed, "k1", (B, n_kv, Tk, d), "bf16")
    k2, k2r = host_tensor(seed, "k2", (B, n_kv, Tk, d), "bf16")
    v, vr = host_tensor(seed, "v", (B, n_kv, Tk, d), "bf16")
    return (q1, k1, q2, k2, v), (q1r, k1r, q2r, k2r, vr)


@pytest.mark.parametrize("B,H,n_kv,Tq,Tk,d,lam,lens,W", [
    (2, 8, 2, 300, 300, 128, 0.8, None, 0),        # causal, ragged tail, GQA
    (1, 4, 4, 256, 256, 256, 0.5, None, 0),        # d = 256
    (2, 4, 2, 130, 640, 128, 0.6, [600, 640], 0),  # chunk at an offset, per-sequence lengths
    (1, 4, 1, 400, 400, 128, 0.7, None, 100),      # window
])
def test_diff_attention_matches_oracle(B, H, n_kv, Tq, Tk, d, lam, lens, W):
    dev, ref = _inputs(B, H, n_kv, Tq, Tk, d, seed=301 + d)
    k_lens = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = ga.ga_attend_diff(*dev, lam, k_lens=k_lens, window=W)
    assert ga.ga_read_device_status() == ga.GA_OK
    expect = oracle.diff_attend(*ref, lam, k_lens=lens, window=W)
    assert_close(to_f64(out), expect, "bf16", f"diff d={d} lam={lam}")


def test_diff_reductions():
    dev, _ = _inputs(1, 8, 2, 384, 384, 128, seed=311)
    q1, k1, q2, k2, v = dev
    plain = ga.ga_attend(q1, k1, v)
    assert torch.equal(ga.ga_attend_diff(q1, k1, q2, k2, v, 0.0), plain)
    same = ga.ga_attend_diff(q1, k1, q1, k1, v, 0.75)
    assert (same.float() - 0.25 * plain.float()).abs().max().item() <= 4e-3
    assert ga.ga_read_device_status() == ga.GA_OK
