"""GPU parity of MLA decode in the absorbed form ("Attention in Code", section 4) against the
float64 oracle: DeepSeek-V2-Lite's sizes (latent 512, rope 64, head dims 128), ragged cache
lengths split over the decode CTAs' shares (an empty one among them), poisoned cache rows past
each length, and the bench's full-size workload on sampled sequences."""
import numpy as np
import pytest
import torch

import sparse_prefill_gqa_b300 as ga
from oracle.mla import mla_absorbed
from tests.helpers import assert_close, host_tensor, to_f64

pytestmark = pytest.mark.gpu


def _weights(H, seed):
    # w ~ N(0, 1/128) keeps q_lat and the expanded output at unit scale
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((2, H, 512, 128)) / np.sqrt(128)).astype(np.float32)
    t = torch.from_numpy(w).to(torch.bfloat16)
    return t[0].cuda().contiguous(), t[1].cuda().contiguous(), t[0].double().numpy(), t[1].double().numpy()


def _inputs(B, H, L_max, seed):
    qn, qnr = host_tensor(seed, "qn", (B, 1, H, 128), "bf16")
    qp, qpr = host_tensor(seed, "qp", (B, 1, H, 64), "bf16")
    lat, latr = host_tensor(seed, "lat", (B, 1, L_max, 576), "bf16")
    return qn[:, 0].contiguous(), qnr[:, 0], qp[:, 0].contiguous(), qpr[:, 0], lat[:, 0].contiguous(), latr[:, 0]


def _oracle(qnr, qpr, latr, wuk, wuv, b, n):
    """The decode row of sequence b: its query at position n - 1 over tokens 0 .. n-1."""
    return mla_absorbed(qnr[b][:, None], qpr[b][:, None], latr[b, :n, :512], latr[b, :n, 512:], wuk, wuv)[:, 0]


_SHORT = [int(x) for x in np.random.default_rng(704).integers(0, 201, size=200)]


@pytest.mark.parametrize("B,H,L_max,lens,poison", [
    (3, 16, 700, [700, 333, 1], False),
    (2, 8, 3000, [3000, 1717], True),        # a sequence over many CTAs; rows past each length hold NaN
    # shares that end inside one sequence, hold short ones whole, and skip an empty one
    (8, 16, 8192, [8192, 32, 5, 0, 64, 8192, 1, 700], True),
    (200, 4, 200, _SHORT, True),             # several short sequences in each CTA's share
    (5, 1, 5000, [0, 4999, 1, 2500, 0], True),   # one head; empty sequences at both ends
    (4, 5, 2048, [33, 2048, 31, 1000], False),   # an odd head count (rows 5..15 of the MMA padded)
])
def test_mla_decode_matches_oracle(B, H, L_max, lens, poison):
    qn, qnr, qp, qpr, lat, latr = _inputs(B, H, L_max, seed=701 + H)
    w_uk, w_uv, wuk, wuv = _weights(H, 702)
    if poison:
        for b, n in enumerate(lens):
            lat[b, n:] = float("nan")
    out = ga.ga_mla_decode(qn, qp, lat, w_uk, w_uv, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert ga.ga_read_device_status() == ga.GA_OK
    got = to_f64(out)
    for b, n in enumerate(lens):
        if n == 0:                           # an empty cache gives a zero row
            assert np.all(got[b] == 0.0), f"mla b={b} empty"
            continue
        assert_close(got[b], _oracle(qnr, qpr, latr, wuk, wuv, b, n), "bf16", f"mla b={b} n={n}")


def test_mla_decode_full_size_sampled():
    """The bench's workload: B64 H16, cache lengths U[4096, 8192]."""
    from workloads import bf16_bits_to_f32, randn_bhtd, uniform_lengths
    B, H, L_max = 64, 16, 8192
    lens = uniform_lengths(711, B, 4096, 8192)
    qn, qnr = host_tensor(711, "qn", (B, 1, H, 128), "bf16")
    qp, qpr = host_tensor(711, "qp", (B, 1, H, 64), "bf16")
    qn, qnr, qp, qpr = qn[:, 0].contiguous(), qnr[:, 0], qp[:, 0].contiguous(), qpr[:, 0]
    latb = randn_bhtd(711, "lat", (B, 1, L_max, 576), "bf16")[:, 0]    # bits; float64 only where sampled
    lat = torch.from_numpy(np.ascontiguousarray(latb).view(np.int16)).view(torch.bfloat16).cuda()
    w_uk, w_uv, wuk, wuv = _weights(H, 712)
    out = to_f64(ga.ga_mla_decode(qn, qp, lat, w_uk, w_uv, torch.from_numpy(lens).cuda()))
    assert ga.ga_read_device_status() == ga.GA_OK
    for b in np.random.default_rng(713).choice(B, size=4, replace=False):
        n = int(lens[b])
        lr = bf16_bits_to_f32(latb[b, :n]).astype(np.float64)
        ref = mla_absorbed(qnr[b][:, None], qpr[b][:, None], lr[:, :512], lr[:, 512:], wuk, wuv)[:, 0]
        assert_close(out[b], ref, "bf16", f"mla full b={b}")
