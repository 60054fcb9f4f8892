"""GPU parity of the ring-buffer decode ("Attention in Code", section 2): ga_ring_append writes
token n into slot n mod W and ga_attend_ring attends over the filled slots.  Checked against
the float64 oracle token by token, the ring contents byte for byte, and the property the
page states: once token 0 has left the window its value has exactly no influence."""
import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from tests.helpers import assert_close, host_tensor, to_f64
from workloads import bf16_bits_to_f32, randn_bhtd

pytestmark = pytest.mark.gpu


def _stream(B, H, n_kv, T, d, seed):
    q, qr = host_tensor(seed, "q", (B, H, T, d), "bf16")
    k, kr = host_tensor(seed, "k", (B, n_kv, T, d), "bf16")
    v, vr = host_tensor(seed, "v", (B, n_kv, T, d), "bf16")
    return q, qr, k, kr, v, vr


def _run_stream(q, k, v, W, sink=None, n0=None):
    """Feed every token through append + attend; returns ([B, H, T, d] outputs, rings, n_seen)."""
    B, H, T, d = q.shape
    n_kv = k.shape[1]
    k_ring = torch.zeros(B, n_kv, W, d, dtype=torch.bfloat16, device="cuda")
    v_ring = torch.zeros_like(k_ring)
    n_seen = torch.zeros(B, dtype=torch.int32, device="cuda") if n0 is None else n0.clone()
    outs = torch.empty(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        ga.ga_ring_append(k_ring, v_ring, k[:, :, t].contiguous(), v[:, :, t].contiguous(), n_seen)
        o = ga.ga_attend_ring(q[:, :, t:t + 1].contiguous(), k_ring, v_ring, n_seen, sink=sink)
        outs[:, :, t] = o[:, :, 0]
    assert ga.ga_read_device_status() == ga.GA_OK
    return outs, k_ring, v_ring, n_seen


@pytest.mark.parametrize("d,W,T,H,n_kv,use_sink", [
    (128, 8, 50, 8, 2, False),      # the page's W = 8, 50 tokens; GQA
    (256, 8, 50, 4, 2, True),       # the window workload's head dim, with a sink
    (64, 33, 70, 16, 1, False),     # MQA, a window that is not a power of two
])
def test_ring_stream_matches_oracle(d, W, T, H, n_kv, use_sink):
    B = 2
    q, qr, k, kr, v, vr = _stream(B, H, n_kv, T, d, seed=91 + d)
    sink = skr = None
    if use_sink:
        skr = np.random.default_rng(5).standard_normal(H).astype(np.float32)
        sink = torch.from_numpy(skr).cuda()
    outs, k_ring, v_ring, n_seen = _run_stream(q, k, v, W, sink)
    assert n_seen.cpu().tolist() == [T] * B
    for b in range(B):
        ref = oracle.ring_decode(qr[b], kr[b], vr[b], W, sink=skr)
        assert_close(to_f64(outs[b]), ref, "bf16", f"ring d={d} W={W} b={b}")
        bits = lambda t: t.view(torch.int16).cpu().numpy()
        rk, rv = oracle.ring_contents(bits(k[b]), bits(v[b]), W)
        assert np.array_equal(bits(k_ring[b]), rk), "ring keys differ"
        assert np.array_equal(bits(v_ring[b]), rv), "ring values differ"


def test_ring_token_zero_has_no_influence_after_the_window():
    """Changing token 0's value leaves every output from step W on bit-identical."""
    B, H, n_kv, T, d, W = 1, 8, 2, 40, 128, 8
    q, _, k, _, v, _ = _stream(B, H, n_kv, T, d, seed=77)
    out1, *_ = _run_stream(q, k, v, W)
    v2 = v.clone()
    v2[:, :, 0] += 100.0
    out2, *_ = _run_stream(q, k, v2, W)
    assert torch.equal(out1[:, :, W:], out2[:, :, W:])
    assert (out1[:, :, :W].float() - out2[:, :, :W].float()).abs().max().item() > 1.0


def test_ring_ragged_counters():
    """Sequences at different points of their streams in one batch: sequence 1 has already
    seen 5 tokens and sequence 2 has seen 13 (more than W) when the common stream starts."""
    H, n_kv, d, W, T = 4, 2, 128, 8, 12
    pre = [0, 5, 13]
    B = len(pre)
    q, qr, k, kr, v, vr = _stream(B, H, n_kv, max(pre) + T, d, seed=83)
    k_ring = torch.zeros(B, n_kv, W, d, dtype=torch.bfloat16, device="cuda")
    v_ring = torch.zeros_like(k_ring)
    n_seen = torch.zeros(B, dtype=torch.int32, device="cuda")
    for b, p in enumerate(pre):                       # each sequence's own earlier tokens
        for t in range(p):
            ga.ga_ring_append(k_ring[b:b + 1], v_ring[b:b + 1], k[b:b + 1, :, t].contiguous(),
                              v[b:b + 1, :, t].contiguous(), n_seen[b:b + 1])
    assert n_seen.cpu().tolist() == pre
    for s in range(T):                                # then one token per sequence and step
        kt = torch.stack([k[b, :, pre[b] + s] for b in range(B)]).contiguous()
        vt = torch.stack([v[b, :, pre[b] + s] for b in range(B)]).contiguous()
        qt = torch.stack([q[b, :, pre[b] + s:pre[b] + s + 1] for b in range(B)]).contiguous()
        ga.ga_ring_append(k_ring, v_ring, kt, vt, n_seen)
        o = ga.ga_attend_ring(qt, k_ring, v_ring, n_seen)
        for b in range(B):
            t = pre[b] + s
            ref = oracle.ring_decode(qr[b, :, :t + 1], kr[b, :, :t + 1], vr[b, :, :t + 1], W)[:, t]
            assert_close(to_f64(o[b, :, 0]), ref, "bf16", f"ragged b={b} t={t}")
    assert ga.ga_read_device_status() == ga.GA_OK


def test_ring_decode_full_size_sampled():
    """The bench's ring workload (B64 H16 Hkv8 d256 W1024, counters around and past W): the
    ring is any set of W keys in any order, so random ring contents stand in for a stream;
    sampled (sequence, head) pairs are checked against attention over the filled slots."""
    B, H, n_kv, d, W = 64, 16, 8, 256, 1024
    q, qr = host_tensor(97, "q", (B, H, 1, d), "bf16")
    kb = randn_bhtd(97, "k", (B, n_kv, W, d), "bf16")      # bf16 bits; float64 only where sampled
    vb = randn_bhtd(97, "v", (B, n_kv, W, d), "bf16")
    k_ring = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda()
    v_ring = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).cuda()
    f64 = lambda x: bf16_bits_to_f32(x).astype(np.float64)
    n = np.random.default_rng(97).integers(W // 2, 4 * W + 1, size=B).astype(np.int32)
    n[0], n[1] = 1, W                                 # a single token; exactly full
    n_seen = torch.from_numpy(n).cuda()
    skr = np.random.default_rng(98).standard_normal(H).astype(np.float32)
    lse = torch.empty(B, H, 1, device="cuda")
    out = ga.ga_attend_ring(q, k_ring, v_ring, n_seen, sink=torch.from_numpy(skr).cuda(), lse=lse)
    assert ga.ga_read_device_status() == ga.GA_OK
    rng = np.random.default_rng(99)
    for b in [0, 1] + list(rng.choice(np.arange(2, B), size=6, replace=False)):
        filled = min(int(n[b]), W)
        ref, ref_lse = oracle.attend(qr[b:b + 1], f64(kb[b:b + 1, :, :filled]), f64(vb[b:b + 1, :, :filled]),
                                     causal=False, sink=skr)
        assert_close(to_f64(out[b:b + 1]), ref, "bf16", f"full-size b={b} n={n[b]}")
        assert np.max(np.abs(to_f64(lse[b:b + 1]) - ref_lse)) <= 2e-3
