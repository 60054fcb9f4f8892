"""Canary padding around every output: each entry point writes into a view in the middle of a
larger buffer whose margins hold a sentinel byte pattern, and afterwards every margin byte must
be unchanged -- a write past either end of an output (a wrong tile bound, a ragged tail, an index
off by one) shows up here even when the values inside are right.  Small ragged shapes, so that
partial tiles, tails and padding rows are all exercised."""
import numpy as np
import pytest
import torch

import sparse_prefill_gqa_b300 as ga
from tests.helpers import host_tensor

pytestmark = pytest.mark.gpu

PAD = 4096            # margin bytes on each side (a multiple of 256: the views stay aligned)
SENTINEL = 0xA5


class Canary:
    """Output buffers carved from sentinel-filled allocations, checked on demand."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((PAD + ((n + 255) // 256) * 256 + PAD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n))
        return raw[PAD:PAD + n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        for raw, n in self.bufs:
            head = raw[:PAD]
            tail = raw[PAD + n:]
            assert bool((head == SENTINEL).all()), f"{what}: write before the start of an output"
            assert bool((tail == SENTINEL).all()), f"{what}: write past the end of an output"


def _qkv(B, H, n_kv, Tq, Tk, d, seed, dtype="bf16"):
    q, _ = host_tensor(seed, "q", (B, H, Tq, d), dtype)
    k, _ = host_tensor(seed, "k", (B, n_kv, Tk, d), dtype)
    v, _ = host_tensor(seed, "v", (B, n_kv, Tk, d), dtype)
    return q, k, v


@pytest.mark.parametrize("B,H,n_kv,Tq,Tk,d,dtype,window,masked", [
    (2, 4, 2, 200, 333, 128, "bf16", 0, False),      # tensor-core prefill d=128, ragged tiles
    (1, 2, 1, 130, 300, 256, "bf16", 77, False),     # d=256, window
    (2, 4, 2, 257, 257, 128, "bf16", 0, True),       # block mask (unit lists)
    (3, 8, 2, 2, 5000, 128, "bf16", 0, False),       # split-K decode, several chunks + combine
    (2, 4, 4, 1, 700, 64, "bf16", 0, False),         # decode d=64, one chunk
    (2, 3, 1, 37, 90, 40, "f32", 0, False),          # CUDA-core fp32 path
])
def test_attend_writes_only_its_outputs(B, H, n_kv, Tq, Tk, d, dtype, window, masked):
    q, k, v = _qkv(B, H, n_kv, Tq, Tk, d, 801 + d, dtype)
    cn = Canary()
    out = cn.empty(q.shape, q.dtype)
    lse = cn.empty((B, H, Tq), torch.float32)
    lens = torch.tensor([Tk - 7 * b for b in range(B)], dtype=torch.int32, device="cuda")
    bm = None
    if masked:
        nQb, nKb = -(-Tq // 128), -(-Tk // 64)
        bm = (torch.rand(B, H, nQb, nKb, device="cuda") < 0.5).to(torch.uint8)
    need = ga.ga_workspace_size(B, H, n_kv, d, Tq, Tk, q.dtype)
    ws = cn.empty((max(need, 1),), torch.uint8) if need else None
    ga.ga_attend(q, k, v, out, k_lens=lens, window=window, block_mask=bm, lse=lse, workspace=ws)
    assert ga.ga_read_device_status() == ga.GA_OK
    cn.check("ga_attend")


def test_block_stats_and_selection_write_only_their_outputs():
    B, H, n_kv, T, d = 2, 4, 2, 1000, 128
    q, k, _ = _qkv(B, H, n_kv, T, T, d, 811)
    nKb, nQb = -(-T // 64), -(-T // 128)
    cn = Canary()
    cen = cn.empty((B, n_kv, nKb, d), torch.float32)
    rad = cn.empty((B, n_kv, nKb), torch.float32)
    ga.ga_block_stats(k, 64, centroid=cen, radius=rad, k_lens=torch.tensor([T, T - 100], dtype=torch.int32,
                                                                          device="cuda"))
    for kw in ({}, {"radius_rule": "mad"}, {"tau_bound": -1.0}, {"group_shared": True}):
        mask = cn.empty((B, H, nQb, nKb), torch.uint8)
        nsel = cn.empty((B, H, nQb), torch.int32)
        wsb = ga.lib().ga_select_workspace_size(B, H, n_kv, d, T, T, 128, 64, int(kw.get("group_shared", False)))
        ws = cn.empty((wsb,), torch.uint8)
        ga.ga_select_blocks(q, cen, rad, Tk=T, tau_mean=0.05, block_mask=mask, n_selected=nsel, workspace=ws, **kw)
    assert ga.ga_read_device_status() == ga.GA_OK
    cn.check("block stats / selection")


def test_variants_write_only_their_outputs():
    cn = Canary()
    # differential attention
    q1, k1, v = _qkv(1, 4, 2, 300, 300, 128, 821)
    q2, k2, _ = _qkv(1, 4, 2, 300, 300, 128, 822)
    out = cn.empty(q1.shape, torch.bfloat16)
    ws = cn.empty((1 * 4 * 300 * 128 * 4,), torch.uint8)
    ga.ga_attend_diff(q1, k1, q2, k2, v, 0.7, out, workspace=ws)
    # top-k sparse decode: indexer, top-k, gathered decode
    B, H, n_kv, Lm, d, Hi, di, topk = 3, 8, 2, 3000, 128, 8, 128, 700
    q, k, v = _qkv(B, H, n_kv, 1, Lm, d, 823)
    qi, _ = host_tensor(824, "qi", (B, 1, Hi, di), "bf16")
    ki, _ = host_tensor(824, "ki", (B, 1, Lm, di), "bf16")
    qi, ki = qi[:, 0].contiguous(), ki[:, 0].contiguous()
    wi = torch.rand(B, Hi, device="cuda")
    lens = torch.tensor([3000, 1234, 500], dtype=torch.int32, device="cuda")
    scores = cn.empty((B, Lm), torch.float32)
    ga.ga_dsa_indexer(qi, wi, ki, lens, scores)
    idx = cn.empty((B, topk), torch.int32)
    n_sel = cn.empty((B,), torch.int32)
    ga.ga_topk_indices(scores, topk, lens, idx, n_sel)
    out = cn.empty(q.shape, torch.bfloat16)
    lse = cn.empty((B, H, 1), torch.float32)
    need = int(ga.lib().ga_attend_gather_workspace_size(B, H, n_kv, d, topk))
    ws = cn.empty((max(need, 1),), torch.uint8)
    ga.ga_attend_gather(q, k, v, idx, n_sel, out, lse=lse, workspace=ws)
    # ring append and ring decode
    W = 64
    k_ring = cn.empty((2, n_kv, W, d), torch.bfloat16)
    v_ring = cn.empty((2, n_kv, W, d), torch.bfloat16)
    k_ring.zero_()
    v_ring.zero_()
    n_seen = torch.tensor([5, 70], dtype=torch.int32, device="cuda")
    kn, _ = host_tensor(825, "kn", (2, n_kv, 1, d), "bf16")
    vn, _ = host_tensor(825, "vn", (2, n_kv, 1, d), "bf16")
    ga.ga_ring_append(k_ring, v_ring, kn[:, :, 0].contiguous(), vn[:, :, 0].contiguous(), n_seen)
    qr, _ = host_tensor(826, "qr", (2, H, 1, d), "bf16")
    out = cn.empty(qr.shape, torch.bfloat16)
    ga.ga_attend_ring(qr, k_ring, v_ring, n_seen, out)
    # MLA decode
    B, Hm, L = 3, 16, 1500
    qn, _ = host_tensor(827, "qn", (B, 1, Hm, 128), "bf16")
    qp, _ = host_tensor(827, "qp", (B, 1, Hm, 64), "bf16")
    lat, _ = host_tensor(827, "lat", (B, 1, L, 576), "bf16")
    w, _ = host_tensor(827, "w", (2, Hm, 512, 128), "bf16")
    out = cn.empty((B, Hm, 128), torch.bfloat16)
    ws = cn.empty((int(ga.lib().ga_mla_decode_workspace_size(B, Hm, L)),), torch.uint8)
    ga.ga_mla_decode(qn[:, 0].contiguous(), qp[:, 0].contiguous(), lat[:, 0].contiguous(), w[0].contiguous(),
                     w[1].contiguous(), torch.tensor([1500, 700, 1], dtype=torch.int32, device="cuda"), out,
                     workspace=ws)
    assert ga.ga_read_device_status() == ga.GA_OK
    cn.check("variants")
