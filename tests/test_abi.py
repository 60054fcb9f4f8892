"""The C-ABI library without a GPU: it loads, exports every entry point include/ga.h
declares, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import math
import os
import re

import pytest

import sparse_prefill_gqa_b300 as ga
from sparse_prefill_gqa_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return ga.lib()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ga_[a-z_0-9]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"ga_attend", "ga_block_stats", "ga_select_blocks", "ga_workspace_size"} <= names
    for n in sorted(names):
        assert hasattr(L, n), n


def test_debug_build_exports_the_same_symbols_and_only_it_reports_checks(L):
    """libga_debug.so (GA_DEBUG: in-kernel bounds checks) is the same ABI; the ordinary build
    answers ga_debug_violation with GA_ERR_UNSUPPORTED before any CUDA call."""
    dbg = ctypes.CDLL(build.build(debug=True))
    for n in sorted(_declared()):
        assert hasattr(dbg, n), n
    v = ctypes.c_uint64(7)
    assert L.ga_debug_violation(ctypes.byref(v), None) == ga.GA_ERR_UNSUPPORTED


def test_status_strings_and_version(L):
    assert ga.ga_status_string(0) == "GA_OK"
    for s in (-1, -2, -3, -4, -5):
        assert ga.ga_status_string(s).startswith("GA_ERR")
    assert ga.ga_version() >= 100


def _attend(L, **kw):
    p = ctypes.c_void_p(4096)        # aligned, never dereferenced: validation fails first
    a = dict(q=p, k=p, v=p, out=p, batch=1, n_heads=8, n_kv=2, d=128, Tq=16, Tk=32, k_lens=None,
             causal=1, window=0, sink=None, mask=None, qb=128, kb=64, lse=None, dtype=1, ws=None,
             wsb=0, stream=None)
    a.update(kw)
    return L.ga_attend(a["q"], a["k"], a["v"], a["out"], a["batch"], a["n_heads"], a["n_kv"], a["d"],
                       a["Tq"], a["Tk"], a["k_lens"], a["causal"], a["window"], a["sink"], a["mask"],
                       a["qb"], a["kb"], a["lse"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(out=None), dict(n_heads=6, n_kv=4), dict(n_kv=0), dict(n_kv=16),
    dict(d=0), dict(d=257), dict(Tq=0), dict(Tq=33, Tk=32), dict(causal=2), dict(window=-1),
    dict(causal=0, window=4), dict(mask=ctypes.c_void_p(4096), qb=0), dict(dtype=7),
    dict(q=ctypes.c_void_p(4100)), dict(sink=ctypes.c_void_p(4104)), dict(batch=0),
])
def test_attend_rejects_invalid_arguments(L, kw):
    assert _attend(L, **kw) == ga.GA_ERR_INVALID_ARG


def test_decode_workspace_is_checked_before_launch(L):
    # GQA decode (g * Tq <= 16, bf16, d = 128) over a long cache needs split-K workspace.
    need = ga.ga_workspace_size(64, 32, 8, 128, 1, 32768, __import__("torch").bfloat16)
    assert need > 0
    assert _attend(L, batch=64, n_heads=32, n_kv=8, Tq=1, Tk=32768) == ga.GA_ERR_WORKSPACE
    assert L.ga_workspace_size(1, 8, 2, 128, 512, 4096, 1) == 0          # prefill needs none
    assert L.ga_workspace_size(1, 8, 3, 128, 1, 4096, 1) == 2 ** 64 - 1  # invalid sizes


def test_block_calls_reject_invalid_arguments(L):
    p = ctypes.c_void_p(4096)
    assert L.ga_block_stats(None, None, 1, 1, 128, 64, 64, p, p, 1, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_block_stats(p, None, 1, 1, 128, 64, 0, p, p, 1, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_block_stats(p, None, 1, 1, 300, 64, 64, p, p, 1, None) == ga.GA_ERR_INVALID_ARG
    ws = L.ga_select_workspace_size(1, 8, 2, 128, 256, 256, 128, 64, 0)
    assert 0 < ws < 2 ** 64 - 1
    assert L.ga_select_workspace_size(1, 8, 3, 128, 256, 256, 128, 64, 0) == 2 ** 64 - 1
    args = [p, p, p, 1, 8, 2, 128, 256, 256, 4, 128, 64, 1, 0, math.inf, 3.0, p, None, 1, p, ws, None]
    bad = list(args)
    bad[19] = None                              # no workspace
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_WORKSPACE
    bad = list(args)
    bad[20] = ws - 1                            # workspace too small
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_WORKSPACE
    bad = list(args)
    bad[5] = 3                                  # n_heads % n_kv != 0
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_INVALID_ARG
    bad = list(args)
    bad[9] = 3                                  # nKb_out < ceil(Tk / k_block)
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_INVALID_ARG
    bad = list(args)
    bad[14] = math.nan                          # NaN threshold
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_INVALID_ARG
    bad = list(args)
    bad[16] = None                              # no output
    assert L.ga_select_blocks(*bad) == ga.GA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,n_kv,d,Tq,Tk,qb,kb,gs", [
    (1, 8, 2, 128, 256, 256, 128, 64, 0),
    (2, 32, 8, 128, 131072, 131072, 128, 64, 0),
    (1, 4, 1, 40, 1000, 3000, 64, 16, 1),
    (3, 6, 3, 256, 77, 5000, 200, 128, 0),
])
def test_select_workspace_size_matches_the_stated_formula(L, B, H, n_kv, d, Tq, Tk, qb, kb, gs):
    """The header states the selection workspace as seven 256-byte-rounded parts; the library's
    figure is exactly that."""
    up = lambda x: (x + 255) // 256 * 256
    nQb, nKb = -(-Tq // qb), -(-Tk // kb)
    P = n_kv if gs else H
    D = -(-d // 32) * 32
    S = -(-nKb // 128) * 128
    want = (2 * up(B * P * nQb * D * 4) + 2 * up(B * n_kv * nKb * D * 4) + 2 * up(B * P * nQb * 4)
            + up(B * n_kv * nKb) + up(B * P * nQb * S * 4))
    assert L.ga_select_workspace_size(B, H, n_kv, d, Tq, Tk, qb, kb, gs) == want


@pytest.mark.parametrize("B,H,L_max", [(1, 1, 1), (64, 16, 8192), (3, 16, 700), (200, 4, 200), (1000, 7, 65536)])
def test_mla_workspace_size_matches_the_stated_formula(L, B, H, L_max):
    """The header states the MLA workspace as four 256-byte-rounded parts over n_ids = 384 +
    batch - 1 partial slots; the library's figure is exactly that."""
    up = lambda x: (x + 255) // 256 * 256
    n_ids = 384 + B - 1
    want = up(B * H * 576 * 2) + up(n_ids * H * 512 * 4) + up(n_ids * H * 2 * 4) + up(B * 8)
    assert L.ga_mla_decode_workspace_size(B, H, L_max) == want


def test_ring_calls_reject_invalid_arguments(L):
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4098)                 # not 4-byte aligned
    # ga_ring_append(k_ring, v_ring, k_new, v_new, n_seen, batch, n_kv, d, W, stream)
    assert L.ga_ring_append(p, p, p, p, p, 1, 2, 128, 0, None) == ga.GA_ERR_INVALID_ARG      # W = 0
    assert L.ga_ring_append(p, p, p, p, p, 1, 2, 100, 8, None) == ga.GA_ERR_INVALID_ARG      # d % 8
    assert L.ga_ring_append(p, p, p, p, None, 1, 2, 128, 8, None) == ga.GA_ERR_INVALID_ARG   # no counter
    assert L.ga_ring_append(p, p, p, p, odd, 1, 2, 128, 8, None) == ga.GA_ERR_INVALID_ARG    # misaligned
    # ga_attend_ring(q, k_ring, v_ring, out, batch, n_heads, n_kv, d, W, n_seen, sink, lse, ws, bytes, stream)
    assert L.ga_attend_ring(p, p, p, p, 1, 8, 2, 128, 0, p, None, None, None, 0, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_attend_ring(p, p, p, p, 1, 8, 3, 128, 8, p, None, None, None, 0, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_attend_ring(p, p, p, p, 1, 8, 2, 96, 8, p, None, None, None, 0, None) == ga.GA_ERR_UNSUPPORTED
    assert L.ga_attend_ring(p, p, p, p, 1, 64, 2, 128, 8, p, None, None, None, 0, None) == ga.GA_ERR_UNSUPPORTED
    assert L.ga_attend_ring(p, p, p, p, 1, 8, 2, 128, 8, None, None, None, None, 0, None) == ga.GA_ERR_INVALID_ARG


def test_select_ex_rejects_invalid_rule_and_nan_bound(L):
    p = ctypes.c_void_p(4096)
    ws = L.ga_select_workspace_size(1, 8, 2, 128, 256, 256, 128, 64, 0)
    args = [p, p, p, 1, 8, 2, 128, 256, 256, 4, 128, 64, 1, 0, math.inf, 3.0, 0, -math.inf, 0, p, None, 1, p, ws,
            None]
    bad = list(args)
    bad[16] = 2                                 # unknown radius rule
    assert L.ga_select_blocks_ex(*bad) == ga.GA_ERR_INVALID_ARG
    bad = list(args)
    bad[17] = math.nan                          # NaN bound threshold
    assert L.ga_select_blocks_ex(*bad) == ga.GA_ERR_INVALID_ARG
    bad = list(args)
    bad[18] = 2                                 # group_shared is 0 or 1
    assert L.ga_select_blocks_ex(*bad) == ga.GA_ERR_INVALID_ARG


def test_mla_rejects_invalid_arguments(L):
    p = ctypes.c_void_p(4096)
    # ga_mla_decode(q_nope, q_rope, latent, w_uk, w_uv, lens, out, batch, n_heads, L_max, ws, bytes, stream)
    assert L.ga_mla_decode(p, p, p, p, p, None, p, 1, 32, 64, p, 1 << 20, None) == ga.GA_ERR_UNSUPPORTED
    assert L.ga_mla_decode(p, p, p, p, p, None, p, 0, 16, 64, p, 1 << 20, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_mla_decode(p, p, p, p, p, None, p, 1, 16, 64, p, 16, None) == ga.GA_ERR_WORKSPACE
    assert L.ga_mla_decode_workspace_size(1, 17, 64) == 2 ** 64 - 1


def test_diff_rejects_invalid_arguments(L):
    p = ctypes.c_void_p(4096)

    def diff(**kw):
        a = dict(q1=p, k1=p, q2=p, k2=p, v=p, out=p, batch=1, n_heads=8, n_kv=2, d=128, Tq=16, Tk=32,
                 causal=1, window=0, lam=0.5, ws=p, wsb=1 << 20)
        a.update(kw)
        return L.ga_attend_diff(a["q1"], a["k1"], a["q2"], a["k2"], a["v"], a["out"], a["batch"], a["n_heads"],
                                a["n_kv"], a["d"], a["Tq"], a["Tk"], None, a["causal"], a["window"], a["lam"],
                                a["ws"], a["wsb"], None)
    assert diff(q2=None) == ga.GA_ERR_INVALID_ARG
    assert diff(lam=float("nan")) == ga.GA_ERR_INVALID_ARG
    assert diff(lam=float("inf")) == ga.GA_ERR_INVALID_ARG
    assert diff(Tq=33) == ga.GA_ERR_INVALID_ARG                      # Tk_max < Tq
    assert diff(causal=0, window=4) == ga.GA_ERR_INVALID_ARG
    assert diff(k2=ctypes.c_void_p(4104)) == ga.GA_ERR_INVALID_ARG   # not 16-byte aligned
    assert diff(d=64) == ga.GA_ERR_UNSUPPORTED                       # tensor-core head dims only
    assert diff(ws=None) == ga.GA_ERR_WORKSPACE
    assert diff(wsb=1 * 8 * 16 * 128 * 4 - 1) == ga.GA_ERR_WORKSPACE  # A1 v in fp32 needs B*H*Tq*d*4
    assert diff(ws=ctypes.c_void_p(4104)) == ga.GA_ERR_WORKSPACE


def test_topk_sparse_decode_calls_reject_invalid_arguments(L):
    p = ctypes.c_void_p(4096)
    # ga_dsa_indexer(qi, wi, ki, lens, batch, n_idx_heads, di, L_max, scores, stream)
    assert L.ga_dsa_indexer(p, p, p, None, 1, 8, 96, 64, p, None) == ga.GA_ERR_UNSUPPORTED   # di
    assert L.ga_dsa_indexer(p, p, p, None, 1, 3, 128, 64, p, None) == ga.GA_ERR_UNSUPPORTED  # not 2^n
    assert L.ga_dsa_indexer(p, p, p, None, 1, 32, 128, 64, p, None) == ga.GA_ERR_UNSUPPORTED  # > di/8
    assert L.ga_dsa_indexer(p, p, p, None, 0, 8, 128, 64, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_dsa_indexer(p, p, p, None, 1, 8, 128, 0, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_dsa_indexer(p, p, p, None, 1, 8, 128, 64, None, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_dsa_indexer(ctypes.c_void_p(4104), p, p, None, 1, 8, 128, 64, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_dsa_indexer(p, ctypes.c_void_p(4098), p, None, 1, 8, 128, 64, p, None) == ga.GA_ERR_INVALID_ARG
    # ga_topk_indices(scores, lens, batch, L_max, topk, idx, n_sel, stream)
    assert L.ga_topk_indices(p, None, 1, 64, 0, p, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_topk_indices(p, None, 0, 64, 8, p, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_topk_indices(p, None, 1, 64, 8, None, p, None) == ga.GA_ERR_INVALID_ARG
    assert L.ga_topk_indices(ctypes.c_void_p(4098), None, 1, 64, 8, p, p, None) == ga.GA_ERR_INVALID_ARG

    def gather(**kw):
        a = dict(q=p, k=p, v=p, out=p, batch=1, n_heads=8, n_kv=2, d=128, Tk=32768, idx=p, n_sel=p,
                 topk=8192, sink=None, lse=None, ws=p, wsb=1 << 24)
        a.update(kw)
        return L.ga_attend_gather(a["q"], a["k"], a["v"], a["out"], a["batch"], a["n_heads"], a["n_kv"], a["d"],
                                  a["Tk"], a["idx"], a["n_sel"], a["topk"], a["sink"], a["lse"], a["ws"],
                                  a["wsb"], None)
    assert gather(d=96) == ga.GA_ERR_UNSUPPORTED
    assert gather(n_heads=64) == ga.GA_ERR_UNSUPPORTED                 # 32 query heads per kv head
    assert gather(batch=2, n_kv=8, n_heads=8, Tk=1 << 28) == ga.GA_ERR_UNSUPPORTED   # 2^32 cache rows
    assert gather(topk=0) == ga.GA_ERR_INVALID_ARG
    assert gather(idx=None) == ga.GA_ERR_INVALID_ARG
    assert gather(idx=ctypes.c_void_p(4098)) == ga.GA_ERR_INVALID_ARG
    assert gather(n_sel=ctypes.c_void_p(4100)) == ga.GA_ERR_INVALID_ARG
    assert gather(lse=ctypes.c_void_p(4100)) == ga.GA_ERR_INVALID_ARG
    assert gather(ws=None) == ga.GA_ERR_WORKSPACE                      # 16 key chunks: partials needed
    assert gather(wsb=16) == ga.GA_ERR_WORKSPACE
    # the gathered decode needs only the split-K partials over topk keys: one sequence with two
    # kv heads splits 8192 selected keys into 32 chunks of 256 (about four CTAs per SM over the
    # launch, at least 256 keys a chunk), one fp32 partial row of d plus (max, sum) per head
    need = L.ga_attend_gather_workspace_size(1, 8, 2, 128, 8192)
    assert need == 1 * 8 * 32 * (128 + 2) * 4
    assert L.ga_attend_gather_workspace_size(64, 32, 8, 128, 2048) == 64 * 32 * 2 * (128 + 2) * 4   # 2 x 1024
    assert L.ga_attend_gather_workspace_size(1, 6, 4, 128, 8192) == 2 ** 64 - 1
