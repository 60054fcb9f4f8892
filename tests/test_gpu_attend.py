"""GPU parity of ga_attend against the float64 oracle, element by element, at sizes the
oracle finishes in seconds: several tiles, ragged tails, every mask feature, every kernel
path (tensor-core prefill d=128/256, split-K decode d=64/128, CUDA-core fp32 and bf16)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_prefill_gqa_b300 as ga
from tests.helpers import assert_close, host_tensor, to_f64
from workloads import uniform_lengths

pytestmark = pytest.mark.gpu


def run_case(B, H, n_kv, Tq, Tk, d, dtype, *, causal=True, window=0, sink=False, lens=None,
             mask_density=None, q_block=128, k_block=64, seed=0, want_lse=True, poison_tail=False):
    q, qr = host_tensor(seed, "q", (B, H, Tq, d), dtype)
    k, kr = host_tensor(seed, "k", (B, n_kv, Tk, d), dtype)
    v, vr = host_tensor(seed, "v", (B, n_kv, Tk, d), dtype)
    k_lens = None
    if lens is not None:
        k_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
        if poison_tail:   # cache slots past each sequence's length hold NaN
            for b, n in enumerate(lens):
                k[b, :, n:] = float("nan")
                v[b, :, n:] = float("nan")
    sk = None
    skr = None
    if sink:
        skr = np.random.default_rng(seed + 7).standard_normal(H).astype(np.float32)
        sk = torch.from_numpy(skr).cuda()
    bm = None
    bmr = None
    if mask_density is not None:
        nQb, nKb = -(-Tq // q_block), -(-Tk // k_block)
        bmr = (np.random.default_rng(seed + 9).random((B, H, nQb, nKb)) < mask_density).astype(np.uint8)
        bm = torch.from_numpy(bmr).cuda()
    lse = torch.empty(B, H, Tq, dtype=torch.float32, device="cuda") if want_lse else None
    out = ga.ga_attend(q, k, v, k_lens=k_lens, causal=causal, window=window, sink=sk, block_mask=bm,
                       q_block=q_block, k_block=k_block, lse=lse)
    assert ga.ga_read_device_status() == ga.GA_OK
    ref, ref_lse = oracle.attend(qr, kr, vr, k_lens=lens, causal=causal, window=window, sink=skr,
                                 block_mask=bmr, q_block=q_block, k_block=k_block)
    return to_f64(out), ref, (to_f64(lse) if want_lse else None), ref_lse


def check(case_out, dtype, what):
    out, ref, lse, ref_lse = case_out
    assert_close(out, ref, dtype, what)
    if lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse)), what + " lse finiteness"
        tol = 1e-5 if dtype == "f32" else 2e-3
        assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0) <= tol, what + " lse"


# ---------------------------------------------------------------------------- fp32 (CUDA cores)
def test_fp32_tiny_prefill_and_token_by_token_decode():
    """fp32 tiny GQA workload: B1 H8 Hkv2 d16 T40, prefill, then decode Tq=1, Tk=1..40 through
    a cache allocated at 40 with per-sequence lengths, and through sliced caches."""
    check(run_case(1, 8, 2, 40, 40, 16, "f32", seed=1001), "f32", "prefill")
    q, qr = host_tensor(1001, "q", (1, 8, 40, 16), "f32")
    k, kr = host_tensor(1001, "k", (1, 2, 40, 16), "f32")
    v, vr = host_tensor(1001, "v", (1, 2, 40, 16), "f32")
    full, _ = oracle.attend(qr, kr, vr)
    for t in range(40):
        lens = torch.tensor([t + 1], dtype=torch.int32, device="cuda")
        o = ga.ga_attend(q[:, :, t:t + 1].contiguous(), k, v, k_lens=lens)
        o2 = ga.ga_attend(q[:, :, t:t + 1].contiguous(), k[:, :, :t + 1].contiguous(),
                          v[:, :, :t + 1].contiguous())
        assert np.max(np.abs(to_f64(o)[:, :, 0] - full[:, :, t])) <= 1e-5
        assert np.max(np.abs(to_f64(o2)[:, :, 0] - full[:, :, t])) <= 1e-5


@pytest.mark.parametrize("kw", [
    dict(B=2, H=4, n_kv=4, Tq=37, Tk=70, d=33, window=9, sink=True, lens=[70, 51]),
    dict(B=1, H=6, n_kv=1, Tq=20, Tk=20, d=256, causal=False, sink=True),
    dict(B=1, H=4, n_kv=2, Tq=64, Tk=100, d=8, mask_density=0.5, q_block=16, k_block=8),
])
def test_fp32_general(kw):
    check(run_case(dtype="f32", seed=5, **kw), "f32", str(kw))


# ---------------------------------------------------------------------------- bf16 tensor cores
@pytest.mark.parametrize("kw", [
    dict(B=2, H=8, n_kv=2, Tq=421, Tk=421, d=128),                       # causal, ragged tail
    dict(B=1, H=4, n_kv=4, Tq=256, Tk=256, d=128, causal=False),         # MHA, no mask
    dict(B=1, H=8, n_kv=1, Tq=300, Tk=300, d=128, window=77, sink=True), # MQA, window + sink
    dict(B=2, H=4, n_kv=2, Tq=200, Tk=1024, d=128, lens=[1000, 777]),    # chunk at an offset
    dict(B=2, H=4, n_kv=2, Tq=130, Tk=1024, d=128, lens=[650, 1024], poison_tail=True),
    dict(B=1, H=4, n_kv=2, Tq=512, Tk=640, d=128, mask_density=0.4),     # block-sparse
    dict(B=1, H=2, n_kv=1, Tq=384, Tk=384, d=128, mask_density=0.3, k_block=128, q_block=256),
])
def test_bf16_tensor_core_prefill_d128(kw):
    check(run_case(dtype="bf16", seed=11, **kw), "bf16", str(kw))


@pytest.mark.parametrize("kw", [
    dict(B=1, H=4, n_kv=2, Tq=700, Tk=700, d=256, window=100, sink=True),
    dict(B=1, H=2, n_kv=2, Tq=333, Tk=333, d=256),
    dict(B=2, H=2, n_kv=1, Tq=129, Tk=600, d=256, lens=[600, 415], sink=True, poison_tail=True),
    dict(B=1, H=2, n_kv=1, Tq=256, Tk=512, d=256, mask_density=0.5),
])
def test_bf16_tensor_core_prefill_d256(kw):
    check(run_case(dtype="bf16", seed=13, **kw), "bf16", str(kw))


# ---------------------------------------------------------------------------- bf16 decode
@pytest.mark.parametrize("kw", [
    dict(B=4, H=8, n_kv=2, Tq=1, Tk=5000, d=128, lens=[5000, 4100, 1, 2999], poison_tail=True),
    dict(B=3, H=8, n_kv=8, Tq=1, Tk=777, d=128, lens=[777, 70, 500], sink=True),
    dict(B=2, H=16, n_kv=4, Tq=4, Tk=3000, d=64, lens=[3000, 1234], window=300),
    dict(B=1, H=4, n_kv=1, Tq=2, Tk=9000, d=128, sink=True),
])
def test_bf16_split_k_decode(kw):
    check(run_case(dtype="bf16", seed=17, **kw), "bf16", str(kw))


def test_bf16_decode_token_by_token_matches_prefill():
    """GQA decode of the last 24 tokens of a 300-token prompt, one at a time through the
    cache, equals the rows of one prefill over the whole prompt (both within tolerance of
    the oracle, and within bf16 rounding of each other)."""
    B, H, n_kv, T, d = 1, 8, 2, 300, 128
    q, qr = host_tensor(23, "q", (B, H, T, d), "bf16")
    k, kr = host_tensor(23, "k", (B, n_kv, T, d), "bf16")
    v, vr = host_tensor(23, "v", (B, n_kv, T, d), "bf16")
    full = to_f64(ga.ga_attend(q, k, v))
    ref, _ = oracle.attend(qr, kr, vr)
    assert_close(full, ref, "bf16", "prefill")
    for t in range(T - 24, T):
        lens = torch.tensor([t + 1], dtype=torch.int32, device="cuda")
        o = to_f64(ga.ga_attend(q[:, :, t:t + 1].contiguous(), k, v, k_lens=lens))
        assert_close(o[:, :, 0], ref[:, :, t], "bf16", f"decode t={t}")
        assert np.max(np.abs(o[:, :, 0] - full[:, :, t])) <= 2e-2


# ---------------------------------------------------------------------------- bf16 CUDA cores
@pytest.mark.parametrize("kw", [
    dict(B=1, H=4, n_kv=2, Tq=100, Tk=100, d=64),                       # prefill d=64
    dict(B=1, H=4, n_kv=2, Tq=50, Tk=90, d=16, window=7, sink=True),
    dict(B=1, H=2, n_kv=1, Tq=1, Tk=500, d=256, lens=[321]),            # decode d=256
    dict(B=1, H=2, n_kv=1, Tq=96, Tk=96, d=128, mask_density=0.5, q_block=32, k_block=16),
])
def test_bf16_cuda_core_paths(kw):
    check(run_case(dtype="bf16", seed=19, **kw), "bf16", str(kw))


# ---------------------------------------------------------------------------- properties
def test_empty_rows_give_zero_and_minus_inf_lse():
    """A block mask that leaves rows with no key: out = 0 and lse = -inf (no sink), lse =
    sink (with a sink), on the tensor-core path."""
    B, H, n_kv, T, d = 1, 2, 1, 256, 128
    q, _ = host_tensor(29, "q", (B, H, T, d), "bf16")
    k, _ = host_tensor(29, "k", (B, n_kv, T, d), "bf16")
    v, _ = host_tensor(29, "v", (B, n_kv, T, d), "bf16")
    bm = torch.zeros(B, H, 2, 4, dtype=torch.uint8, device="cuda")
    bm[0, 0, 1, :] = 1
    lse = torch.empty(B, H, T, device="cuda")
    out = ga.ga_attend(q, k, v, block_mask=bm, lse=lse)
    assert torch.all(out[0, 1] == 0) and torch.all(out[0, 0, :128] == 0)
    assert torch.all(torch.isinf(lse[0, 1])) and torch.all(lse[0, 1] < 0)
    sink = torch.tensor([0.5, -0.25], device="cuda")
    ga.ga_attend(q, k, v, block_mask=bm, lse=lse, sink=sink)
    assert torch.allclose(lse[0, 1], torch.full_like(lse[0, 1], -0.25))


def test_dense_mask_matches_no_mask():
    """An all-ones block mask computes what no mask computes.  At d = 128 the two run different
    kernels (the block-mask one walks a compacted tile list), so they agree within the bf16
    tolerance and each matches the oracle; two masked runs with identical masks agree bitwise."""
    B, H, n_kv, T, d = 1, 4, 2, 640, 128
    q, qr = host_tensor(31, "q", (B, H, T, d), "bf16")
    k, kr = host_tensor(31, "k", (B, n_kv, T, d), "bf16")
    v, vr = host_tensor(31, "v", (B, n_kv, T, d), "bf16")
    a = ga.ga_attend(q, k, v)
    bm = torch.ones(B, H, 5, 10, dtype=torch.uint8, device="cuda")
    b = ga.ga_attend(q, k, v, block_mask=bm)
    c = ga.ga_attend(q, k, v, block_mask=bm.clone())
    ref, _ = oracle.attend(qr, kr, vr)
    assert_close(to_f64(a), ref, "bf16", "no mask")
    assert_close(to_f64(b), ref, "bf16", "all-ones mask")
    assert_close(to_f64(a), to_f64(b), "bf16", "no mask vs all-ones mask")
    assert torch.equal(b.view(torch.int16), c.view(torch.int16))


def test_window_at_least_length_equals_full_causal_bitwise():
    B, H, n_kv, T, d = 1, 2, 1, 300, 256
    q, _ = host_tensor(37, "q", (B, H, T, d), "bf16")
    k, _ = host_tensor(37, "k", (B, n_kv, T, d), "bf16")
    v, _ = host_tensor(37, "v", (B, n_kv, T, d), "bf16")
    a = ga.ga_attend(q, k, v)
    b = ga.ga_attend(q, k, v, window=300)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_gqa_equals_mha_on_replicated_kv():
    B, H, n_kv, T, d = 1, 8, 2, 260, 128
    q, _ = host_tensor(41, "q", (B, H, T, d), "bf16")
    k, _ = host_tensor(41, "k", (B, n_kv, T, d), "bf16")
    v, _ = host_tensor(41, "v", (B, n_kv, T, d), "bf16")
    a = ga.ga_attend(q, k, v)
    b = ga.ga_attend(q, k.repeat_interleave(4, dim=1).contiguous(), v.repeat_interleave(4, dim=1).contiguous())
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_failure_path_reports_device_timeout_and_context_survives():
    """A kernel that waits on a flag nothing sets gives up after its limit, records
    GA_ERR_DEVICE_TIMEOUT, and the context keeps working."""
    assert ga.ga_read_device_status() == ga.GA_OK
    assert ga.ga_selftest_wait_timeout(50_000_000) == ga.GA_OK
    assert ga.ga_read_device_status() == ga.GA_ERR_DEVICE_TIMEOUT
    assert ga.ga_read_device_status() == ga.GA_OK        # cleared by the read
    check(run_case(1, 2, 1, 64, 64, 128, "bf16", seed=43), "bf16", "after timeout")


@pytest.mark.parametrize("d,masked", [(128, False), (256, False), (128, True)])
def test_prefill_pipeline_wait_runs_out_then_recovers(d, masked):
    """The waits inside the tensor-core prefill's TMA/MMA pipeline are bounded too: with one K
    chunk never loaded (a test-only switch) on a one-CTA launch (one query tile over 1024 keys,
    8 key tiles) and a 1 ms limit, the launch ends by itself with GA_ERR_DEVICE_TIMEOUT
    recorded -- its warps leave together, drain their loads and MMAs and free tensor memory --
    and the next launches on the same context are exact again."""
    B, H, n_kv, Tq, Tk = 1, 1, 1, 128, 1024
    q, _ = host_tensor(45, "q", (B, H, Tq, d), "bf16")
    k, _ = host_tensor(45, "k", (B, n_kv, Tk, d), "bf16")
    v, _ = host_tensor(45, "v", (B, n_kv, Tk, d), "bf16")
    bm = torch.ones(B, H, 1, Tk // 64, dtype=torch.uint8, device="cuda") if masked else None
    assert ga.ga_read_device_status() == ga.GA_OK
    ga.ga_set_wait_timeout_ns(1_000_000)
    ga.ga_selftest_drop_prefill_chunk(3)
    try:
        ga.ga_attend(q, k, v, block_mask=bm)
        assert ga.ga_read_device_status() == ga.GA_ERR_DEVICE_TIMEOUT
    finally:
        ga.ga_selftest_drop_prefill_chunk(-1)
        ga.ga_set_wait_timeout_ns(2_000_000_000)
    assert ga.ga_read_device_status() == ga.GA_OK
    check(run_case(1, 4, 2, 300, 300, d, "bf16", seed=46, mask_density=0.6 if masked else None),
          "bf16", "after a pipeline timeout")
