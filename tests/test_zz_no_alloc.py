"""ga_attend_decode_static: the split-K decode for callers that cannot allocate device memory
(an engine that owns the whole device-memory pool, or a loop where cudaMalloc/cudaFree would
synchronise the device).  Its scratch is a static device array inside the library, shared by
every call, so these tests check that two calls in a row -- different shapes, the second
reading scratch the first one left behind -- each give exactly what ga_attend gives with a
workspace the caller allocated (the same kernels run the same arithmetic, so the outputs must
be bit-identical), and that a call allocates no device memory.

The file name makes pytest collect it last, so that a run stopping at the first failure has
already run every other test when this one runs (``pytest --collect-only`` shows the order);
the tests also pass alone, in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_prefill_gqa_b300 as ga
from tests.helpers import host_tensor, to_f64


def test_oversized_shape_is_rejected_before_any_cuda_call():
    """Runs without a GPU: the size check comes before the library touches CUDA."""
    L = ga.lib()
    p = ctypes.c_void_p(4096)
    need = ga.ga_workspace_size(512, 32, 8, 128, 1, 32768, torch.bfloat16)
    assert need > ga.GA_DECODE_STATIC_SCRATCH_BYTES
    st = L.ga_attend_decode_static(p, p, p, p, 512, 32, 8, 128, 1, 32768, None, 1, 0, None, None, None)
    assert st == ga.GA_ERR_SCRATCH_LIMIT
    assert "static" in ga.ga_status_string(st)
    # shapes off the split-K decode path (prefill-sized Tq) are not taken
    st = L.ga_attend_decode_static(p, p, p, p, 1, 8, 2, 128, 512, 4096, None, 1, 0, None, None, None)
    assert st == ga.GA_ERR_UNSUPPORTED


def _decode_case(seed, B, H, n_kv, Tq, Tk, d, lens, window=0, sink=False):
    q, _ = host_tensor(seed, "q", (B, H, Tq, d), "bf16")
    k, _ = host_tensor(seed, "k", (B, n_kv, Tk, d), "bf16")
    v, _ = host_tensor(seed, "v", (B, n_kv, Tk, d), "bf16")
    k_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sk = None
    if sink:
        sk = torch.from_numpy(np.random.default_rng(seed).standard_normal(H).astype(np.float32)).cuda()
    need = ga.ga_workspace_size(B, H, n_kv, d, Tq, Tk, torch.bfloat16)
    assert 0 < need <= ga.GA_DECODE_STATIC_SCRATCH_BYTES     # the scratch really is used
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    lse_ref = torch.empty(B, H, Tq, device="cuda")
    lse_got = torch.empty(B, H, Tq, device="cuda")
    ref = ga.ga_attend(q, k, v, k_lens=k_lens, window=window, sink=sk, lse=lse_ref, workspace=ws)
    got = ga.ga_attend_decode_static(q, k, v, k_lens=k_lens, window=window, sink=sk, lse=lse_got)
    assert ga.ga_read_device_status() == ga.GA_OK
    return to_f64(got), to_f64(ref), to_f64(lse_got), to_f64(lse_ref)


@pytest.mark.gpu
def test_static_scratch_decode_matches_workspace_decode_on_two_calls_in_a_row():
    cases = [
        dict(seed=61, B=8, H=32, n_kv=8, Tq=1, Tk=20000, d=128,
             lens=[20000, 17001, 1, 9999, 12345, 20000, 640, 5000], sink=True),
        dict(seed=62, B=3, H=16, n_kv=4, Tq=2, Tk=9000, d=64, lens=[9000, 4321, 700], window=500),
    ]
    for c in cases:
        got, ref, lse_got, lse_ref = _decode_case(**c)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, ref), (c["seed"], np.abs(got - ref).max())
        assert np.array_equal(lse_got, lse_ref), c["seed"]


@pytest.mark.gpu
def test_static_scratch_decode_allocates_no_device_memory():
    """After a first call (which may load the kernels' code on the device), a second call with
    every output passed in leaves the device's free memory and PyTorch's allocator unchanged."""
    B, H, n_kv, Tq, Tk, d = 4, 32, 8, 1, 16384, 128
    q, _ = host_tensor(71, "q", (B, H, Tq, d), "bf16")
    k, _ = host_tensor(71, "k", (B, n_kv, Tk, d), "bf16")
    v, _ = host_tensor(71, "v", (B, n_kv, Tk, d), "bf16")
    assert ga.ga_workspace_size(B, H, n_kv, d, Tq, Tk, torch.bfloat16) > 0
    out = torch.empty_like(q)
    lse = torch.empty(B, H, Tq, device="cuda")
    ga.ga_attend_decode_static(q, k, v, out, lse=lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    ga.ga_attend_decode_static(q, k, v, out, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == reserved0
    assert ga.ga_read_device_status() == ga.GA_OK
