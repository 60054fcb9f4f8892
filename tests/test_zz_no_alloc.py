"""ga_attend_decode_static: the split-K decode for callers that cannot allocate device memory
(an engine that owns the whole device-memory pool, or a loop where cudaMalloc/cudaFree would
synchronise the device).  Its scratch is a static device array inside the library, shared by
every call, so these tests check that two calls in a row -- different shapes, the second
reading scratch the first one left behind -- each give what ga_attend gives with a workspace
the caller allocated.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_prefill_gqa_b300 as ga
from tests.helpers import BF16_MAX_ABS, BF16_REL_L2, host_tensor, to_f64


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
        err = np.abs(got - ref).max()
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err <= BF16_MAX_ABS and rel <= BF16_REL_L2, (c["seed"], err, rel)
        assert np.max(np.abs(lse_got - lse_ref)) <= 2e-3, c["seed"]
