"""Shared test helpers: seeded tensors on host and device, and the parity tolerances."""
from __future__ import annotations

import numpy as np
import torch

from workloads import bf16_bits_to_f32, randn_bhtd

# Tolerances (stated for unit-variance inputs):
#   fp32 storage: max |gpu - oracle| <= 1e-5
#   bf16 storage: max |gpu - oracle| <= 2e-2 and ||gpu - oracle|| / ||oracle|| <= 5e-3
F32_MAX_ABS = 1e-5
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3


def host_tensor(seed, tag, shape, dtype, lengths=None):
    """(device tensor, float64 host copy of exactly the stored values)."""
    bits = randn_bhtd(seed, tag, shape, dtype, lengths=lengths)
    if dtype == "bf16":
        dev = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        ref = bf16_bits_to_f32(bits).astype(np.float64)
    else:
        dev = torch.from_numpy(bits)
        ref = bits.astype(np.float64)
    return dev.cuda(), ref


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    err = np.abs(gpu - ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{what}: max abs {err.max():.3g}"
    else:
        rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err.max() <= BF16_MAX_ABS, f"{what}: max abs {err.max():.3g}"
        assert rel <= BF16_REL_L2, f"{what}: rel L2 {rel:.3g}"


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 values rounded to the nearest bf16 (for oracle inputs built on the host)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.float().numpy().astype(np.float64)
