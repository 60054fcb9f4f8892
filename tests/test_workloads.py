"""The seeded input generators: determinism, slice regeneration and the bf16 storage cast."""
import numpy as np
import torch

from workloads import (bf16_bits_to_f32, f32_to_bf16_bits, normal_slices, planted_outliers,
                       randn_bhtd, sample_rows, uniform_lengths)


def test_bf16_cast_matches_torch():
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 37.0
    x[:6] = [0.0, -0.0, 1.0, 3.1415927, 1e-30, -65504.0]
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_slices_regenerate_and_do_not_depend_on_threads():
    a = randn_bhtd(7, "k", (2, 3, 50, 8), lengths=[50, 20], threads=1)
    b = randn_bhtd(7, "k", (2, 3, 50, 8), lengths=[50, 20], threads=4)
    assert np.array_equal(a, b)
    assert np.array_equal(a[1, 2, :20], normal_slices(7, "k", 1, 2, 20, 8))
    assert np.all(a[1, :, 20:] == 0)
    assert not np.array_equal(a[0, 0], randn_bhtd(7, "v", (2, 3, 50, 8))[0, 0])


def test_lengths_plants_and_rows():
    lens = uniform_lengths(3, 64, 16384, 32768)
    assert lens.dtype == np.int32 and lens.min() >= 16384 and lens.max() <= 32768
    p = planted_outliers(5, 2, 64 * 100, 16, 64)
    assert len(p) == 10 and all(tok // 64 == blk for _, blk, tok, _ in p)
    assert all(abs(np.linalg.norm(vec) - 32.0) < 1e-3 for _, _, _, vec in p)
    rows = sample_rows(8192, 256, seed=9, q_block=128, window=1024)
    assert len(rows) == 256 and rows[0] == 0 and rows[-1] == 8191 and 1023 in rows
    assert np.all(np.diff(rows) > 0)
