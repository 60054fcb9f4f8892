"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package holds input generation only: random draws, the fp32 -> bf16 storage cast,
the workload shapes and the choice of sampled query rows.  It contains none of the
attention, block-statistics or block-selection arithmetic, so the oracle and the CUDA
path can both be fed from it without sharing any of the method's code.
"""
from .gen import (bf16_bits_to_f32, f32_to_bf16_bits, normal_slices, planted_outliers,
                  randn_bhtd, sample_rows, uniform_lengths)
from .configs import CONFIGS, Config, get_config

__all__ = [
    "CONFIGS", "Config", "get_config", "bf16_bits_to_f32", "f32_to_bf16_bits",
    "normal_slices", "planted_outliers", "randn_bhtd", "sample_rows", "uniform_lengths",
]
