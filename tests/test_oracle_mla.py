"""Pins of the MLA oracle ("Attention in Code", section 4): the naive and absorbed forms agree
for arbitrary weights (the page reports 1.1e-15), in prefill and at a single decode step, with
DeepSeek-V2-Lite's shapes (latent 512, rope 64, head dims 128)."""
import numpy as np

from oracle.mla import mla_absorbed, mla_naive


def _rand(shape, seed, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal(shape)


def test_naive_equals_absorbed_small():
    H, T, L, dn, dr, r, dv = 4, 9, 9, 8, 4, 16, 8
    args = (_rand((H, T, dn), 601), _rand((H, T, dr), 602), _rand((L, r), 603), _rand((L, dr), 604),
            _rand((H, r, dn), 605, 0.3), _rand((H, r, dv), 606, 0.3))
    assert np.max(np.abs(mla_naive(*args) - mla_absorbed(*args))) <= 1e-12


def test_naive_equals_absorbed_decode_step_at_v2_lite_shapes():
    """One new token (T = 1) over 300 cached latents, 16 heads, r = 512, dr = 64, dn = dv = 128."""
    H, T, L, dn, dr, r, dv = 16, 1, 300, 128, 64, 512, 128
    args = (_rand((H, T, dn), 611), _rand((H, T, dr), 612), _rand((L, r), 613), _rand((L, dr), 614),
            _rand((H, r, dn), 615, 1 / np.sqrt(r)), _rand((H, r, dv), 616, 1 / np.sqrt(r)))
    a, b = mla_naive(*args), mla_absorbed(*args)
    assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(a)))
