"""The Python binding has no CPU path: host tensors are refused before any call into the library,
tensors shorter than the kernels index are refused, and a missing libga.so raises."""
import pytest
import torch

import sparse_prefill_gqa_b300 as ga


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def _f(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def _i(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


CALLS = {
    "ga_attend": lambda: ga.ga_attend(_bf(1, 2, 4, 128), _bf(1, 1, 4, 128), _bf(1, 1, 4, 128)),
    "ga_attend_decode_static": lambda: ga.ga_attend_decode_static(_bf(1, 2, 1, 128), _bf(1, 1, 4, 128),
                                                                  _bf(1, 1, 4, 128)),
    "ga_attend_diff": lambda: ga.ga_attend_diff(_bf(1, 2, 4, 128), _bf(1, 1, 4, 128), _bf(1, 2, 4, 128),
                                                _bf(1, 1, 4, 128), _bf(1, 1, 4, 128), 0.5),
    "ga_dsa_indexer": lambda: ga.ga_dsa_indexer(_bf(1, 8, 128), _f(1, 8), _bf(1, 64, 128)),
    "ga_topk_indices": lambda: ga.ga_topk_indices(_f(1, 64), 8),
    "ga_attend_gather": lambda: ga.ga_attend_gather(_bf(1, 2, 1, 128), _bf(1, 1, 64, 128), _bf(1, 1, 64, 128),
                                                    _i(1, 8), _i(1)),
    "ga_mla_decode": lambda: ga.ga_mla_decode(_bf(1, 2, 128), _bf(1, 2, 64), _bf(1, 16, 576), _bf(2, 512, 128),
                                              _bf(2, 512, 128)),
    "ga_ring_append": lambda: ga.ga_ring_append(_bf(1, 1, 8, 64), _bf(1, 1, 8, 64), _bf(1, 1, 64),
                                                _bf(1, 1, 64), _i(1)),
    "ga_attend_ring": lambda: ga.ga_attend_ring(_bf(1, 2, 1, 64), _bf(1, 1, 8, 64), _bf(1, 1, 8, 64), _i(1)),
    "ga_block_stats": lambda: ga.ga_block_stats(_bf(1, 1, 128, 128)),
    "ga_select_blocks": lambda: ga.ga_select_blocks(_bf(1, 2, 128, 128), _f(1, 1, 2, 128), _f(1, 1, 2)),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA tensor"):
        CALLS[name]()


def test_short_tensors_are_refused():
    with pytest.raises(ValueError, match="at least 4 elements"):
        ga._need_size(_i(3), "k_lens", 4)
    ga._need_size(_i(4), "k_lens", 4)


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(ga, "_LIB", None)
    monkeypatch.setattr(ga, "library_path", lambda: "/nonexistent/libga.so")
    with pytest.raises(RuntimeError, match="not built"):
        ga.lib()


class _OnDevice:
    """Stands in for a tensor or stream by its device alone (no GPU is needed to check the rule)."""

    def __init__(self, dev):
        self.device = torch.device(dev)


def test_tensors_on_several_devices_are_refused():
    """The library launches on the calling thread's current device with that device's stream and
    static scratch: tensors (or an explicit stream) on another device are refused before any call."""
    a, b = _OnDevice("cuda:0"), _OnDevice("cuda:1")
    assert ga._one_device([a, None, a]) == torch.device("cuda:0")
    assert ga._one_device([b], stream=_OnDevice("cuda:1")) == torch.device("cuda:1")
    with pytest.raises(ValueError, match="one CUDA device"):
        ga._one_device([a, b])
    with pytest.raises(ValueError, match="one CUDA device"):
        ga._one_device([a, a], stream=_OnDevice("cuda:1"))
