import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of CPU oracle time)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _debug_build_records_no_violation(request):
    """Under the debug build (GA_DEBUG_RUN set, the library libga_debug.so), every GPU test also
    requires that no in-kernel bounds check failed while it ran."""
    if not os.environ.get("GA_DEBUG_RUN") or "gpu" not in request.keywords:
        yield
        return
    import sparse_prefill_gqa_b300 as ga
    assert ga.ga_debug_violation() == 0, "a check failed before the test"
    yield
    first = ga.ga_debug_violation()
    assert first is not None, "GA_DEBUG_RUN is set but the loaded library has no checks"
    assert first == 0, f"in-kernel bounds check failed: site {first >> 48}, offset {first & ((1 << 48) - 1)}"
