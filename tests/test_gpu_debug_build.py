"""The debug build (libga_debug.so: the same sources with GA_DEBUG, in-kernel bounds checks of
every output store and TMA coordinate, first failure recorded in a sticky word) under the
small ragged-shape suites: the canary-padding tests (every entry point), the attention tests
(prefill and decode paths, masks, windows, sinks, poisoned tails), top-k and MLA.  They run in a
child process with the debug library loaded, and every test there also requires that no check
failed while it ran (tests/conftest.py)."""
import os
import subprocess
import sys

import pytest

from sparse_prefill_gqa_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_small_suites_under_the_debug_build_record_no_violation():
    lib = build.build(debug=True)
    env = dict(os.environ, GA_LIBRARY=lib, GA_DEBUG_RUN="1")
    suites = ["tests/test_gpu_canary.py", "tests/test_gpu_attend.py", "tests/test_gpu_dsa.py", "tests/test_gpu_mla.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *suites, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
