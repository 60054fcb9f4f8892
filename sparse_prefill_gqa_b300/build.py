"""Builds libga.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc, and its debug build
libga_debug.so (the same sources with GA_DEBUG defined: in-kernel bounds checks of the output
stores and TMA coordinates, see ga_debug_violation in include/ga.h).

    python -m sparse_prefill_gqa_b300.build [-v] [--debug]

The library links the CUDA runtime statically and takes cuTensorMapEncodeTiled from the
driver at run time, so the .so loads on a machine without a GPU (it then only fails at the
first CUDA call).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libga.so")
LIB_DEBUG = os.path.join(HERE, "libga_debug.so")
SOURCES = [os.path.join(CSRC, "ga.cu")]
HEADERS = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cuh", ".h"))]
HEADERS.append(os.path.join(ROOT, "include", "ga.h"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libga")
    return path


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile libga.so (libga_debug.so with `debug`) if any source is newer than it; returns the
    library path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not stale(lib):
        return lib
    cmd = [nvcc(), *ARCH, *FLAGS, *(["-DGA_DEBUG"] if debug else []), *(["-Xptxas", "-v"] if verbose else []),
           *SOURCES, "-o", lib + ".tmp"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
