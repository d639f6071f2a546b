"""Build the sm_103a shared library in-tree with nvcc (no CMake, one TU)."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")
MAIN_SRC = os.path.join(HERE, "csrc", "fa_fwd.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def _sources():
    return (glob.glob(os.path.join(HERE, "csrc", "*.cu")) + glob.glob(os.path.join(HERE, "csrc", "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu into libfa_gb300.so next to this file; returns its path."""
    stale = force or not os.path.exists(LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(LIB_PATH) for s in _sources())
    if stale:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *NVCC_FLAGS, *( ["-Xptxas", "-v"] if verbose else []), "-o", tmp, MAIN_SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
