"""Build the CUDA library ``libspfused.so`` in-tree for sm_103a.

One translation unit, one ``-gencode``: ``nvcc -gencode arch=compute_103a,code=sm_103a -O3
-lineinfo -shared``. The CUDA runtime is linked statically, so the library needs only the
driver (``libcuda.so.1``) at run time, and loading it on a machine without a GPU works (every
CUDA call then fails with SP_ERR_CUDA).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "libspfused.so")
MAIN = os.path.join(CSRC, "sp_fused.cu")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library if it is missing or older than any of its sources."""
    stale = force or not os.path.exists(LIBRARY) or any(
        os.path.getmtime(s) > os.path.getmtime(LIBRARY) for s in _sources())
    if not stale and not verbose_ptxas:
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *NVCC_FLAGS, "-I", INCLUDE, MAIN, "-o", tmp]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv))
