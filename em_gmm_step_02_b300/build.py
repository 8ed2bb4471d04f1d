"""Build the CUDA library ``libgmm_b300.so`` in this folder (sm_103a only).

    python -m em_gmm_step_02_b300.build [--force]

nvcc compiles every ``csrc/*.cu`` for ``-gencode arch=compute_103a,code=sm_103a``
and links them with the CUDA runtime into one shared library whose C ABI is
``include/gmm.h``.  Object files go to ``_build/`` at the repository root.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libgmm_b300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include")]


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(HERE, "csrc", "*.cuh")) + \
        [os.path.join(ROOT, "include", "gmm.h"), __file__]


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(p) <= t for p in _inputs()):
            return LIB
    bdir = os.path.join(ROOT, "_build")
    os.makedirs(bdir, exist_ok=True)
    objs = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        objs.append(obj)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                           "-o", tmp, *objs, "-lcudart"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
