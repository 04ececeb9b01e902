"""Compile the CUDA library in tree (sm_103a only).

``build_library()`` compiles each translation unit under ``csrc/`` to an object file
with nvcc (in parallel, one process per unit), then links them into
``libspecreject.so`` next to this file.  No CMake.
"""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
HEADERS = [os.path.join(ROOT, "include", "spec_reject.h")] + sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
LIBRARY = os.path.join(HERE, "libspecreject.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def nvcc_path() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def build_library(force: bool = False, verbose: bool = False, defines=()) -> str:
    """Build (or reuse, when newer than every source and header) the shared library.
    `defines` are extra -D settings of the kernels' compile-time tunables."""
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS)
    if not force and not defines and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= newest:
        return LIBRARY
    tag = f".tmp{os.getpid()}"
    extra = [f"-D{d}" for d in defines] + (["-Xptxas=-v"] if verbose else [])
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(CSRC, os.path.basename(src) + tag + ".o")
        objs.append(obj)
        procs.append(subprocess.Popen([nvcc_path(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]))
    rcs = [p.wait() for p in procs]
    try:
        if any(rcs):
            raise subprocess.CalledProcessError(max(rcs), "nvcc")
        tmp = LIBRARY + tag
        subprocess.check_call([nvcc_path(), *ARCH, "-shared", *objs, "-o", tmp, "-lcudart"])
        os.replace(tmp, LIBRARY)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.unlink(o)
    return LIBRARY


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
