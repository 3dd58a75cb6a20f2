"""In-tree build of libccl.so for sm_103a with nvcc (no cmake, one TU)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = [os.path.join(HERE, "csrc", "ccl.cu")]
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libccl.so")
# the same library with event counters compiled in (ccl_debug_counters); never
# the one the product path loads
COUNTERS_LIB_PATH = os.path.join(BUILD_DIR, "libccl_counters.so")

NVCC_FLAGS = ["-std=c++17", "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
              "-lineinfo", "-Xcompiler", "-fPIC", "-shared"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(path):
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = SRC + [os.path.join(INCLUDE, "ccl.h")] + [
        os.path.join(HERE, "csrc", f) for f in os.listdir(os.path.join(HERE, "csrc"))]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, counters: bool = False) -> str:
    """Compile csrc/*.cu into _build/libccl.so (skipped when up to date); with
    ``counters``, into _build/libccl_counters.so with the event counters on."""
    path = COUNTERS_LIB_PATH if counters else LIB_PATH
    if not force and not _stale(path):
        return path
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = path + ".tmp%d" % os.getpid()
    cmd = [_nvcc()] + NVCC_FLAGS + (["-DCCL_COUNTERS"] if counters else []) + \
        ["-I", INCLUDE, "-o", tmp] + SRC
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, path)
    return path
