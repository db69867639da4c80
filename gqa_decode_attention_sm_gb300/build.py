"""Build libgqa_decode.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libgqa_decode.so")
INCLUDE = os.path.join(ROOT, "include")
MAIN_SRC = os.path.join(PKG, "csrc", "gqa_decode.cu")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def _sources():
    return ([MAIN_SRC] + glob.glob(os.path.join(PKG, "csrc", "**", "*.cuh"), recursive=True)
            + glob.glob(os.path.join(PKG, "csrc", "**", "*.cu"), recursive=True)
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than any source."""
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(s) for s in _sources())
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-I" + INCLUDE, "-o", tmp, MAIN_SRC]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


CHECKED_LIB_PATH = os.path.join(PKG, "libgqa_decode_checked.so")


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """The same library with every kernel access range-checked (-DGQA_CHECKED):
    an access outside its buffer sets GQA_FLAG_BOUNDS and is redirected inside
    it.  For tests only; the product library is built without the checks."""
    if not force and os.path.exists(CHECKED_LIB_PATH):
        newest = max(os.path.getmtime(s) for s in _sources())
        if os.path.getmtime(CHECKED_LIB_PATH) >= newest:
            return CHECKED_LIB_PATH
    tmp = CHECKED_LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-DGQA_CHECKED", "-I" + INCLUDE, "-o", tmp, MAIN_SRC]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, CHECKED_LIB_PATH)
    return CHECKED_LIB_PATH
