"""Build the gbthist CUDA library in-tree with nvcc for sm_103a.

``build()`` compiles ``csrc/gbthist.cu`` (one translation unit) into
``_build/libgbthist.so``; it is re-run when any source or the public header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC_DIR = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libgbthist.so")
HEADER = os.path.join(ROOT, "include", "gbthist.h")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _sources():
    return sorted(glob.glob(os.path.join(SRC_DIR, "*.cu")) + glob.glob(os.path.join(SRC_DIR, "*.cuh"))) + [HEADER]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the gbthist CUDA library cannot be built")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB_PATH):
        lib_m = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(s) <= lib_m for s in _sources()):
            return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
           "-o", tmp, os.path.join(SRC_DIR, "gbthist.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
