"""Builds the sm_103a shared library in-tree with nvcc.

The library is a plain C-ABI ``.so`` (see ``include/gqa_decode.h``); nothing
here links against PyTorch.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
HEADER = os.path.join(ROOT, "include", "gqa_decode.h")
LIB = os.path.join(PKG, "libgqa_decode_sm103.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh"))] + [HEADER]


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, out: str = LIB, extra_flags=(), verbose: bool = False) -> str:
    """Compile csrc/gqa_decode.cu for sm_103a into ``out`` (skipped if current)."""
    if not force and up_to_date(out):
        return out
    cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), *extra_flags,
           "-o", out + ".tmp", os.path.join(CSRC, "gqa_decode.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
