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
# The same library with device-side bounds checks (-DGQA_DEBUG): every
# global write of the decode kernel is checked against its buffer and
# skipped if outside it, every TMA tile origin against its tensor; either
# shows as GQA_ERR_BOUNDS from gqa_decode_get_error.  For testing only.
DEBUG_LIB = os.path.join(PKG, "libgqa_decode_sm103_debug.so")
# The same library with the decode kernel's clock64 event trace
# (-DGQA_TRACE): gqa_trace_attach() names a device buffer that the following
# launches stamp per CTA, role and block.  For measurement only.
TRACE_LIB = os.path.join(PKG, "libgqa_decode_sm103_trace.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh", ".h"))] + [HEADER]


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(s) <= t for s in sources())


# Translation units: the host side (C ABI, planning, combine kernel) and one
# unit per head_dim and merge mode holding that combination's decode kernels,
# compiled in parallel and linked into one shared library.
INSTANCES = [(hd, cl) for hd in (64, 128, 256) for cl in (0, 1)]


def _units(build_dir: str):
    units = [(os.path.join(CSRC, "gqa_decode.cu"), [], os.path.join(build_dir, "gqa_decode.o"))]
    for hd, cl in INSTANCES:
        units.append((os.path.join(CSRC, "decode_instances.cu"), [f"-DGQA_INST_HD={hd}", f"-DGQA_INST_CLUSTER={cl}"],
                      os.path.join(build_dir, f"decode_{hd}_{cl}.o")))
    return units


def build(force: bool = False, out: str = LIB, extra_flags=(), verbose: bool = False) -> str:
    """Compile the csrc translation units for sm_103a (in parallel) and link
    them into ``out`` (skipped if current)."""
    if not force and up_to_date(out):
        return out
    build_dir = os.path.join(os.path.dirname(os.path.abspath(out)), "_build",
                             os.path.splitext(os.path.basename(out))[0])
    os.makedirs(build_dir, exist_ok=True)
    base = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), *extra_flags]
    if verbose:
        base.insert(1, "-Xptxas=-v")
    procs = []
    for src, defs, obj in _units(build_dir):
        procs.append((obj, subprocess.Popen([*base, *defs, "-c", src, "-o", obj])))
    failed = [obj for obj, p in procs if p.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, f"nvcc ({', '.join(os.path.basename(f) for f in failed)})")
    subprocess.run([_nvcc(), ARCH, "-shared", *[obj for obj, _ in procs], "-o", out + ".tmp"], check=True)
    os.replace(out + ".tmp", out)
    return out


def build_debug(force: bool = False) -> str:
    """The -DGQA_DEBUG build of the library (bounds-checked), beside the other."""
    return build(force=force, out=DEBUG_LIB, extra_flags=("-DGQA_DEBUG",))


def build_trace(force: bool = False) -> str:
    """The -DGQA_TRACE build of the library (event stamps), beside the other."""
    return build(force=force, out=TRACE_LIB, extra_flags=("-DGQA_TRACE",))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
