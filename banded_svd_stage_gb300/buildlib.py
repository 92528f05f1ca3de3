"""Build libbb.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel, then linked into a shared
library next to this file.  Object files go to ``_build/`` (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")
LIB_PATH = os.path.join(HERE, "libbb.so")
SOURCES = ["bb_api.cu", "bb_kernels_f32.cu", "bb_kernels_f64.cu", "bb_kernels_f32_narrow.cu",
           "bb_kernels_f32_wide.cu", "bb_kernels_f64_narrow.cu", "bb_kernels_f64_wide.cu", "bb_noalloc.cu",
           "bb_svals.cu", "bb_plan.cu", "bb_sym.cu", "bb_sym_group_f32.cu", "bb_sym_group_f64.cu",
           "bb_vectors.cu", "bb_half.cu", "bb_stage1.cu"]
# The pass kernels: their device code and the host planner that fixes their
# launch shape.  The C-ABI checks (bb_api.cu), the allocation-free entry
# (bb_noalloc.cu) and the singular-value kernel (bb_svals.cu) are not part of
# them.
PASS_KERNEL_SOURCES = ["bb_device.cuh", "bb_group.cuh", "bb_launch.cuh", "bb_internal.h", "bb_plan.cu",
                       "bb_kernels_f32.cu", "bb_kernels_f64.cu", "bb_kernels_f32_narrow.cu",
                       "bb_kernels_f32_wide.cu", "bb_kernels_f64_narrow.cu", "bb_kernels_f64_wide.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", CSRC, "-I", INCLUDE, *extra]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "bb.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not extra_flags and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [exe, *_flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ())
    print(LIB_PATH)


def source_digest() -> str:
    """sha256 of the pass kernels' sources (PASS_KERNEL_SOURCES): it changes
    exactly when a pass kernel or its launch plan may have changed, so DRAM
    counters taken under another digest no longer describe the kernel."""
    import hashlib
    h = hashlib.sha256()
    for f in PASS_KERNEL_SOURCES:
        h.update(f.encode())
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]
