"""Build libw4a16sv.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled to an object in parallel, then linked into
speculative_decode_verify_w4a16_gb300/libw4a16sv.so (CUDA runtime linked
statically, so the library needs no particular libcudart on the loader path).
Usage: python -m speculative_decode_verify_w4a16_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(os.path.dirname(PKG), "_build", "w4a16sv")
LIB = os.path.join(PKG, "libw4a16sv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*"))) + [os.path.join(os.path.dirname(PKG), "include", "w4a16sv.h")]


# Debug build for the tests that make a kernel's bounded wait run out: a
# separate library outside the package (the product never loads it) with a
# 5 ms wait limit and the test hooks compiled in.
DEBUG_LIB = os.path.join(os.path.dirname(PKG), "_build", "libw4a16sv_debug.so")
DEBUG_FLAGS = ["-DW4A16_WAIT_LIMIT_NS=5000000ull", "-DW4A16_TEST_HOOKS=1"]


def build_debug(force: bool = False) -> str:
    """Build the debug library (see DEBUG_FLAGS) and return its path."""
    return build(force=force, extra_flags=DEBUG_FLAGS, out=DEBUG_LIB,
                 obj_dir=os.path.join(os.path.dirname(PKG), "_build", "w4a16sv_debug"))


# Bounds-checked library for the tests: every instrumented global index is
# checked against its buffer and a miss is recorded in the device error word
# (W4A16_ERR_BOUNDS) instead of being performed. Outside the package; the
# product never loads it.
BOUNDS_LIB = os.path.join(os.path.dirname(PKG), "_build", "libw4a16sv_bounds.so")
BOUNDS_FLAGS = ["-DW4A16_BOUNDS_CHECK=1"]


def build_bounds(force: bool = False) -> str:
    """Build the bounds-checked library (see BOUNDS_FLAGS) and return its path."""
    return build(force=force, extra_flags=BOUNDS_FLAGS, out=BOUNDS_LIB,
                 obj_dir=os.path.join(os.path.dirname(PKG), "_build", "w4a16sv_bounds"))


def build(force: bool = False, verbose: bool = False, extra_flags=None, out: str = LIB, obj_dir: str = BUILD) -> str:
    stale = not os.path.exists(out) or any(os.path.getmtime(f) > os.path.getmtime(out) for f in _deps())
    if not force and not stale:
        return out
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc] + ARCH + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)
    print(LIB)
