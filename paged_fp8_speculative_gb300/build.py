"""Build libmtpattn.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Every ``csrc/*.cu`` file compiles to an object in parallel, then one link makes
``paged_fp8_speculative_gb300/libmtpattn.so``.  Run as ``python -m
paged_fp8_speculative_gb300.build`` or through ``__graft_entry__.build()``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmtpattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmtpattn.so")


def build(verbose: bool = False, extra_flags=(), lib_path: str = LIB) -> str:
    """Compile every csrc/*.cu and link ``lib_path``.  ``extra_flags`` (e.g. the test-only
    -DMTPATTN_WAIT_CYCLES / -DMTPATTN_TEST_STALL of the wait-limit test) go to every nvcc;
    such builds use their own object folder and library path."""
    obj_dir = BUILD if lib_path == LIB else os.path.join(BUILD, os.path.splitext(
        os.path.basename(lib_path))[0])
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cc = nvcc()
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0 or (verbose and out):
            sys.stdout.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.check_call(cmd)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB)
