"""Build libmoe.so (the CUDA kernels and the C ABI) in-tree for sm_103a with nvcc.

    python -m mixture_experts_sparse_02_b300.build [--force] [--debug-bounds]

Object files and the ptxas resource report (-Xptxas -v) go to _build/ at the repository root.
--debug-bounds builds libmoe_debug.so instead: the same library compiled with MOE_DEBUG_BOUNDS,
whose kernels also report (in the device error word, bit ERR_BOUNDS) any index they read from
offsets, perm_tok, inv_pos or pos_of that is out of range.  The binding loads it when the
environment variable MOE_LIBRARY is "debug".
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
LIB_DEBUG = os.path.join(PKG, "libmoe_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    out_dir = os.path.join(BUILD, "debug") if debug_bounds else BUILD
    lib = LIB_DEBUG if debug_bounds else LIB
    defines = ["-DMOE_DEBUG_BOUNDS=1"] if debug_bounds else []
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    hdrs = _headers()
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [cc, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(obj + ".log", "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (os.path.basename(src), r.stderr[-4000:]))
        return obj

    with cf.ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(compile_one, jobs))
    if force or jobs or _stale(lib, objs):
        cmd = [cc, *ARCH, "-shared", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stderr[-4000:])
    with open(os.path.join(out_dir, "ptxas.txt"), "w") as f:
        for obj in objs:
            if os.path.exists(obj + ".log"):
                f.write(open(obj + ".log").read())
    if verbose:
        print(open(os.path.join(out_dir, "ptxas.txt")).read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
