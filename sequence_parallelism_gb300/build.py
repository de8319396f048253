"""Compile the CUDA library in-tree for sm_103a.

    python sequence_parallelism_gb300/build.py     (or __graft_entry__.build())

Every translation unit under csrc/ is compiled by nvcc in parallel into
_build/, then linked into sequence_parallelism_gb300/libsp_gb300.so (CUDA
runtime linked statically, so the library needs only the driver).  Set
SP_NVCC_EXTRA for extra nvcc flags (e.g. "-Xptxas -v").
"""

import concurrent.futures
import glob
import os
import shlex
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsp_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsp_gb300.so")


def _flags():
    extra = shlex.split(os.environ.get("SP_NVCC_EXTRA", ""))
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC] + extra


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    deps = [src] + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include",
                                                                          "sp_gb300.h")]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, force=False):
    """Build libsp_gb300.so; returns its path.  Raises on a compiler error."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, src):
            jobs.append([nvcc] + _flags() + ["-c", src, "-o", obj])
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in _sources()]

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    failed = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose or p.returncode != 0:
                sys.stdout.write(p.stdout)
                sys.stderr.write(p.stderr)
            if p.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB)
                                             for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            sys.stderr.write(p.stdout + p.stderr)
            raise RuntimeError("link of libsp_gb300.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
