"""Build libdsc.so (the CUDA kernels + C ABI) in-tree for sm_103a.

Each .cu file under csrc/ is compiled with nvcc for
``-gencode arch=compute_103a,code=sm_103a`` into _build/, then linked into
lm_local_sequence_causal_b300/libdsc.so with the static CUDA runtime, so the
library loads without a GPU (the C ABI's argument checks run anywhere).
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdsc.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale(obj, src, hdr_mtime):
    return (not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(src)
            or os.path.getmtime(obj) < hdr_mtime)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile every kernel file and link libdsc.so; return the library path."""
    os.makedirs(BUILD, exist_ok=True)
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [0])
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, src, hdr_mtime):
            jobs.append([NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj])
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in _sources()]

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if (force or jobs or not os.path.exists(LIB)
            or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs)):
        tmp = LIB + ".tmp"
        subprocess.run([NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs],
                       check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    xtra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force="--force" in sys.argv or bool(xtra), verbose=v or bool(xtra), extra=xtra))
