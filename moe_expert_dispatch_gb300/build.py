"""Builds libmoe_gb300.so (and libmoe_gb300_debug.so, the same sources with
MOE_DEBUG's device-side bounds checks) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then the objects are
linked into one shared library per variant (CUDA runtime linked statically,
no link to libcuda: the tensor-map encoder is fetched through the runtime at
first use).
Run as `python moe_expert_dispatch_gb300/build.py` (or __graft_entry__.build()).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["route.cu", "gemm_bf16.cu", "gemm_mxfp8.cu", "capi.cu", "counts_static.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _needs(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


_SAN = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined"]
VARIANTS = {
    # release: the product library; debug: the same sources with MOE_DEBUG,
    # whose kernels bounds-check the row indices they take from row maps;
    # sanitize (built only on request): the host code under AddressSanitizer
    # and UndefinedBehaviorSanitizer, for the host-side argument and size
    # checks on a machine without a GPU (its process preloads the runtimes)
    "release": (BUILD, LIB, [], []),
    "debug": (os.path.join(PKG, "_build_debug"), os.path.join(PKG, "libmoe_gb300_debug.so"),
              ["-DMOE_DEBUG"], []),
    "sanitize": (os.path.join(PKG, "_build_sanitize"),
                 os.path.join(PKG, "libmoe_gb300_sanitize.so"),
                 _SAN + ["-Xcompiler", "-fno-omit-frame-pointer"], _SAN),
}


def build(verbose: bool = False, force: bool = False, variants=("release", "debug")) -> str:
    """Compiles the named variants (all their translation units in one
    parallel pool) and links each library; returns the release library's path."""
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "moe_expert.h"))
    jobs, links = [], []
    for v in variants:
        bdir, lib, extra, link_extra = VARIANTS[v]
        os.makedirs(bdir, exist_ok=True)
        objs = []
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(bdir, src.replace(".cu", ".o"))
            objs.append(o)
            if force or _needs(o, [s] + headers):
                jobs.append([nvcc(), *_flags(), *extra, "-c", s, "-o", o])
        links.append((lib, objs, link_extra))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))

    if jobs:
        with cf.ThreadPoolExecutor(len(jobs)) as ex:
            list(ex.map(run, jobs))
    for lib, objs, link_extra in links:
        if force or _needs(lib, objs):
            run([nvcc(), *ARCH, "-shared", "-o", lib, *objs, *link_extra])
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
