"""Builds libmoe_gb300.so in-tree with nvcc for sm_103a.

Each CUDA source compiles to an object in parallel, then one shared library
is linked next to this file. The CUDA runtime is the shared libcudart (the
one PyTorch has already loaded when the binding is used; otherwise found via
the rpath); the tensor-map encoder is fetched from the driver at run time, so
nothing links against libcuda.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")
# The debug variant: every gathered or scattered index range-checked, the GEMM
# tile scheduler's offsets checked (-DMOE_DEBUG_CHECKS); its own objects and library.
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmoe_gb300_debug.so")
SOURCES = ["api.cu", "route.cu", "permute.cu", "front.cu", "gather.cu", "ep.cu", "fp8.cu",
           "grouped_gemm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, *extra]


def _stale(src: str, obj: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src, os.path.join(INCLUDE, "moe_gb300.h")]
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    return any(os.path.getmtime(p) > t for p in deps)


def _flags_digest(cc: str, flags) -> str:
    """The compiler and flags the objects were built with: a change of either
    rebuilds every object (objects built with other flags are never reused)."""
    import hashlib
    return hashlib.sha256(("\0".join([cc, *flags])).encode()).hexdigest()


def build(verbose: bool = False, force: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Builds the library (or, with debug=True, the debug-checks variant) and
    returns its path; objects are rebuilt when a source, the shared header or the
    compiler flags changed."""
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = _flags(tuple(extra_flags) + (("-DMOE_DEBUG_CHECKS",) if debug else ()))
    stamp = os.path.join(bdir, "flags.sha256")
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    digest = _flags_digest(cc, flags)
    try:
        with open(stamp) as f:
            force = force or f.read().strip() != digest
    except OSError:
        force = True
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(bdir, s.replace(".cu", ".o"))
        if force or _stale(src, obj):
            jobs.append([cc, *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(lib):
        run([cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
             "-o", lib, *objs])
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
