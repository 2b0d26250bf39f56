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
SOURCES = ["api.cu", "route.cu", "permute.cu", "gather.cu", "ep.cu", "fp8.cu", "grouped_gemm.cu"]
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
    deps = [src, os.path.join(CSRC, "common.cuh"), os.path.join(INCLUDE, "moe_gb300.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def _flags_digest(cc: str, flags) -> str:
    """The compiler and flags the objects were built with: a change of either
    rebuilds every object (objects built with other flags are never reused)."""
    import hashlib
    return hashlib.sha256(("\0".join([cc, *flags])).encode()).hexdigest()


STAMP = os.path.join(BUILD, "flags.sha256")


def build(verbose: bool = False, force: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    digest = _flags_digest(cc, _flags(extra_flags))
    try:
        with open(STAMP) as f:
            force = force or f.read().strip() != digest
    except OSError:
        force = True
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        if force or _stale(src, obj):
            jobs.append([cc, *_flags(extra_flags), "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(LIB):
        run([cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
             "-o", LIB, *objs])
    with open(STAMP, "w") as f:
        f.write(digest + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
