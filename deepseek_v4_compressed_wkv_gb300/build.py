"""Builds the compressor's CUDA library (libcsa.so) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file in
csrc/_build/, then linked into csrc/_build/libcsa.so.  Nothing is installed.

build(variant="bounds") builds the bounds-checked library instead (csrc/_build_bounds/,
-DCSA_DEBUG_BOUNDS): every kernel store with a computed index is checked against its buffer's
extent, skipped if outside and reported through the handle's device flag (bit 8).  The tests
run the parity cases against it; the binding loads it when CSA_LIBRARY_VARIANT=bounds.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(CSRC, "_build")
LIB = os.path.join(BUILD, "libcsa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libcsa.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, "csa.h")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def lib_path(variant: str = "") -> str:
    """Path of the library of a variant: "" (the product) or "bounds" (bounds-checked)."""
    return LIB if not variant else os.path.join(CSRC, "_build_" + variant, "libcsa.so")


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, variant: str = "") -> str:
    if variant not in ("", "bounds"):
        raise ValueError(f"unknown variant {variant!r}")
    bdir = os.path.dirname(lib_path(variant))
    lib = lib_path(variant)
    extra = ["-DCSA_DEBUG_BOUNDS"] if variant == "bounds" else []
    os.makedirs(bdir, exist_ok=True)
    srcs = sources()
    hdrs = headers()
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    nv = nvcc()

    def compile_one(src, obj):
        if not force and not _stale(obj, [src] + hdrs + [__file__]):
            return None
        cmd = [nv, *ARCH, *FLAGS, *extra, *(["-Xptxas", "-v"] if ptxas_info else []), "-c", src, "-o",
               obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr if (verbose or ptxas_info) else None

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        for out in ex.map(lambda so: compile_one(*so), zip(srcs, objs)):
            if out:
                sys.stderr.write(out)
    if force or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nv, *ARCH, "-shared", "-o", tmp, *objs, "-lcuda"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "bounds" if "--bounds" in sys.argv else ""
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv, variant=v))
