"""Build libccl.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into
``ring_allreduce_rank_gb300/_build/libccl.so`` (static CUDA runtime, so the
library only needs the driver at run time).  No fast-math and no FMA
contraction: the ring's per-hop rounding must be exactly one IEEE operation
followed by one round to the buffer type.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(BUILD, "libccl.so")
# the bounds-checking debug build: every global access of every kernel is
# checked against the call's buffers (CCL_DEBUG_BOUNDS; device globals shared
# across translation units, hence relocatable device code)
DEBUG_LIB = os.path.join(BUILD, "libccl_debug.so")
DEBUG_FLAGS = ["-DCCL_DEBUG_BOUNDS", "-rdc=true"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false", "-ftz=false",
              "-prec-div=true", "-prec-sqrt=true", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libccl.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(paths: list[str], extra: list[str]) -> str:
    h = hashlib.sha256()
    for p in sorted(paths):
        with open(p, "rb") as f:
            h.update(p.encode() + b"\0" + f.read())
    h.update(" ".join(extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug_bounds: bool = False) -> str:
    """Build libccl.so (or, with debug_bounds, libccl_debug.so) unless the
    sources and flags are unchanged since the last build."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    flags = ARCH + NVCC_FLAGS + (DEBUG_FLAGS if debug_bounds else []) + (["-Xptxas", "-v"] if ptxas_verbose else [])
    lib = DEBUG_LIB if debug_bounds else LIB
    tag = "debug." if debug_bounds else ""
    stamp = os.path.join(BUILD, "libccl.%sstamp" % tag)
    digest = _digest(deps, flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read() == digest:
        return lib
    exe = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.basename(src) + "." + tag + "o")
        cmd = [exe, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), res.stderr))
        if verbose or ptxas_verbose:
            print(res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [exe, *ARCH, *(["-rdc=true"] if debug_bounds else []), "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
