"""Build the sm_103a shared library libw4a16_gb300.so in-tree (nvcc, no cmake).

Each .cu file under csrc/ is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared
library with a plain C ABI (include/w4a16.h).  The output goes to
``w4a16_decode_paged_gb300/_build/``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libw4a16_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


TRACE_BUILD = os.path.join(HERE, "_build_trace")
TRACE_LIB = os.path.join(TRACE_BUILD, "libw4a16_gb300_trace.so")


def build_trace(force: bool = False) -> str:
    """Kernel-timeline build (-DW4A16_TRACE): a separate library that adds
    w4a16_trace_start / w4a16_trace_count; the product library is untouched."""
    # separately compiled device functions must fit the register budget of
    # the kernels that call them (the persistent kernel runs 512 threads)
    return build(force=force, extra_flags=["-DW4A16_TRACE", "-rdc=true", "-maxrregcount=128"], out=TRACE_LIB)


def build(force: bool = False, verbose: bool = False, extra_flags=None, out: str = None) -> str:
    lib = out or LIB
    bdir = os.path.dirname(lib)
    if not force and os.path.exists(lib) and all(os.path.getmtime(p) <= os.path.getmtime(lib) for p in _deps()):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    rdc = ["-rdc=true"] if "-rdc=true" in flags else []
    cmd = [cc, *ARCH, *rdc, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra_flags=extra))
