"""Build the CUDA library ``_build/liblin.so`` for sm_103a with nvcc.

Each translation unit under ``csrc/`` compiles in parallel to an object file
(``-gencode arch=compute_103a,code=sm_103a -lineinfo``), then one shared
library is linked with the static CUDA runtime. The driver API is reached at
run time through ``cudaGetDriverEntryPointByVersion``, so the library loads on
a machine without a GPU driver (its calls then return errors).

    python -m transformer_linear_layer_gb300.build [--force] [--verbose] [--timeline]

--timeline builds a second library, ``_build/liblin_timeline.so``, with
-DLIN_TIMELINE: the tcgen05 and skinny kernels then record %globaltimer
stamps that ``lin_timeline`` copies out (a measurement aid; the library
build compiles them out).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liblin.so")
TIMELINE_LIB = os.path.join(BUILD, "liblin_timeline.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ("lin_api.cu", "skinny.cu", "ffma.cu", "tc.cu", "gemv.cu", "backward.cu", "noalloc.cu", "fold.cu", "probe.cu", "attn.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "lin.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, timeline: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library (the
    timeline build with ``timeline=True``)."""
    lib = TIMELINE_LIB if timeline else LIB
    objdir = os.path.join(BUILD, "timeline") if timeline else BUILD
    os.makedirs(objdir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if timeline:
        extra.append("-DLIN_TIMELINE")

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / shared memory")
    ap.add_argument("--timeline", action="store_true", help="build the timeline library instead")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, ptxas_info=args.ptxas_info, timeline=args.timeline))
