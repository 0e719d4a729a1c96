"""Builds libfp4lin.so (the CUDA library) in-tree with nvcc for sm_103a.

Each .cu file compiles to its own object in parallel; the objects link into
one shared library with the CUDA runtime linked statically, so loading the
library needs no CUDA driver until a call touches the GPU.
"""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp4lin.so")
LIB_PEAK = os.path.join(HERE, "libfp4peak.so")
ROOT = os.path.dirname(HERE)
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "gemm_pair.cu", "gemm_noalloc.cu"]
PEAK_SOURCES = ["mma_peak.cu"]
HEADERS = ["ptx.cuh", "formats.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


STAMP = os.path.join(BUILD, "sources.sha256")


def _source_digest() -> str:
    """sha256 over every input of the build (sources, headers, the public
    header, the compiler flags and this machine's architecture): a library is
    reused only when it was built from exactly these inputs here."""
    import platform

    h = hashlib.sha256()
    h.update(" ".join(ARCH + FLAGS).encode())
    h.update(platform.machine().encode())
    files = [os.path.join(CSRC, f) for f in SOURCES + PEAK_SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fp4lin.h")]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _up_to_date(digest: str) -> bool:
    if not all(os.path.exists(f) for f in (LIB, LIB_PEAK)) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as fh:
        return fh.read().strip() == digest


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Builds libfp4lin.so (the library) and libfp4peak.so (the FP4 MMA
    issue-rate probe the benchmark uses), unless both were built here from
    the current sources (a stamp of their hash sits beside the objects)."""
    digest = _source_digest()
    if not force and _up_to_date(digest):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES) + len(PEAK_SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES + PEAK_SOURCES))
    for lib, lib_objs in ((LIB, objs[: len(SOURCES)]), (LIB_PEAK, objs[len(SOURCES):])):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *lib_objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    tmp = STAMP + f".tmp{os.getpid()}"
    with open(tmp, "w") as fh:
        fh.write(digest + "\n")
    os.replace(tmp, STAMP)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
