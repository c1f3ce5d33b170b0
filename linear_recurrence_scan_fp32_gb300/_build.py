"""Build liblinrec.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu file compiles to an object in parallel; the objects link into one
shared library next to this file.  A stamp of the sources and flags skips the
build when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblinrec.so")
SOURCES = ["linrec_api.cu", "chunked.cu", "chunked16.cu", "backward.cu", "regcarry.cu", "regcarry16.cu", "copy.cu",
           "noalloc.cu", "host_pipeline.cu", "rows.cu", "chain.cu",
           "chunked_fixed.cu", "chunked16_fixed.cu"]
HEADERS = ["kernels.cuh", "ptx.cuh", "lookback.cuh", "chunked_kernel.cuh", "storage.cuh", "checked.cuh"]
# the index-checked build (every plain global access tested against its array first)
CHECKED_BUILD = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(PKG, "liblinrec_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: liblinrec needs the CUDA 13 toolkit to build")


def _stamp(flags) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "linrec.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile every kernel for sm_103a and link liblinrec.so; returns its path.  checked=True
    builds the index-checked library (-DLINREC_DEBUG) as liblinrec_checked.so instead."""
    build_dir, lib = (CHECKED_BUILD, CHECKED_LIB) if checked else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DLINREC_DEBUG"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    stamp_path = os.path.join(build_dir, "stamp")
    stamp = _stamp(flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return lib
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *flags, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
