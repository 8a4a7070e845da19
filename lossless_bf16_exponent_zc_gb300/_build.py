"""Builds libzc.so in-tree for sm_103a with nvcc (one process per translation unit)."""
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
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libzc.so")
# AddressSanitizer + UndefinedBehaviorSanitizer build of the host code (device
# code is unchanged), for running the CPU-side tests under the sanitizers.
SAN_BUILD = os.path.join(BUILD, "san")
SAN_LIB = os.path.join(LIBDIR, "libzc_san.so")
SAN_FLAGS = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer", "-g"]
SOURCES = ["zc_api.cu", "zc_encode.cu", "zc_decode.cu", "zc_reduce.cu", "zc_hist.cu", "zc_noalloc.cu", "zc_pipeline.cu", "zq.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libzc needs the CUDA toolkit to build")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "zc.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, extra: list[str], outdir: str = BUILD) -> str:
    obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, sanitize: bool = False) -> str:
    """Compile every translation unit in parallel and link libzc.so; skip if up to date.

    sanitize=True builds libzc_san.so instead: the same library with its host
    code instrumented by AddressSanitizer and UndefinedBehaviorSanitizer.  A
    process that loads it must load the ASan runtime first (LD_PRELOAD)."""
    lib, outdir = (SAN_LIB, SAN_BUILD) if sanitize else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(outdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    host = [f for flag in SAN_FLAGS for f in ("-Xcompiler", flag)] if sanitize else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra + host, outdir), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + host + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, sanitize="--sanitize" in sys.argv))
