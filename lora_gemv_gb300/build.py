"""Builds the CUDA library ``liblora_gemv.so`` in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file.  Sources newer than the library trigger a
rebuild; ``force=True`` always rebuilds.  ``debug=True`` builds the
``LORA_DEBUG`` variant, ``liblora_gemv_debug.so``: the same kernels with
device-side bounds checks on every plan entry they read, counted into the
plan's error word (LORA_PLANERR_BOUNDS) instead of trapping.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblora_gemv.so")
OBJDIR_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "liblora_gemv_debug.so")
SOURCES = ["api.cu", "plan.cu", "shrink.cu", "expand.cu", "bgmv.cu", "decode_fused.cu", "noalloc.cu",
           "tmap.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for c in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build lora_gemv_gb300")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "lora_gemv.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib, objdir = (LIB_DEBUG, OBJDIR_DEBUG) if debug else (LIB, OBJDIR)
    flags = FLAGS + (["-DLORA_DEBUG"] if debug else [])
    if not force and not stale(debug):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
