"""Builds libpic.so in-tree for GB300 (sm_103a) with nvcc.

The translation units (host C++ and the CUDA kernel files) are compiled in parallel and
linked against the shared CUDA runtime, so the process uses one runtime with
PyTorch.  The library is written under a temporary name and renamed into
place, so a concurrent reader never sees a half-written file.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libpic.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

SOURCES = ["pic_host.cpp", "pic_kernels.cu", "pic_kernels_tma.cu", "pic_attention.cu", "pic_attention_tc.cu",
           "pic_noalloc.cu", "pic_cdc.cu", "pic_stage.cu"]
HEADERS = [os.path.join(CSRC, "pic_internal.h"), os.path.join(INCLUDE, "pic.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _cuda_lib_dir() -> str:
    home = os.path.dirname(os.path.dirname(_nvcc()))
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        d = os.path.join(home, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(home, "lib64")


def _sources():
    return [os.path.join(CSRC, s) for s in SOURCES]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _sources() + HEADERS + [__file__])


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)
    return res


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles and links libpic.so next to this file; returns its path."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-std=c++17", "-O3", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC,-O3,-Wall"]
    ptxas_v = ["-Xptxas", "-v"] if os.environ.get("PIC_PTXAS_VERBOSE") else []
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{os.getpid()}.o")
        objs.append(obj)
        if src.endswith(".cu"):
            cmd = [nvcc, "-c", src, "-o", obj, *common, *ARCH, "-lineinfo", *ptxas_v]
        else:
            cmd = [nvcc, "-c", src, "-o", obj, *common]
        jobs.append(cmd)
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda c: _run(c, verbose), jobs))
    if ptxas_v:
        for r in results:
            sys.stdout.write(r.stderr)
    fd, tmp = tempfile.mkstemp(prefix=".libpic.", suffix=".so", dir=PKG_DIR)
    os.close(fd)
    try:
        libdir = _cuda_lib_dir()
        _run([nvcc, "-shared", "-o", tmp, *objs, *ARCH, "-cudart", "shared",
              "-Xlinker", f"-rpath,{libdir}", "-L", libdir], verbose)
        os.replace(tmp, LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
        for o in objs:
            if os.path.exists(o):
                os.unlink(o)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
