"""Build libmxgemm.so and libmxgemm_debug.so in-tree with nvcc for sm_103a.

Seven translation units (host API + relayout/reduce kernels, MXFP8 GEMM,
MXFP4 GEMM, BF16 GEMM, MX quantiser, scale-placement checker, tensor-pipe
probe) are compiled in parallel and linked into
``mx_block_scaled_gb300/lib/libmxgemm.so``.  The four that hold the GEMM
kernels and their host code are compiled a second time with MXGEMM_DEBUG
(bounds-checked loads and stores, NaN-filled C, synchronous status) and linked
with the other three into ``lib/libmxgemm_debug.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libmxgemm.so")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libmxgemm_debug.so")

SOURCES = ["mxgemm.cu", "gemm_fp8.cu", "gemm_fp4.cu", "gemm_bf16.cu", "quantize.cu", "placement.cu", "probe.cu"]
DEBUG_SOURCES = ["mxgemm.cu", "gemm_fp8.cu", "gemm_fp4.cu", "gemm_bf16.cu"]  # the rest is shared
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmxgemm.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "mxgemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(DEBUG_LIB_PATH):
        return True
    t = min(os.path.getmtime(LIB_PATH), os.path.getmtime(DEBUG_LIB_PATH))
    return any(os.path.getmtime(f) > t for f in _deps())


def _link(nvcc: str, objs, path: str) -> None:
    tmp = path + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(path)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libmxgemm.so and libmxgemm_debug.so if either is missing
    or stale; return the release library's path."""
    if not force and not needs_build():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)

    def compile_one(job):
        src, debug = job
        obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + ("_debug.o" if debug else ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *(["-DMXGEMM_DEBUG"] if debug else []), "-c", os.path.join(CSRC, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}{' (debug)' if debug else ''}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    jobs = [(src, False) for src in SOURCES] + [(src, True) for src in DEBUG_SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    release = objs[:len(SOURCES)]
    debug = objs[len(SOURCES):] + [o for (src, _), o in zip(jobs, release) if src not in DEBUG_SOURCES]
    _link(nvcc, release, LIB_PATH)
    _link(nvcc, debug, DEBUG_LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
