"""Build libpact.so in-tree for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel with nvcc, then linked into a
shared library next to this file.  The CUDA runtime is linked statically and the
driver's cuTensorMapEncodeTiled is fetched at run time, so the library has no
link-time dependency on libcuda and loads on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpact.so")
# the debug build: every source as one unit (debug_all.cu), stores bounds-checked
DEBUG_LIB = os.path.join(HERE, "libpact_debug.so")
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "lora.cu", "norm_act.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v", "-Wno-deprecated-gpu-targets"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "pact.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build_debug(force: bool = False) -> str:
    """Compile libpact_debug.so (-DPACT_DEBUG, one translation unit) if it is missing or
    older than its sources.  The library's bounds checks then record a failed check
    in the status word (pact_check_status) instead of writing out of bounds."""
    if not force and os.path.exists(DEBUG_LIB) and os.path.getmtime(DEBUG_LIB) >= _deps_mtime():
        return DEBUG_LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    obj = os.path.join(OBJ_DIR, "debug_all.o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-DPACT_DEBUG", "-c", os.path.join(CSRC, "debug_all.cu"),
           "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for the debug build:\n{r.stdout}\n{r.stderr}")
    tmp = DEBUG_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, obj, "-Xcompiler", "-fPIC"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, DEBUG_LIB)
    return DEBUG_LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpact.so if it is missing or older than its sources."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    if "--debug" in sys.argv:
        print(build_debug(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
