"""Build libsot.so in-tree with nvcc for sm_103a (GB300).

Compiles every ``csrc/*.cu`` translation unit in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo`` and links them into
``_build/libsot.so`` (git-ignored).  Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsot.so")
PEAKS_LIB = os.path.join(BUILD, "libsotpeaks.so")
PEAKS_SRC = "peaks.cu"  # throughput probes for the benchmark; not part of libsot
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return p


def _inputs():
    return sorted(f for f in glob.glob(os.path.join(CSRC, "*.cu")) if os.path.basename(f) != PEAKS_SRC), \
        sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
               glob.glob(os.path.join(INCLUDE, "*.h")))


def stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(PEAKS_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(PEAKS_LIB))
    srcs, hdrs = _inputs()
    return any(os.path.getmtime(f) > t for f in srcs + hdrs + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libsot.so; returns its path."""
    if not force and not stale():
        return LIB
    nvcc = nvcc_path()
    objdir = os.path.join(BUILD, "obj")
    os.makedirs(objdir, exist_ok=True)
    srcs, _ = _inputs()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs) + 1, os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs + [os.path.join(CSRC, PEAKS_SRC)]))
    peaks_obj = objs.pop()
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", PEAKS_LIB + ".tmp", peaks_obj], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(PEAKS_LIB + ".tmp", PEAKS_LIB)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
