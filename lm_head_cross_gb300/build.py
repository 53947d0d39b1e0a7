"""Builds ``libflce.so`` in-tree with nvcc for sm_103a (no cmake, no torch), and
beside it ``libflce_debug.so``, the same sources compiled with FLCE_DEBUG_CHECKS
(every computed index and TMA coordinate checked before use, failures recorded
in the status word).

    python -m lm_head_cross_gb300.build
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libflce.so")
DEBUG_LIB = os.path.join(HERE, "libflce_debug.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["flce_kernels.cu", "flce_api.cu", "flce_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, verbose_ptxas: bool, debug: bool) -> str:
    out_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
           "-c", os.path.join(CSRC, src), "-o", obj]
    if debug:
        cmd.insert(1, "-DFLCE_DEBUG_CHECKS")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _link(objs, lib):
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    srcs.append(os.path.join(INCLUDE, "flce.h"))
    srcs.append(os.path.abspath(__file__))
    if not force and all(os.path.exists(lib) for lib in (LIB, DEBUG_LIB)):
        lib_m = min(os.path.getmtime(LIB), os.path.getmtime(DEBUG_LIB))
        if all(os.path.getmtime(s) <= lib_m for s in srcs):
            return LIB
    os.makedirs(os.path.join(BUILD_DIR, "debug"), exist_ok=True)
    jobs = [(s, d) for d in (False, True) for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose_ptxas and not j[1], j[1]), jobs))
    _link(objs[:len(SOURCES)], LIB)
    _link(objs[len(SOURCES):], DEBUG_LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
