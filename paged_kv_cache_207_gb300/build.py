"""Build the CUDA library ``libpaged_kv.so`` in-tree with nvcc for sm_103a.

Translation units compile in parallel into ``_build/`` at the repository root
and link into ``paged_kv_cache_207_gb300/libpaged_kv.so`` (the CUDA runtime is
linked statically).  Run ``python -m paged_kv_cache_207_gb300.build``.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpaged_kv.so")

SOURCES = ["pa_api.cu", "pa_decode.cu", "pa_append.cu", "pa_prefill.cu", "pa_noalloc.cu",
           "pa_block_manager.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpaged_kv.so")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, ptxas_verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [_nvcc(), "-c", src, "-o", obj, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC] + ARCH
    # optional extra flags, e.g. -DPA_DECODE_WARPS=8 -DPA_DECODE_STAGES=2 for tuning builds
    cmd += os.environ.get("PA_EXTRA_NVCC_FLAGS", "").split()
    if src.endswith(".cu"):
        cmd += ["--expt-relaxed-constexpr"]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if ptxas_verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not ptxas_verbose and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, ptxas_verbose), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose))
