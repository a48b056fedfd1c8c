"""Builds libtq.so in-tree (``kv_cache_quantization_gb300/lib/libtq.so``) for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked against the shared CUDA
runtime.  No cmake, no setuptools: ``python -m kv_cache_quantization_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libtq.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["host.cpp", "quantize.cu", "quantize_tc.cu", "attention.cu", "scores.cu",
           "decode_tc.cu", "decode_asym.cu", "decode_noalloc.cu", "store.cu", "quality.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtq.so")
    return cand


def _cuda_lib_dir(nvcc):
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        p = os.path.join(root, sub)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    return os.path.join(root, "lib64")


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, "-c", src, "-o", obj, "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I" + INCLUDE] + extra
    if src.endswith(".cu"):
        cmd += ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose: bool = False, extra=None) -> str:
    """Compiles every source and links libtq.so; returns its path."""
    nvcc = _nvcc()
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    extra = list(extra or [])
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    objs = [os.path.join(objdir, s + ".o") for s in srcs]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        futs = [ex.submit(_compile, nvcc, os.path.join(CSRC, s), o, extra)
                for s, o in zip(srcs, objs)]
        logs = [f.result() for f in futs]
    if verbose:
        for s, log in zip(srcs, logs):
            if log.strip():
                print(f"--- {s}\n{log}", file=sys.stderr)
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + [
        "-cudart", "shared", "-Xlinker", "-rpath=" + libdir, "-L" + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(verbose=v or bool(extra), extra=extra))
