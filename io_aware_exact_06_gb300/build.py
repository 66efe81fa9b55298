"""Builds the sm_103a attention library in-tree: _build/libattn_fwd.so.

nvcc compiles the CUDA sources for sm_103a only and links the CUDA runtime
statically, so the library loads on a machine without a GPU (every CUDA call
then fails cleanly) and needs no libcuda at link time (the TMA descriptor
encoder is looked up through the runtime's driver entry-point query).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_fwd.so")
SOURCES = [os.path.join(CSRC, "attn_fwd.cu"), os.path.join(CSRC, "attn_bwd.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _deps():
    deps = list(SOURCES)
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return deps


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in _deps()):
            return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    # one translation unit per source, compiled in parallel, then one link
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, os.path.basename(src) + tag + ".o")
        cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, pr in procs if pr.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIB + tag
        subprocess.run([nvcc(), *ARCH, "-shared", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
