"""Builds libspecdec.so in-tree with nvcc for sm_103a.

    python -m speculative_decoding_rejection_decode_gb300.build
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libspecdec.so")
SOURCES = ["specdec.cu", "noalloc.cu", "tree.cu"]
HEADERS = ["device_common.cuh", "kernels.cuh", "tree.cuh"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths.append(os.path.join(ROOT, "include", "specdec.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tag = f".tmp{os.getpid()}"
    flags = [ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
             "-I", os.path.join(ROOT, "include")]
    if verbose:
        flags.insert(0, "-Xptxas=-v")
    # one object per translation unit, compiled side by side, then one link
    objs = [os.path.join(CSRC, f + tag + ".o") for f in SOURCES]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc] + flags + ["-c", "-o", obj, os.path.join(CSRC, src)]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append(subprocess.Popen(cmd))
    failed = [p.wait() for p in procs]
    try:
        if any(failed):
            raise subprocess.CalledProcessError(max(failed), "nvcc")
        tmp = LIB + tag
        subprocess.run([nvcc, ARCH, "-shared", "-o", tmp] + objs, check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
