"""Build libll.so (the C-ABI library) in-tree for sm_103a with nvcc.

Usage: ``python -m windowed_sink_attention_ll_b300.build_lib [--force]``.
Objects go to ``_build/`` at the repository root; the library is written next
to this file so the Python binding finds it.  cudart is linked statically and
the driver's tensor-map encoder is looked up at run time, so the library loads
on a machine without a GPU driver (every compute call then fails cleanly).
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libll.so")
SOURCES = ["ll_host.cu", "ll_copy_frames.cu", "ll_attend_simt.cu", "ll_attend_tc.cu", "ll_attend_pair.cu",
           "ll_noalloc.cu"]
HEADERS = [os.path.join(CSRC, "ll_internal.h"), os.path.join(CSRC, "ll_tc_common.cuh"),
           os.path.join(ROOT, "include", "ll.h")]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-cudart", "static",
         "-I" + os.path.join(ROOT, "include")]


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    newest_header = max(_mtime(h) for h in HEADERS)
    objs = []
    relinked = force or not os.path.exists(LIB)
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _mtime(o) < max(_mtime(s), newest_header, _mtime(__file__)):
            cmd = [NVCC] + FLAGS + ["-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.run(cmd, check=True)
            relinked = True
    if relinked or _mtime(LIB) < max(_mtime(o) for o in objs):
        cmd = [NVCC, "-shared", "-cudart", "static", "-o", LIB] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
