"""Build libpkv.so (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu file compiles in its own nvcc process (in parallel), then one nvcc
call links the shared library. Up-to-date outputs are not rebuilt.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(PKG, "libpkv.so")
SOURCES = ["api.cu", "kv_append.cu", "copy_blocks.cu", "paged_decode.cu", "paged_decode_umma.cu",
           "static_scratch.cu",
           "host_step.cu", "block_manager.cpp", "query_plan.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    return "nvcc"


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, *extra]


def _deps() -> float:
    newest = 0.0
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            newest = max(newest, os.path.getmtime(os.path.join(d, f)))
    return newest


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= _deps():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmds.append([nvcc(), *_flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
        return r.stdout + r.stderr

    with ThreadPoolExecutor(len(cmds)) as ex:
        list(ex.map(run, cmds))
    tmp = LIBRARY + f".tmp{os.getpid()}"
    run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [])
