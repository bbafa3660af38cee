"""Builds the CUDA library libpkv.so for sm_103a with nvcc (in-tree, no cmake).

Every translation unit in csrc/ is compiled in parallel to an object file and
the objects are linked into one shared library with the CUDA runtime linked
statically.  Re-running is cheap: objects newer than their sources and the
headers are reused.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _flags():
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr",
                   "-Xptxas", "-warn-spills"]


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(verbose: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = (glob.glob(os.path.join(CSRC, "*.h")) +
               glob.glob(os.path.join(CSRC, "*.cuh")) +
               glob.glob(os.path.join(INCLUDE, "*.h")))
    hdr_time = _newest(headers) if headers else 0.0
    objs = []
    todo = []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if (not os.path.exists(obj) or os.path.getmtime(obj) <
                max(os.path.getmtime(src), hdr_time)):
            todo.append((src, obj))

    def compile_one(pair):
        src, obj = pair
        tmp = obj + f".{os.getpid()}.tmp.o"
        cmd = [NVCC] + _flags() + ["-c", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, obj)
        return src, r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), 8)) as ex:
            for src, err in ex.map(compile_one, todo):
                if verbose and err.strip():
                    print(f"[{os.path.basename(src)}]\n{err}", file=sys.stderr)
    if todo or not os.path.exists(LIB) or os.path.getmtime(LIB) < _newest(objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
