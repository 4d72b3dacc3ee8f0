"""In-tree build of libhs.so (the C ABI of include/hs.h) for sm_103a with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into a shared
library next to this file. Nothing is installed into site-packages.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhs.so")
SOURCES = ["hs_api.cu", "hs_kernels.cu", "hs_noalloc.cu", "hs_consume.cu", "hs_attend.cu", "hs_pool.cu"]
HEADERS = [os.path.join(CSRC, "hs_internal.h"), os.path.join(ROOT, "include", "hs.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libhs.so if any source or header changed; returns its path."""
    os.makedirs(OBJDIR, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(OBJDIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [sp] + HEADERS):
            log = obj + ".log"
            cmd = [nvcc()] + ARCH + NVCC_FLAGS + ["-c", sp, "-o", obj]
            procs.append((cmd, log, subprocess.Popen(cmd, stdout=open(log, "w"), stderr=subprocess.STDOUT)))
    for cmd, log, p in procs:
        rc = p.wait()
        text = open(log).read()
        if verbose or rc != 0:
            sys.stderr.write(text)
        if rc != 0:
            raise RuntimeError(f"nvcc failed ({rc}): {' '.join(cmd)}\n{text}")
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
