"""Build libcbt.so (the engine's CUDA kernels and C ABI) in-tree for sm_103a.

Each .cu translation unit is compiled in parallel with nvcc, then linked into a shared
library under ``_build/``.  Nothing is installed outside the source tree.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcbt.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: a row's result must not depend on how many rows share the step, and the
# kernels are instantiated per operand width; left free, the compiler contracts a*b + c into
# a fused multiply-add differently in different instantiations (seen: the hi/lo split of an
# epilogue's output), so every fused multiply-add in the sources is an explicit fmaf.
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, "cbt.h")]


def _mtime(p):
    return os.path.getmtime(p)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    deps = [src] + _headers()
    if os.path.exists(obj) and all(_mtime(d) <= _mtime(obj) for d in deps) and not verbose_ptxas:
        return obj
    cmd = ["nvcc"] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose_ptxas else []) + \
        ["-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        print(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    if os.path.exists(LIB) and all(_mtime(o) <= _mtime(LIB) for o in objs):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["nvcc"] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv))
