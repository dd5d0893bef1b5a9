"""Build libpagedkv.so in-tree with nvcc for sm_103a (B300).

Usage: ``python paged_kv_cache_494_b300/build.py [--force] [--ptxas-verbose]`` (a script path, so the
package itself, which refuses to import without the library, is not imported).
"""
from __future__ import annotations

import argparse
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libpagedkv.so")
SOURCES = [os.path.join(CSRC, "pkv_ops.cu"), os.path.join(CSRC, "pkv_alloc.cpp")]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _inputs():
    files = list(SOURCES)
    for d in (CSRC, INCLUDE):
        files += [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".h", ".hpp", ".cuh"))]
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> str:
    """Compile every CUDA and C++ source of the library into ``libpagedkv.so``; returns its path."""
    if not force and not needs_build():
        return LIB
    cmd = [NVCC, *ARCH, "-lineinfo", "-O3", "--use_fast_math", "-std=c++17", "-shared", "-cudart", "shared",
           "-Xcompiler", "-fPIC,-O3,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           "--expt-relaxed-constexpr", "-o", LIB + ".tmp", *SOURCES]
    if ptxas_verbose:
        cmd.insert(1, "-Xptxas=-v")
    if not quiet:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.ptxas_verbose))
