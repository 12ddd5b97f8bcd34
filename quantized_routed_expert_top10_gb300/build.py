"""Builds libstrata_moe.so in-tree: every .cu of csrc/ compiled for sm_103a in parallel, then linked."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libstrata_moe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def compile_objects(nvcc: str = "nvcc", extra=None, verbose_ptxas: bool = False):
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *(extra or []), "-c", src, "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        procs.append((src, subprocess.Popen(cmd)))
        objs.append(obj)
    return procs, objs


def build(nvcc: str = "nvcc", extra=None, verbose_ptxas: bool = False) -> str:
    procs, objs = compile_objects(nvcc, extra, verbose_ptxas)
    failed = [src for src, p in procs if p.wait() != 0]
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    if subprocess.call(cmd) != 0:
        raise RuntimeError("link of libstrata_moe.so failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv)
    print(LIB)
