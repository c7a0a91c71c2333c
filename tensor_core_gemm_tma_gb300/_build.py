"""Builds the in-tree CUDA library libstage_gemm.so for sm_103a with nvcc.

The host API unit and the kernel-instantiation units (sg_inst_*.cu) are
compiled in parallel (one -gencode), then linked into one shared library
that sits next to this file, so the binding loads it from the source tree."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libstage_gemm.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libstage_gemm.so")


def _units():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _sources():
    return sorted(_units() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    nvcc = _nvcc()
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in _units():
        obj = os.path.join(CSRC, os.path.basename(src)[:-3] + tag + ".o")
        cmd = [nvcc, *ARCH_FLAGS, *COMMON, "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"{' '.join(cmd)}\n{out}")
        elif verbose and out:
            print(out)
    try:
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp = LIB + tag
        link = [nvcc, *ARCH_FLAGS, "-shared", *objs, "-o", tmp]
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(link)}\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB
