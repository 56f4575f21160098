"""Compiles libswe (the CUDA kernels and the C ABI of include/swe.h) in-tree
with nvcc for sm_103a: ``finite_volume_shallow_gb300/_build/libswe.so``.

Every translation unit is compiled in parallel, then linked into one shared
library.  Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libswe.so")
SOURCES = ["swe_api.cu", "swe_cart1.cu", "swe_cart2.cu", "swe_mesh.cu", "swe_mesh_prep.cpp",
           "swe_noalloc.cu", "swe_probe.cu", "swe_wetdry.cu"]
HEADERS = [os.path.join(CSRC, "swe_internal.h"), os.path.join(CSRC, "swe_roe2.cuh"),
           os.path.join(CSRC, "swe_fastmath.cuh"), os.path.join(CSRC, "swe_plan.h"),
           os.path.join(ROOT, "include", "swe.h"), os.path.join(ROOT, "include", "swe_probe.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-ftz=true",
                     "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libswe")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Build libswe.so if needed and return its path."""
    if not force and not ptxas_info and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_info else [])
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    errors = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode):
            print(out, file=sys.stderr)
        if p.returncode:
            errors.append(" ".join(cmd))
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
