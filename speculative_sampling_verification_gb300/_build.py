"""In-tree build of libspecverify.so for sm_103a (nvcc, no cmake).

The CUDA translation units compile in parallel, then link into one shared
library next to this file (lib/libspecverify.so). A rebuild happens when any
source is newer than the library.
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libspecverify.so")
SOURCES = ["sv_kernels.cu", "sv_api.cu", "sv_static_scratch.cu", "sv_lmhead.cu"]
# Translation units: (source, extra nvcc flags, object). sv_kernels.cu is
# compiled three times, each unit holding one group of its kernels (SV_TU).
UNITS = [("sv_kernels.cu", ["-DSV_TU=1"], "sv_kernels_verify.o"),
         ("sv_kernels.cu", ["-DSV_TU=2"], "sv_kernels_filters.o"),
         ("sv_kernels.cu", ["-DSV_TU=3"], "sv_kernels_topp.o"),
         ("sv_api.cu", [], "sv_api.o"),
         ("sv_static_scratch.cu", [], "sv_static_scratch.o"),
         ("sv_lmhead.cu", [], "sv_lmhead.o")]
HEADERS = ["sv_device.cuh", "sv_internal.h", "sv_exp_table.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-diag-suppress=177",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libspecverify.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    objs, procs = [], []
    for src, extra, name in UNITS:
        obj = os.path.join(LIBDIR, name)
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{out.decode(errors='replace')}")
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd))
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout.decode(errors='replace')}")
    os.replace(tmp, LIB)
    for o in objs:
        os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
