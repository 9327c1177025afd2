"""Builds the engine's shared library (libkvb.so) in-tree for sm_103a.

The translation units (host engine, kernels, allocation-free backup,
descriptor ring and its resident server kernel, L3 record store) compile in parallel with nvcc, then link
into ``lib/libkvb.so`` with the CUDA runtime linked statically, so the library
loads on a machine without a GPU and exports the C ABI of ``include/kvb.h``.
``-Xptxas -v`` output of each ``.cu`` file goes to
``_build/<file>.ptxas.log`` (registers, spills, shared memory).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libkvb.so")

SOURCES = ["kvb_api.cpp", "kvb_kernels.cu", "kvb_noalloc.cu", "kvb_ring.cpp", "kvb_ring_kernels.cu",
           "kvb_l3.cpp"]
HEADERS = [os.path.join(CSRC, "kvb_internal.h"), os.path.join(CSRC, "kvb_ring_internal.h"),
           os.path.join(INCLUDE, "kvb.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libkvb.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(LIB, srcs + HEADERS + [__file__]):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    procs, objs = [], []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        log = None
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
            log = open(os.path.join(BUILD, os.path.basename(src) + ".ptxas.log"), "w")
        procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                       text=True), cmd, log))
        objs.append(obj)
    failed = []
    for p, cmd, log in procs:
        out, _ = p.communicate()
        if log is not None:
            log.write(out)
            log.close()
        if verbose and out:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError(f"libkvb.so build failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
