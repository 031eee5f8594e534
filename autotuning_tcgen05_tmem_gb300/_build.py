"""Builds the native library in-tree: csrc/*.cu with nvcc for sm_103a,
csrc/*.cpp with g++, linked into _lib/libgemm_gb300.so (static cudart).

The objects of one build are tied to the machine that made them: a stamp
records the CPU architecture and a hash of the sources, and any difference
triggers a rebuild (the library built on an x86 host is never loaded on an
aarch64 host, or the other way round).
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libgemm_gb300.so")
STAMP = os.path.join(LIBDIR, "build.stamp")

CU_SOURCES = ["gemm_kernel.cu", "noalloc.cu"]
CPP_SOURCES = ["planner.cpp", "runtime.cpp", "capi.cpp"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _sources_digest() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    with open(os.path.join(INCLUDE, "gemm_gb300.h"), "rb") as f:
        h.update(f.read())
    with open(__file__, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def _stamp_text() -> str:
    return f"{platform.machine()} {_sources_digest()}\n"


def is_current() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as f:
        return f.read() == _stamp_text()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and is_current():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    inc = os.path.join(home, "include")
    jobs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        jobs.append([nvcc, *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v" if verbose else "-O3", "-I", INCLUDE, "-c",
                     os.path.join(CSRC, src), "-o", obj])
    cxx = os.environ.get("CXX", "g++")
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        jobs.append([cxx, "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", inc, "-I", INCLUDE, "-c",
                     os.path.join(CSRC, src), "-o", obj])
    procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for j in jobs]
    failed = []
    for j, p in zip(jobs, procs):
        out, _ = p.communicate()
        if verbose and out:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append((j, out))
    if failed:
        msg = "\n".join(" ".join(j) + "\n" + out for j, out in failed)
        raise RuntimeError("native build failed:\n" + msg)
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs,
            "-Xlinker", "-z,defs", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("native link failed:\n" + " ".join(link) + "\n" + r.stdout)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_stamp_text())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
