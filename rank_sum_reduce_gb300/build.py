"""Build libcar.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to its own object in parallel, then one nvcc call
links the shared library.  The CUDA runtime is linked statically, so the
library loads without a GPU (the driver is only needed when a call runs).
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libcar.so")

SOURCES = ["api.cu", "reduce.cu", "fused.cu", "fused_tma.cu", "ll128.cu", "ll.cu", "ll128_noalloc.cu", "lamport.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libcar")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "car.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    """Compile and link; returns the path of libcar.so."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        log = open(os.path.join(BUILD_DIR, src + ".log"), "w")
        procs.append((src, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    failed = []
    for src, obj, log, p in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD_DIR, src + ".log")) as f:
                msgs.append(f"--- {src} ---\n{f.read()}")
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o, _, _ in procs]]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB_PATH)
    if not quiet or verbose_ptxas:
        for src in SOURCES:
            with open(os.path.join(BUILD_DIR, src + ".log")) as f:
                out = f.read()
            if out.strip():
                sys.stdout.write(f"--- {src} ---\n{out}")
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False)
    print(LIB_PATH)
