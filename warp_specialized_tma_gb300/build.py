"""Builds libgemm_bf16.so in-tree from csrc/ with nvcc for sm_103a.

The translation units compile in parallel; the CUDA runtime is linked
statically and every symbol except the C ABI of include/gemm_bf16.h is hidden,
so the library loads (and exports its ABI) on a machine without a GPU.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgemm_bf16.so")
BUILD_DIR = os.path.join(PKG, "_build")

SOURCES = ["gemm_bf16_api.cu", "gemm_ws_c1.cu", "gemm_ws_c2.cu", "gemm_nows.cu", "gemm_bf16_noalloc.cu",
           "gemm_repack.cu", "gemm_thin.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm_bf16.so")


def source_digest() -> str:
    """sha256 over every file under csrc/ and include/ (identifies a kernel build)."""
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            path = os.path.join(d, name)
            if os.path.isfile(path):
                h.update(name.encode())
                with open(path, "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()


# What decides the GEMM kernel's behaviour on a given problem: its device code
# and the host planner that picks its launch shape (not the public header's
# documentation, the binding or the other kernels).
KERNEL_FILES = ["gemm_ws.cuh", "gemm_common.cuh", "ptx.cuh", "ring_index.h", "gemm_kernels.h", "gemm_ws_c1.cu",
                "gemm_ws_c2.cu", "gemm_bf16_api.cu"]


def kernel_digest() -> str:
    """sha256 over the files in KERNEL_FILES: identifies a measured kernel."""
    h = hashlib.sha256()
    for name in KERNEL_FILES:
        with open(os.path.join(CSRC, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()


def _stamp_path() -> str:
    return os.path.join(BUILD_DIR, "stamp.txt")


def _nvcc_version(cc: str) -> str:
    try:
        res = subprocess.run([cc, "--version"], capture_output=True, text=True)
        return res.stdout.strip().splitlines()[-1] if res.stdout.strip() else "unknown"
    except OSError:
        return "unknown"


def build_stamp(cc: str | None = None) -> str:
    """What a built library depends on: its sources, the host architecture it
    was linked for, the compiler and the flags.  A library built on another
    machine (an x86_64 build seen on an aarch64 host) never matches."""
    cc = cc or nvcc()
    return "\n".join([source_digest(), "machine=" + platform.machine(), "nvcc=" + _nvcc_version(cc),
                      "flags=" + " ".join(ARCH + FLAGS)])


def up_to_date(cc: str | None = None) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(_stamp_path()):
        return False
    with open(_stamp_path()) as fh:
        return fh.read().strip() == build_stamp(cc)


def build(force: bool = False, verbose: bool = False) -> str:
    cc = nvcc()
    if not force and up_to_date(cc):
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--exclude-libs,ALL", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(_stamp_path(), "w") as fh:
        fh.write(build_stamp(cc))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
