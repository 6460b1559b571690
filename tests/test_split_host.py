"""The kernel's stream-K work split and tile order, checked on the CPU.

tests/split_check.cu includes the kernel's own header (gemm_common.cuh), whose
work-split and tile-order functions are host functions too, and checks every
layout the planner can produce: each (tile, k-block) computed exactly once, one
owner per split tile, the owner's contributor list equal to the items that
computed the rest of the tile, workspace slots distinct and in range, and no
cluster waiting behind its own contributions.  Needs nvcc, not a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_work_split_and_tile_order(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = tmp_path / "split_check"
    build = subprocess.run(
        [nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
         "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "warp_specialized_tma_gb300", "csrc"),
         os.path.join(ROOT, "tests", "split_check.cu"), "-o", str(exe)],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout + run.stderr


def test_thin_kernel_work_split(tmp_path):
    """The thin kernel's split (csrc/thin_split.h, plain C++): ranges, pieces,
    partial slots and owners, the cluster form's ranges, and the automatic
    cluster size on a model of GB300, checked by tests/thin_split_check.cpp.
    Needs a C++ compiler, not a GPU."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "thin_split_check"
    build = subprocess.run(
        [cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "warp_specialized_tma_gb300", "csrc"),
         os.path.join(ROOT, "tests", "thin_split_check.cpp"), "-o", str(exe)],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout + run.stderr
