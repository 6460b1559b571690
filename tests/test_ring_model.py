"""The stage ring's protocol, modelled with host threads (no GPU).

tests/ring_model.cpp runs the kernel's ring index arithmetic
(csrc/ring_index.h, the functions the kernel's producer and MMA issuer call)
with threads standing in for the producer, the copy engine, the MMA issuer and
the tensor pipe, over a model of the mbarrier's phases, arrivals and
transaction bytes.  It checks read-after-write and write-after-read order over
600 ring iterations for 1 to 8 stages, single and paired release, and that
injected faults end in a bounded-wait timeout while broken protocols are caught.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ring_protocol_model(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "ring_model"
    build = subprocess.run([cxx, "-std=c++17", "-O2", "-pthread", "-I",
                            os.path.join(ROOT, "warp_specialized_tma_gb300", "csrc"),
                            os.path.join(ROOT, "tests", "ring_model.cpp"), "-o", str(exe)],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.rstrip().endswith("ok"), run.stdout + run.stderr
