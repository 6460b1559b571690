"""Host-only checks of the C ABI: the library builds, loads without a GPU and
exports every entry point include/gemm_bf16.h declares; problem validation and
status strings behave as documented.  No kernel runs here."""
from __future__ import annotations

import os
import re

import pytest

from warp_specialized_tma_gb300 import binding
from warp_specialized_tma_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_bf16.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load()


def declared_entry_points():
    text = open(HEADER).read()
    return re.findall(r"GEMM_BF16_API\s+[\w\s\*]+?\b(gemm_bf16_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = set(declared_entry_points())
    for n in ("gemm_bf16_create", "gemm_bf16_plan", "gemm_bf16_run", "gemm_bf16_destroy",
              "gemm_bf16_set_option", "gemm_bf16_device_status", "gemm_bf16_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    # the binding mirrors every entry point under the same name
    for n in names:
        assert hasattr(binding, n), f"binding lacks {n}"


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    syms = {line.split()[-1] for line in out.stdout.splitlines() if line.strip()}
    exported = {s for s in syms if not s.startswith("_")}
    assert exported == set(declared_entry_points())


def test_strerror_and_version(lib):
    assert binding.gemm_bf16_strerror(0) == "ok"
    for st in range(-7, 0):
        s = binding.gemm_bf16_strerror(st)
        assert s and s != "unknown status"
    assert binding.gemm_bf16_strerror(-99) == "unknown status"
    assert "sm_103a" in binding.gemm_bf16_version()


@pytest.mark.parametrize("args,want", [
    ((256, 256, 256, 256, 256, 256), binding.OK),
    ((6143, 5999, 4104, 4104, 4104, 5999), binding.OK),      # odd ldd is allowed (masked epilogue)
    ((1, 1, 1, 8, 8, 1), binding.OK),
    ((0, 4, 8, 8, 8, 4), binding.ERR_INVALID_ARG),
    ((4, 0, 8, 8, 8, 4), binding.ERR_INVALID_ARG),
    ((4, 4, 0, 8, 8, 4), binding.ERR_INVALID_ARG),
    ((-1, 4, 8, 8, 8, 4), binding.ERR_INVALID_ARG),
    ((4, 4, 16, 8, 16, 4), binding.ERR_INVALID_ARG),          # lda < K
    ((4, 4, 16, 16, 8, 4), binding.ERR_INVALID_ARG),          # ldb < K
    ((4, 8, 16, 16, 16, 7), binding.ERR_INVALID_ARG),         # ldd < N
    ((4, 4, 12, 12, 16, 4), binding.ERR_ALIGNMENT),           # lda*2 = 24 bytes
    ((4, 4, 12, 16, 12, 4), binding.ERR_ALIGNMENT),           # ldb*2 = 24 bytes
    ((1 << 31, 4, 8, 8, 8, 4), binding.ERR_INVALID_ARG),      # beyond int32
])
def test_check_problem(lib, args, want):
    assert binding.gemm_bf16_check_problem(*args) == want


def test_null_handle_rejected(lib):
    assert binding.gemm_bf16_plan(None, 8, 8, 8, 8, 8, 8) == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_run(None, 16, 16, 16) == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_set_option(None, 1, 0) == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_device_status(None)[0] == binding.ERR_INVALID_ARG
    assert binding.gemm_bf16_destroy(None) == binding.OK


def test_create_without_a_usable_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = binding.gemm_bf16_create(0)
    assert st in (binding.ERR_CUDA, binding.ERR_UNSUPPORTED)
    assert not h.value


def test_plan_info_struct_matches_the_header():
    # the binding's ctypes mirror of gemm_bf16_plan_info_t: same fields, order and types
    text = open(HEADER).read()
    body = re.search(r"typedef struct gemm_bf16_plan_info_s \{(.*?)\} gemm_bf16_plan_info_t;", text, re.S).group(1)
    fields = re.findall(r"^\s*(int32_t|int64_t)\s+(\w+);", body, re.M)
    ctypes_of = {"int32_t": "c_int", "int64_t": "c_long"}
    got = [(name, t.__name__) for name, t in binding.PlanInfo._fields_]
    assert [n for n, _ in got] == [n for _, n in fields]
    for (name, tname), (ctype, _) in zip(got, fields):
        assert tname in (ctypes_of[ctype], "c_" + ctype.replace("_t", "")), (name, tname, ctype)


def test_option_keys_match_the_header():
    # binding.OPTIONS mirrors gemm_bf16_option: same names (lower case) and values
    text = open(HEADER).read()
    body = re.search(r"typedef enum gemm_bf16_option \{(.*?)\} gemm_bf16_option;", text, re.S).group(1)
    declared = {name.lower(): int(value) for name, value in re.findall(r"GEMM_BF16_OPT_(\w+)\s*=\s*(\d+)", body)}
    assert declared == binding.OPTIONS
