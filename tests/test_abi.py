"""The C-ABI library builds, loads, and exports every function include/w8a8.h declares.

No compute call is made here (these run without a GPU).
"""

import ctypes
import os
import re

import pytest

from w8a8_int8_quantized_gb300 import build as wbuild
from w8a8_int8_quantized_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(inc, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = re.sub(r"#[^\n]*", "", src)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(([^;{}]*)\)\s*;", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def libpath():
    return wbuild.build()


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ["w8a8_quantize_act", "w8a8_scaled_mm", "w8a8_linear", "w8a8_quantize_weight", "w8a8_azp_adj",
              "fp8block_to_int8_rowwise", "fp8block_to_int8_rowwise_batched", "w8a8_grouped_mm"]:
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in sorted(header_functions()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    assert set(_binding.SIGNATURES) == header_functions()


def test_status_strings_without_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    lib.w8a8_status_string.restype = ctypes.c_char_p
    assert lib.w8a8_status_string(0) == b"ok"
    assert lib.w8a8_status_string(4).startswith(b"illegal")
    assert lib.w8a8_status_string(99) == b"unknown status"


def test_host_side_argument_checks_need_no_gpu(libpath):
    """Argument errors are returned before any CUDA call, so they work on a GPU-less host."""
    lib = _binding.lib()
    # K not a multiple of 16
    assert lib.w8a8_scaled_mm(None, None, 4, 4, 24, 0, None, None, None, 0, None, None, None, None, None, 0, None,
                              None) == 3
    # negative sizes / bad mode
    assert lib.w8a8_quantize_act(None, -1, 4, 4, 0, None, None, None, None) == 1
    assert lib.w8a8_quantize_act(None, 1, 4, 4, 9, None, None, None, None) == 1
    # empty problems are no-ops
    assert lib.w8a8_quantize_act(None, 0, 4, 4, 0, None, None, None, None) == 0
    assert lib.w8a8_scaled_mm(None, None, 0, 4, 16, 0, None, None, None, 0, None, None, None, None, None, 0, None,
                              None) == 0
    # asymmetric GEMM without azp_adj
    p = ctypes.c_void_p(16)
    assert lib.w8a8_scaled_mm(p, p, 4, 4, 16, 1, p, p, None, 0, p, None, None, p, None, 0, None, None) == 1
    # the tensor-core engine needs its staging workspace
    assert lib.w8a8_scaled_mm(p, p, 64, 4, 16, 0, p, None, None, 0, p, None, None, p, None, 0, None, None) == 7
    assert lib.w8a8_scaled_mm_workspace_size(64, 16) == 2048 + 512  # codes, then 2 * 64 int32 row sums
    assert lib.w8a8_act_packed_size(3, 32) == 256 + 256
    # workspace too small
    assert lib.w8a8_linear(p, 4, 16, 16, 0, None, None, p, 4, 0, p, None, None, None, p, p, 8, None, None) == 7
    # weight sums of squares: negative sizes are argument errors, empty weights no-ops
    assert lib.w8a8_weight_sumsq(p, -1, 16, p, None) == 1
    assert lib.w8a8_weight_sumsq(None, 0, 16, None, None) == 0
    assert lib.w8a8_linear_workspace_size(4, 16, 0) == 256 + 256 + 2 * 256
    # K-split scratch: invalid sizes need none (answered before any CUDA call)
    assert lib.w8a8_splitk_workspace_size(0, 4096, 4096) == 0
    assert lib.w8a8_splitk_workspace_size(128, -1, 4096) == 0
    assert lib.w8a8_splitk_workspace_size(128, 4096, 0) == 0
    # max-scale requantization: widths must sum to N, 1 <= P <= 16
    w2 = (ctypes.c_int64 * 2)(3, 4)
    assert lib.w8a8_requantize_max_scale(p, 8, 16, p, ctypes.cast(w2, ctypes.c_void_p), 2, p, None, None) == 1
    assert lib.w8a8_requantize_max_scale(p, 7, 16, p, ctypes.cast(w2, ctypes.c_void_p), 0, p, None, None) == 1
    assert lib.w8a8_requantize_max_scale(p, 7, 16, p, ctypes.cast(w2, ctypes.c_void_p), 17, p, None, None) == 1
    # requantization with row sums: a negative count is an argument error, zero is a no-op
    assert lib.fp8block_to_int8_rowwise_batched_adj(-1, p, p, p, p, p, p, None, None, None) == 1
    assert lib.fp8block_to_int8_rowwise_batched_adj(0, None, None, None, None, None, None, None, None, None) == 0
    assert lib.w8a8_set_gemm_engine(5) == 1
    assert lib.w8a8_set_gemm_engine(0) == 0
    # the release build is not the bounds-checked one
    assert lib.w8a8_debug_build() == 0
    assert lib.w8a8_debug_set_error_word(None) == 2
    # the timeout test hook: values out of range are refused, (0, 0) switches it off
    assert lib.w8a8_test_requant_wait_fault(8192, 0) == 1
    assert lib.w8a8_test_requant_wait_fault(16, 10) == 1
    assert lib.w8a8_test_requant_wait_fault(0, 0) == 0


def test_noalloc_applies_the_scaled_mm_checks(libpath):
    """w8a8_scaled_mm_noalloc rejects exactly what w8a8_scaled_mm rejects, before any CUDA
    call: here an odd bias pointer (bf16 bias must be 2-byte aligned), a missing azp_adj, a K
    that is not a multiple of 16, and then its own limit (staged codes beyond its buffer)."""
    lib = _binding.lib()
    p = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(257)
    f = lib.w8a8_scaled_mm_noalloc
    assert f(p, p, 4, 4, 16, 0, p, None, None, 0, p, odd, p, None, None) == 3
    assert f(p, p, 4, 4, 16, 1, p, p, None, 0, p, None, p, None, None) == 1
    assert f(p, p, 4, 4, 24, 0, p, None, None, 0, p, None, p, None, None) == 3
    g = lib.w8a8_scaled_mm_packed
    assert g(p, p, 4, 4, 16, 0, p, None, None, 0, p, None, odd, p, None, 0, None, None) == 3
    # a split scratch that is not 256-byte aligned
    assert g(p, p, 4, 4, 16, 0, p, None, None, 0, p, None, None, p, odd, 1 << 20, None, None) == 3
    assert f(p, p, 8192, 16, 4096, 0, p, None, None, 0, p, None, p, None, None) == 7
