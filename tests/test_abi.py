"""CPU-side checks of the C-ABI library: it loads, exports exactly what
include/mmq.h declares, and rejects bad arguments before touching a GPU."""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

from quantized_prefill_gemm_mmq_gb300 import _lib

HAVE_LIB = os.path.exists(_lib.LIB_PATH)
needs_lib = pytest.mark.skipif(not HAVE_LIB, reason="libmmq.so not built (run __graft_entry__.build())")


def test_header_declares_the_boundary():
    names = _lib.header_functions()
    for required in ("mmq_quantize_q8_1", "mmq_gemm_q4K", "mmq_gemm_q4K_subblock", "mmq_gemm_q6K", "mmq_check_status",
                     "mmq_status_str", "mmq_version", "mmq_debug_subdots_q4K", "mmq_debug_subdots_q6K",
                     "mmq_gemm_q4K_splitk", "mmq_splitk_sizes", "mmq_gemm_q4K_splitk_static",
                     "mmq_gemm_q6K_subblock", "mmq_gemm_q4K_small", "mmq_gemm_q4K_small_imma",
                     "mmq_last_failure_info", "mmq_gemv_q4K", "mmq_gemv_q6K", "mmq_gemm_q4K_swiglu",
                     "mmq_gemm_q5K", "mmq_gemm_q5K_subblock", "mmq_gemm_q8_0", "mmq_debug_subdots_q5K",
                     "mmq_debug_subdots_q8_0", "mmq_debug_fault_inject", "mmq_gemv_q4K_f32",
                     "mmq_gemv_q6K_f32"):
        assert required in names
    assert set(names) == set(_lib.SIGNATURES), "binding signatures and header out of sync"


@needs_lib
def test_library_exports_every_header_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _lib.header_functions():
        assert name in exported, name


@needs_lib
def test_library_loads_and_reports():
    lib = _lib.load()
    assert lib.mmq_version() == 8
    assert lib.mmq_status_str(0) == b"ok"
    for code in range(-10, 0):
        assert lib.mmq_status_str(code) not in (b"", b"unknown status")


@needs_lib
def test_argument_errors_without_gpu():
    lib = _lib.load()
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 15) & ~15
    p = ctypes.c_void_p(base)
    odd = ctypes.c_void_p(base + 4)
    null = ctypes.c_void_p(0)
    # shapes
    assert lib.mmq_quantize_q8_1(p, 64, 1, 48, p, p, p, p, null) == -1           # K % 32
    assert lib.mmq_quantize_q8_1(p, 16, 1, 32, p, p, p, p, null) == -1           # ldx < K
    assert lib.mmq_gemm_q4K(p, p, p, p, 1, 1, 300, null) == -1               # K % 256
    assert lib.mmq_gemm_q6K(p, p, p, p, 1, 0, 256, null) == -1               # O < 1
    assert lib.mmq_gemm_q6K_subblock(p, p, p, p, 1, 1, 300, null) == -1      # K % 256
    assert lib.mmq_gemm_q6K(p, p, null, p, 0, 1, 256, null) == 0             # ds unused; T == 0 no-op
    assert lib.mmq_gemm_q4K_small_imma(p, p, p, p, 17, 8, 256, null) == -1   # T > 16
    assert lib.mmq_gemm_q4K_small_imma(p, p, null, p, 16, 8, 256, null) == -6
    assert lib.mmq_gemm_q4K_small(p, p, p, p, 65, 8, 256, null) == -1        # T > 64
    assert lib.mmq_gemm_q4K_small(p, p, p, p, 64, 8, 300, null) == -1        # K % 256
    assert lib.mmq_gemm_q4K_small(p, p, null, p, 64, 8, 256, null) == -6
    assert lib.mmq_gemm_q4K_small(p, odd, p, p, 64, 8, 256, null) == -2
    assert lib.mmq_gemm_q4K_small(p, p, p, p, 0, 8, 256, null) == 0          # T == 0 no-op
    for gemv in (lib.mmq_gemv_q4K, lib.mmq_gemv_q6K):                         # decode-shaped products
        assert gemv(p, p, p, p, 17, 8, 256, null) == -1                       # T > 16
        assert gemv(p, p, p, p, 16, 8, 300, null) == -1                       # K % 256
        assert gemv(p, p, p, p, 16, 0, 256, null) == -1                       # O < 1
        assert gemv(p, p, p, p, 16, 8, 1 << 21, null) == -1                   # K > 2^20
        assert gemv(p, p, null, p, 16, 8, 256, null) == -6
        assert gemv(p, odd, p, p, 16, 8, 256, null) == -2
        assert gemv(p, p, p, p, 0, 8, 256, null) == 0                         # T == 0 no-op
    for dec in (lib.mmq_gemv_q4K_f32, lib.mmq_gemv_q6K_f32):                 # decode with built-in q8_1
        assert dec(p, p, 256, p, 5, 8, 256, null) == -1                       # T > 4
        assert dec(p, p, 300, p, 1, 8, 300, null) == -1                       # K % 256
        assert dec(p, p, 65536, p, 1, 8, 65536, null) == -1                   # K > 32768
        assert dec(p, p, 256, p, 1, 0, 256, null) == -1                       # O < 1
        assert dec(p, p, 252, p, 1, 8, 256, null) == -1                       # ldx < K
        assert dec(null, p, 256, p, 1, 8, 256, null) == -6
        assert dec(p, p, 256, null, 1, 8, 256, null) == -6
        assert dec(p, odd, 256, p, 1, 8, 256, null) == -2
        assert dec(p, p, 258, p, 1, 8, 256, null) == -2                       # ldx % 4
        assert dec(p, p, 256, p, 0, 8, 256, null) == 0                        # T == 0 no-op
    assert lib.mmq_last_failure_info(null) == -6
    assert lib.mmq_debug_fault_inject(2, 1000) == -1                         # unknown mode
    info = (ctypes.c_int * 4)(7, 7, 7, 7)
    assert lib.mmq_last_failure_info(info) == 0 and list(info) == [0, 0, 0, 0]   # nothing reported yet
    assert lib.mmq_gemm_q4K(p, p, p, p, -1, 1, 256, null) == -1              # T < 0
    # T == 0 is a no-op
    assert lib.mmq_gemm_q4K(p, p, p, p, 0, 1, 256, null) == 0
    assert lib.mmq_quantize_q8_1(p, 32, 0, 32, p, p, p, p, null) == 0
    # nulls and alignment
    assert lib.mmq_gemm_q4K(null, p, p, p, 1, 1, 256, null) == -6
    assert lib.mmq_quantize_q8_1(p, 32, 1, 32, null, p, null, null, null) == -6   # no value plane
    assert lib.mmq_gemm_q4K(odd, p, p, p, 1, 1, 256, null) == -2
    assert lib.mmq_quantize_q8_1(p, 34, 1, 32, p, p, p, p, null) == -2          # ldx * 4 not 16-aligned
    # split-K: workspace required when splitting, ksplit >= 1
    assert lib.mmq_gemm_q4K_splitk(p, p, p, p, 16, 256, 1024, 4, null, p, null) == -6
    assert lib.mmq_gemm_q4K_splitk(p, p, p, p, 16, 256, 1024, 4, p, null, null) == -6
    assert lib.mmq_gemm_q4K_splitk(p, p, p, p, 16, 256, 1024, 0, p, p, null) == -1
    assert lib.mmq_gemm_q4K_splitk(p, p, p, p, 16, 256, 1024, 4, odd, p, null) == -2
    # q5_K and q8_0 GEMMs: shapes, nulls, alignment, T == 0
    for fn in (lib.mmq_gemm_q5K, lib.mmq_gemm_q5K_subblock, lib.mmq_gemm_q8_0):
        assert fn(p, p, p, p, 1, 1, 300, null) == -1                            # K % 256
        assert fn(p, p, p, p, 1, 0, 256, null) == -1                            # O < 1
        assert fn(null, p, p, p, 1, 1, 256, null) == -6
        assert fn(odd, p, p, p, 1, 1, 256, null) == -2
        assert fn(p, p, p, p, 0, 1, 256, null) == 0
    for fn in (lib.mmq_debug_subdots_q5K, lib.mmq_debug_subdots_q8_0):
        assert fn(p, p, p, 1, 1, 300, null) == -1
        assert fn(p, p, null, 1, 1, 256, null) == -6
    # fused gate/up + SwiGLU + q8_1: F a multiple of 64, outputs required, alignment
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, p, p, null, 16, 96, 256, null) == -1       # F % 64
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, p, p, null, 16, 0, 256, null) == -1        # F < 64
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, p, p, null, 16, 64, 300, null) == -1       # K % 256
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, null, p, null, 16, 64, 256, null) == -6    # no h_xa
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, p, null, null, 16, 64, 256, null) == -6    # no h_ds
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, odd, p, null, 16, 64, 256, null) == -2
    assert lib.mmq_gemm_q4K_swiglu(p, p, p, p, p, null, 0, 64, 256, null) == 0          # T == 0 no-op
    # static-scratch variant: oversize requests are refused before anything else
    assert lib.mmq_gemm_q4K_splitk_static(p, p, p, p, 4096, 4096, 4096, 4, null) == -9
    assert lib.mmq_gemm_q4K_splitk_static(p, p, p, p, 16, 256, 1024, 0, null) == -1
    # one split needs no scratch: a shape with more output tiles than the static counters
    # (8192 x 16512: 64 x 129 tiles) is not refused for lack of scratch with ksplit == 1
    assert lib.mmq_gemm_q4K_splitk_static(p, p, p, p, 8192, 16512, 4096, 1, null) != -9
    assert lib.mmq_gemm_q4K_splitk_static(p, p, p, p, 8192, 16512, 256, 4, null) != -9   # K = 256: one split


@needs_lib
def test_splitk_sizes():
    lib = _lib.load()
    pf, nc = ctypes.c_int64(), ctypes.c_int64()
    # K = 4096: 16 super-blocks; ksplit 4 -> 4 splits of 4
    assert lib.mmq_splitk_sizes(16, 4096, 4096, 4, ctypes.byref(pf), ctypes.byref(nc)) == 0
    assert (pf.value, nc.value) == (4 * 16 * 4096, 32)
    # K = 11008: 43 super-blocks; ksplit 4 -> 11 per split -> 4 splits
    assert lib.mmq_splitk_sizes(200, 300, 11008, 4, ctypes.byref(pf), ctypes.byref(nc)) == 0
    assert (pf.value, nc.value) == (4 * 200 * 300, 3 * 2)
    # ksplit 5 on 16 super-blocks -> 4 per split -> 4 splits; ksplit 100 -> one per split
    assert lib.mmq_splitk_sizes(1, 128, 4096, 5, ctypes.byref(pf), ctypes.byref(nc)) == 0
    assert pf.value == 4 * 1 * 128
    assert lib.mmq_splitk_sizes(1, 128, 4096, 100, ctypes.byref(pf), ctypes.byref(nc)) == 0
    assert pf.value == 16 * 1 * 128
    # no split: no partial workspace
    assert lib.mmq_splitk_sizes(1, 128, 256, 4, ctypes.byref(pf), ctypes.byref(nc)) == 0
    assert pf.value == 0
    assert lib.mmq_splitk_sizes(1, 128, 4096, 0, ctypes.byref(pf), ctypes.byref(nc)) == -1


@needs_lib
def test_valid_call_without_gpu_fails_loudly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = _lib.load()
    buf = ctypes.create_string_buffer(1 << 16)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    assert lib.mmq_quantize_q8_1(p, 32, 1, 32, p, p, p, p, ctypes.c_void_p(0)) == -3   # no sm_103 device
    assert lib.mmq_gemm_q4K(p, p, p, p, 1, 1, 256, ctypes.c_void_p(0)) == -3
    assert lib.mmq_gemm_q4K_subblock(p, p, p, p, 1, 1, 256, ctypes.c_void_p(0)) == -3
