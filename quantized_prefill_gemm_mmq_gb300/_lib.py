"""Loader for the in-tree C-ABI library libmmq.so (ctypes).

The library is the whole compute path; there is no fallback.  If it is
missing or fails to load, every op raises instead of computing anything
another way.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmmq.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mmq.h")

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64

# name -> (restype, argtypes); mirrors include/mmq.h
SIGNATURES = {
    "mmq_version": (_I, []),
    "mmq_status_str": (ctypes.c_char_p, [_I]),
    "mmq_quantize_q8_1": (_I, [_P, _I64, _I, _I, _P, _P, _P, _P, _P]),
    "mmq_gemm_q4K": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q4K_subblock": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_splitk_sizes": (_I, [_I, _I, _I, _I, _P, _P]),
    "mmq_gemm_q4K_small_imma": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q4K_small": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemv_q4K": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemv_q6K": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemv_q4K_f32": (_I, [_P, _P, _I64, _P, _I, _I, _I, _P]),
    "mmq_gemv_q6K_f32": (_I, [_P, _P, _I64, _P, _I, _I, _I, _P]),
    "mmq_gemm_q4K_splitk": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "mmq_gemm_q4K_splitk_static": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "mmq_gemm_q4K_swiglu": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q6K": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q5K": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q5K_subblock": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q8_0": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_debug_subdots_q5K": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "mmq_debug_subdots_q8_0": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "mmq_gemm_q6K_subblock": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "mmq_debug_subdots_q4K": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "mmq_debug_subdots_q6K": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "mmq_check_status": (_I, [_P, _P]),
    "mmq_last_failure_info": (_I, [_P]),
    "mmq_debug_fault_inject": (_I, [_I, _I]),
    "mmq_probe_tensor_peak": (_I, [_I, _P, _P]),
}

_lib = None


class MMQError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {status} ({status_str(status)})")


def load():
    """Load libmmq.so (building it first only if explicitly allowed by MMQ_AUTOBUILD=1)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if os.environ.get("MMQ_AUTOBUILD") == "1":
            from . import build
            build.build()
        else:
            raise ImportError(f"libmmq.so is not built ({LIB_PATH}); run `python -c \"import __graft_entry__ as g; "
                              f"g.build()\"` or quantized_prefill_gemm_mmq_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    try:
        return load().mmq_status_str(status).decode()
    except Exception:  # pragma: no cover - used only while formatting errors
        return "?"


def header_functions() -> list[str]:
    """Names of the functions declared in include/mmq.h."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mmq_[A-Za-z0-9_]+)\s*\(", text)))
