"""ctypes wrapper around the plain C oracle (mmq_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg, never by the library.  Arrays are NumPy;
every function copies its inputs to contiguous buffers of the exact dtype
the C side expects.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f32.restype = ctypes.c_float
        L.orc_f32_to_f16.argtypes = [ctypes.c_float]
        L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_f16_to_f32_array.argtypes = [P, i64, P]
        L.orc_f32_to_f16_array.argtypes = [P, i64, P]
        L.orc_q4K_scale_min.argtypes = [P, i32, P, P]
        L.orc_q4K_quant.argtypes = [P, i32]
        L.orc_q4K_quant.restype = i32
        L.orc_q6K_quant.argtypes = [P, i32]
        L.orc_q6K_quant.restype = i32
        L.orc_q6K_scale.argtypes = [P, i32]
        L.orc_q6K_scale.restype = i32
        L.orc_dequant_q4K.argtypes = [P, i32, i32, P]
        L.orc_dequant_q6K.argtypes = [P, i32, i32, P]
        L.orc_quantize_q8_1.argtypes = [P, i64, i32, i32, P, P]
        L.orc_subdots_q4K.argtypes = [P, P, i32, i32, i32, P]
        L.orc_subdots_q6K.argtypes = [P, P, i32, i32, i32, P]
        L.orc_gemm_q4K.argtypes = [P, P, P, i32, i32, i32, P, i64]
        L.orc_gemm_q6K.argtypes = [P, P, P, i32, i32, i32, P, i64]
        L.orc_gemm_points.argtypes = [i32, P, P, P, i32, i32, P, P, P]
        L.orc_dequant_q8_1.argtypes = [P, P, i32, i32, P]
        L.orc_gemm_mt.argtypes = [i32, P, P, P, i32, i32, i32, P, i64, i32]
        L.orc_max_threads.restype = i32
        L.orc_swiglu.argtypes = [P, P, i64, P]
        L.orc_q5K_quant.argtypes = [P, i32]
        L.orc_q5K_quant.restype = i32
        L.orc_q8_0_quant.argtypes = [P, i32]
        L.orc_q8_0_quant.restype = i32
        L.orc_q8_0_d.argtypes = [P]
        L.orc_q8_0_d.restype = ctypes.c_float
        L.orc_dequant_q5K.argtypes = [P, i32, i32, P]
        L.orc_dequant_q8_0.argtypes = [P, i32, i32, P]
        L.orc_subdots_b32.argtypes = [i32, P, P, i32, i32, i32, P]
        L.orc_version.restype = i32
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# bytes per 256 weights of one row, and the format code of the C side
BYTES_PER_256 = {"q4_K": 144, "q6_K": 210, "q5_K": 176, "q8_0": 8 * 34}
FMT_CODE = {"q4_K": 4, "q6_K": 6, "q5_K": 5, "q8_0": 8}


def _check_w(w: np.ndarray, fmt: str, O: int, K: int) -> np.ndarray:
    bb = BYTES_PER_256[fmt]
    w = _c(w, np.uint8)
    if K % 256 or w.size != O * (K // 256) * bb:
        raise ValueError("weight buffer does not match O, K")
    return w


# ------------------------------------------------------------------ f16 --

def f16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16).ravel()
    out = np.empty(h.size, np.float32)
    lib().orc_f16_to_f32_array(_p(h), h.size, _p(out))
    return out


def f32_to_f16(f) -> np.ndarray:
    f = _c(f, np.float32).ravel()
    out = np.empty(f.size, np.uint16)
    lib().orc_f32_to_f16_array(_p(f), f.size, _p(out))
    return out


# -------------------------------------------------------- block decode --

def q4K_scale_min(s12: np.ndarray, j: int):
    s12 = _c(s12, np.uint8)
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().orc_q4K_scale_min(_p(s12), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def q4K_quants(blk: np.ndarray) -> np.ndarray:
    blk = _c(blk, np.uint8)
    return np.array([lib().orc_q4K_quant(_p(blk), e) for e in range(256)], np.int32)


def q5K_quants(blk: np.ndarray) -> np.ndarray:
    blk = _c(blk, np.uint8)
    return np.array([lib().orc_q5K_quant(_p(blk), e) for e in range(256)], np.int32)


def q8_0_block(blk: np.ndarray):
    """(d, the 32 int8 quants) of one 34-byte q8_0 block."""
    blk = _c(blk, np.uint8)
    return lib().orc_q8_0_d(_p(blk)), np.array([lib().orc_q8_0_quant(_p(blk), i) for i in range(32)], np.int32)


def q6K_quants(blk: np.ndarray) -> np.ndarray:
    blk = _c(blk, np.uint8)
    return np.array([lib().orc_q6K_quant(_p(blk), e) for e in range(256)], np.int32)


def dequant(fmt: str, w: np.ndarray, O: int, K: int) -> np.ndarray:
    w = _check_w(w, fmt, O, K)
    out = np.empty((O, K), np.float64)
    fn = {"q4_K": lib().orc_dequant_q4K, "q6_K": lib().orc_dequant_q6K, "q5_K": lib().orc_dequant_q5K,
          "q8_0": lib().orc_dequant_q8_0}[fmt]
    fn(_p(w), O, K, _p(out))
    return out


# ---------------------------------------------------------------- q8_1 --

def quantize_q8_1(x: np.ndarray):
    """X f32 [T][K] -> (qs int8 [T][K], ds uint32 [T][K/32])."""
    x = _c(x, np.float32)
    T, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    qs = np.empty((T, K), np.int8)
    ds = np.empty((T, K // 32), np.uint32)
    lib().orc_quantize_q8_1(_p(x), K, T, K, _p(qs), _p(ds))
    return qs, ds


def dequant_q8_1(qs: np.ndarray, ds: np.ndarray) -> np.ndarray:
    qs = _c(qs, np.int8)
    ds = _c(ds, np.uint32)
    T, K = qs.shape
    out = np.empty((T, K), np.float64)
    lib().orc_dequant_q8_1(_p(qs), _p(ds), T, K, _p(out))
    return out


# ---------------------------------------------------------------- GEMM --

def subdots(fmt: str, w: np.ndarray, qs: np.ndarray, O: int) -> np.ndarray:
    """Per-sub-block int32 dots: [T][O][K/32] (q4_K, q5_K, q8_0) or [T][O][K/16] (q6_K)."""
    qs = _c(qs, np.int8)
    T, K = qs.shape
    w = _check_w(w, fmt, O, K)
    if fmt in ("q5_K", "q8_0"):
        out = np.empty((T, O, K // 32), np.int32)
        lib().orc_subdots_b32(FMT_CODE[fmt], _p(w), _p(qs), T, O, K, _p(out))
    elif fmt == "q4_K":
        out = np.empty((T, O, K // 32), np.int32)
        lib().orc_subdots_q4K(_p(w), _p(qs), T, O, K, _p(out))
    else:
        out = np.empty((T, O, K // 16), np.int32)
        lib().orc_subdots_q6K(_p(w), _p(qs), T, O, K, _p(out))
    return out


def gemm(fmt: str, w: np.ndarray, qs: np.ndarray, ds: np.ndarray, O: int, threads: int | None = None) -> np.ndarray:
    """Method-form Y [T][O] f32.  threads=1: the single-thread loop; otherwise the
    output columns are divided among `threads` OpenMP threads (None: every core
    the process may use).  The result is the same bit for bit either way."""
    qs = _c(qs, np.int8)
    ds = _c(ds, np.uint32)
    T, K = qs.shape
    w = _check_w(w, fmt, O, K)
    y = np.empty((T, O), np.float32)
    if threads == 1 and fmt in ("q4_K", "q6_K"):
        fn = lib().orc_gemm_q4K if fmt == "q4_K" else lib().orc_gemm_q6K
        fn(_p(w), _p(qs), _p(ds), T, O, K, _p(y), O)
    else:
        lib().orc_gemm_mt(FMT_CODE[fmt], _p(w), _p(qs), _p(ds), T, O, K, _p(y), O,
                          0 if threads is None else int(threads))
    return y


def max_threads() -> int:
    """Threads the multi-threaded oracle uses by default."""
    return lib().orc_max_threads()


def gemm_points(fmt: str, w: np.ndarray, qs: np.ndarray, ds: np.ndarray, O: int,
                ti: np.ndarray, oi: np.ndarray) -> np.ndarray:
    """Method-form Y[ti[i]][oi[i]] for selected output positions."""
    qs = _c(qs, np.int8)
    ds = _c(ds, np.uint32)
    T, K = qs.shape
    w = _check_w(w, fmt, O, K)
    ti = _c(ti, np.int32)
    oi = _c(oi, np.int32)
    if ti.shape != oi.shape or (ti.size and (ti.min() < 0 or ti.max() >= T or oi.min() < 0 or oi.max() >= O)):
        raise ValueError("bad output positions")
    out = np.empty(ti.size, np.float32)
    lib().orc_gemm_points(6 if fmt == "q6_K" else 4, _p(w), _p(qs), _p(ds), K, ti.size,
                          _p(ti), _p(oi), _p(out))
    return out


def gemm_dequant(fmt: str, w: np.ndarray, qs: np.ndarray, ds: np.ndarray, O: int) -> np.ndarray:
    """Full-dequant form: f64 product of dequant(W) and dequant(q8_1(X))."""
    T, K = np.asarray(qs).shape
    return dequant_q8_1(qs, ds) @ dequant(fmt, w, O, K).T


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u elementwise in f32 (reading R14), same shape as g."""
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    if g.shape != u.shape:
        raise ValueError("g and u must have the same shape")
    h = np.empty(g.shape, np.float32)
    lib().orc_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def version() -> int:
    return lib().orc_version()


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "ctypes", "os", "np")]
