"""Thin PyTorch binding over libmmq's C ABI (argument marshalling only).

Every function checks device, dtype, shape and contiguity, passes raw device
pointers and the current CUDA stream to the library, and raises MMQError on
a non-zero status.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import MMQError, load

BLOCK_BYTES = {"q4_K": 144, "q6_K": 210, "q5_K": 176, "q8_0": 272}   # bytes per 256 weights of a row


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _check(call: str, status: int):
    if status != 0:
        raise MMQError(call, status)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmmq ops need CUDA tensors")


def quantize_q8_1(x: torch.Tensor, want_qs: bool = True, want_xh: bool = True, want_xa: bool = True, out=None):
    """q8_1-quantise activations x [T][K] f32 (row stride may exceed K).

    Returns (qs, ds, xh, xa):
      qs  int8 [T][K] values, or None;
      ds  int32 [T][K/32] holding the uint32 words (f16 d | int16 block sum);
      xh  float16 [T][K], the same integer values as f16 (per-sub-block operand), or None;
      xa  float16 [2][T][K], the dequantised values f32(d)*q as exact hi + lo planes
          (production operand), or None.
    `out` may supply the four buffers (any of qs / xh / xa may be None).
    """
    _need_cuda(x)
    if x.dtype != torch.float32 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D float32 tensor with unit column stride")
    T, K = x.shape
    dev = x.device
    if out is not None:
        qs, ds, xh, xa = out
        for t, dt, shape in ((qs, torch.int8, (T, K)), (ds, torch.int32, (T, K // 32)),
                             (xh, torch.float16, (T, K)), (xa, torch.float16, (2, T, K))):
            if t is not None and (t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous()):
                raise ValueError("bad output buffer")
        if ds is None:
            raise ValueError("ds buffer required")
    else:
        qs = torch.empty((T, K), dtype=torch.int8, device=dev) if want_qs else None
        xh = torch.empty((T, K), dtype=torch.float16, device=dev) if want_xh else None
        xa = torch.empty((2, T, K), dtype=torch.float16, device=dev) if want_xa else None
        ds = torch.empty((T, K // 32), dtype=torch.int32, device=dev)
    _need_cuda(qs, ds, xh, xa)
    with torch.cuda.device(dev):
        st = load().mmq_quantize_q8_1(_ptr(x), x.stride(0), T, K, _ptr(qs), _ptr(ds), _ptr(xh), _ptr(xa),
                                      _stream(dev))
    _check("mmq_quantize_q8_1", st)
    return qs, ds, xh, xa


def _check_gemm_args(fmt: str, w: torch.Tensor, xv: torch.Tensor, O: int, planes: int):
    _need_cuda(w, xv)
    if fmt not in BLOCK_BYTES:
        raise ValueError(f"unknown format {fmt!r}")
    if xv.dtype != torch.float16 or xv.dim() != (2 if planes == 1 else 3) or not xv.is_contiguous() or \
            (planes == 2 and xv.shape[0] != 2):
        raise ValueError("activation operand must be contiguous float16 [T][K] (xh) or [2][T][K] (xa)")
    T, K = xv.shape[-2:]
    if w.dtype != torch.uint8 or not w.is_contiguous() or w.numel() != O * (K // 256) * BLOCK_BYTES[fmt]:
        raise ValueError("w must be contiguous uint8 holding O*(K/256) super-blocks")
    if w.device != xv.device:
        raise ValueError("w and the activations must be on the same device")
    return T, K


def _out(out, T, O, dev):
    if out is None:
        return torch.empty((T, O), dtype=torch.float32, device=dev)
    if out.dtype != torch.float32 or tuple(out.shape) != (T, O) or not out.is_contiguous():
        raise ValueError("out must be contiguous float32 [T][O]")
    return out


def _check_ds(ds, T, K):
    if ds.dtype != torch.int32 or tuple(ds.shape) != (T, K // 32) or not ds.is_contiguous():
        raise ValueError("ds must be contiguous int32 [T][K/32]")


def gemm(fmt: str, w: torch.Tensor, xa: torch.Tensor, ds: torch.Tensor, O: int,
         out: torch.Tensor | None = None) -> torch.Tensor:
    """Production GEMM: Y [T][O] f32 from W (`fmt`: q4_K, q5_K or q6_K) and the xa/ds
    activation planes (q6_K does not read ds)."""
    T, K = _check_gemm_args(fmt, w, xa, O, planes=2)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xa.device)
    fn = {"q4_K": load().mmq_gemm_q4K, "q6_K": load().mmq_gemm_q6K, "q5_K": load().mmq_gemm_q5K}.get(fmt)
    if fn is None:
        raise ValueError(f"no production GEMM for {fmt!r} (q8_0: gemm_subblock)")
    with torch.cuda.device(xa.device):
        st = fn(_ptr(w), _ptr(xa), _ptr(ds), _ptr(out), T, O, K, _stream(xa.device))
    _check(f"gemm({fmt})", st)
    return out


SMALL_T_MAX = 64          # mmq_gemm_q4K_small
SMALL_IMMA_T_MAX = 16     # mmq_gemm_q4K_small_imma


def gemm_small(w: torch.Tensor, xa: torch.Tensor, ds: torch.Tensor, O: int,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """q4_K GEMM for T <= 64 tokens (weight rows on the tensor core's 128-row
    side, fed from tensor memory); same operands and result as gemm("q4_K")."""
    T, K = _check_gemm_args("q4_K", w, xa, O, planes=2)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xa.device)
    with torch.cuda.device(xa.device):
        st = load().mmq_gemm_q4K_small(_ptr(w), _ptr(xa), _ptr(ds), _ptr(out), T, O, K, _stream(xa.device))
    _check("mmq_gemm_q4K_small", st)
    return out


def gemm_small_imma(w: torch.Tensor, qs: torch.Tensor, ds: torch.Tensor, O: int,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """q4_K GEMM for T <= 16 tokens on the int8 warp MMA from the int8 q8_1 values qs [T][K] and ds."""
    _need_cuda(w, qs)
    if qs.dtype != torch.int8 or qs.dim() != 2 or not qs.is_contiguous():
        raise ValueError("qs must be contiguous int8 [T][K]")
    T, K = qs.shape
    if w.dtype != torch.uint8 or not w.is_contiguous() or w.numel() != O * (K // 256) * BLOCK_BYTES["q4_K"]:
        raise ValueError("w must be contiguous uint8 holding O*(K/256) q4_K super-blocks")
    _check_ds(ds, T, K)
    out = _out(out, T, O, qs.device)
    with torch.cuda.device(qs.device):
        st = load().mmq_gemm_q4K_small_imma(_ptr(w), _ptr(qs), _ptr(ds), _ptr(out), T, O, K, _stream(qs.device))
    _check("mmq_gemm_q4K_small_imma", st)
    return out


GEMV_T_MAX = 16           # mmq_gemv_q4K, mmq_gemv_q6K


def gemv(w: torch.Tensor, xh: torch.Tensor, ds: torch.Tensor, O: int,
         out: torch.Tensor | None = None, fmt: str = "q4_K") -> torch.Tensor:
    """Decode-shaped product for T <= 16 tokens from the f16 copies of the int8
    q8_1 values xh [T][K] and ds (per-sub-block integer dots on the f16 warp
    MMA), W in q4_K or q6_K; same result as gemm(fmt) up to f32 summation order."""
    T, K = _check_gemm_args(fmt, w, xh, O, planes=1)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xh.device)
    fn = load().mmq_gemv_q4K if fmt == "q4_K" else load().mmq_gemv_q6K
    with torch.cuda.device(xh.device):
        st = fn(_ptr(w), _ptr(xh), _ptr(ds), _ptr(out), T, O, K, _stream(xh.device))
    _check(f"gemv({fmt})", st)
    return out


DECODE_T_MAX = 4          # mmq_gemv_q4K_f32
DECODE_K_MAX = 32768


def gemv_f32(w: torch.Tensor, x: torch.Tensor, O: int, out: torch.Tensor | None = None,
             fmt: str = "q4_K") -> torch.Tensor:
    """Decode-shaped product for T <= 4 f32 tokens x [T][K] with the q8_1
    quantisation built into the kernel (no quantise launch), W in q4_K or q6_K;
    same result as gemm(fmt) on quantize_q8_1(x) up to f32 summation order."""
    _need_cuda(w, x)
    if x.dim() != 2 or x.dtype != torch.float32 or x.stride(1) != 1:
        raise ValueError("x must be a row-major f32 [T][K] tensor")
    T, K = x.shape
    if fmt not in ("q4_K", "q6_K"):
        raise ValueError(f"no decode product for {fmt!r}")
    if w.dtype != torch.uint8 or w.numel() != O * (K // 256) * BLOCK_BYTES[fmt]:
        raise ValueError(f"w must hold O*(K/256) {fmt} super-blocks (uint8)")
    out = _out(out, T, O, x.device)
    fn = load().mmq_gemv_q4K_f32 if fmt == "q4_K" else load().mmq_gemv_q6K_f32
    with torch.cuda.device(x.device):
        st = fn(_ptr(w), _ptr(x), x.stride(0), _ptr(out), T, O, K, _stream(x.device))
    _check(f"gemv_f32({fmt})", st)
    return out


def interleave_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor, F: int) -> torch.Tensor:
    """The weight layout of gemm_swiglu: gate and up q4_K rows interleaved in groups
    of 64 rows (a permutation of whole rows; no arithmetic)."""
    if w_gate.shape != w_up.shape or w_gate.dtype != torch.uint8 or w_gate.numel() % F or F % 64:
        raise ValueError("gate and up must be uint8 buffers of F rows each, F % 64 == 0")
    rb = w_gate.numel() // F
    g = w_gate.reshape(F // 64, 64, rb)
    u = w_up.reshape(F // 64, 64, rb)
    return torch.cat([g, u], dim=1).reshape(-1).contiguous()


def gemm_swiglu(w_gu: torch.Tensor, xa: torch.Tensor, ds: torch.Tensor, F: int, out=None, want_qs: bool = True):
    """h = silu(X W_gate^T) * (X W_up^T) quantised to q8_1, from the interleaved
    gate/up weights (interleave_gate_up) and the input's xa/ds planes.
    Returns (qs or None, ds, xa) of h [T][F]: the operands of the down projection."""
    T, K = _check_gemm_args("q4_K", w_gu, xa, 2 * F, planes=2)
    _check_ds(ds, T, K)
    dev = xa.device
    if out is not None:
        hq, hd, hx = out
        if hd is None or hx is None:
            raise ValueError("ds and xa buffers required")
        for t, dt, shape in ((hq, torch.int8, (T, F)), (hd, torch.int32, (T, F // 32)), (hx, torch.float16, (2, T, F))):
            if t is not None and (t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous()):
                raise ValueError("bad output buffer")
    else:
        hq = torch.empty((T, F), dtype=torch.int8, device=dev) if want_qs else None
        hd = torch.empty((T, F // 32), dtype=torch.int32, device=dev)
        hx = torch.empty((2, T, F), dtype=torch.float16, device=dev)
    with torch.cuda.device(dev):
        st = load().mmq_gemm_q4K_swiglu(_ptr(w_gu), _ptr(xa), _ptr(ds), _ptr(hx), _ptr(hd), _ptr(hq), T, F, K,
                                        _stream(dev))
    _check("mmq_gemm_q4K_swiglu", st)
    return hq, hd, hx


def splitk_sizes(T: int, O: int, K: int, ksplit: int) -> tuple[int, int]:
    """(floats of partial-sum workspace, ints of tile counters) for a split-K q4_K GEMM."""
    pf, nc = ctypes.c_int64(0), ctypes.c_int64(0)
    _check("mmq_splitk_sizes", load().mmq_splitk_sizes(T, O, K, ksplit, ctypes.byref(pf), ctypes.byref(nc)))
    return pf.value, nc.value


_SM_COUNT: dict[int, int] = {}


def sm_count(device: torch.device | int | None = None) -> int:
    """Streaming multiprocessors of a CUDA device (the current one by default)."""
    idx = torch.cuda.current_device() if device is None else torch.device("cuda", device).index \
        if isinstance(device, int) else (device.index if device.index is not None else torch.cuda.current_device())
    if idx not in _SM_COUNT:
        _SM_COUNT[idx] = torch.cuda.get_device_properties(idx).multi_processor_count
    return _SM_COUNT[idx]


def choose_ksplit(T: int, O: int, K: int, sms: int | None = None) -> int:
    """Splits of K that bring the grid near one wave when the output has few
    tiles; `sms` defaults to the current device's SM count."""
    if sms is None:
        sms = sm_count()
    tiles = -(-O // 128) * -(-T // 128)
    return max(1, min(K // 256, sms // max(1, tiles)))


class SplitKWorkspace:
    """Caller-owned scratch of the split-K q4_K GEMM: partial sums and tile
    counters (the counters start at zero and every call leaves them at zero).
    Calls that share one workspace must be ordered (one stream)."""

    def __init__(self, device, max_partial_floats: int, max_tiles: int):
        self.part = torch.empty(max(1, max_partial_floats), dtype=torch.float32, device=device)
        self.counters = torch.zeros(max(1, max_tiles), dtype=torch.int32, device=device)

    def fits(self, partial_floats: int, tiles: int) -> bool:
        return partial_floats <= self.part.numel() and tiles <= self.counters.numel()


def gemm_splitk(w: torch.Tensor, xa: torch.Tensor, ds: torch.Tensor, O: int, ksplit: int | None = None,
                workspace: SplitKWorkspace | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """q4_K production GEMM with K split over `ksplit` CTAs per output tile (default:
    choose_ksplit); partial sums are added in a fixed order, so results repeat bit
    for bit.  Without `workspace` one is allocated for this call."""
    T, K = _check_gemm_args("q4_K", w, xa, O, planes=2)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xa.device)
    if ksplit is None:
        ksplit = choose_ksplit(T, O, K)
    pf, nc = splitk_sizes(T, O, K, ksplit)
    if workspace is None or not workspace.fits(pf, nc):
        workspace = SplitKWorkspace(xa.device, pf, nc)
    with torch.cuda.device(xa.device):
        st = load().mmq_gemm_q4K_splitk(_ptr(w), _ptr(xa), _ptr(ds), _ptr(out), T, O, K, ksplit,
                                        _ptr(workspace.part), _ptr(workspace.counters), _stream(xa.device))
    _check("mmq_gemm_q4K_splitk", st)
    return out


def gemm_splitk_static(w: torch.Tensor, xa: torch.Tensor, ds: torch.Tensor, O: int, ksplit: int | None = None,
                       out: torch.Tensor | None = None) -> torch.Tensor:
    """gemm_splitk with the library's static scratch (no workspace anywhere);
    calls on one device must not overlap in time."""
    T, K = _check_gemm_args("q4_K", w, xa, O, planes=2)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xa.device)
    if ksplit is None:
        ksplit = choose_ksplit(T, O, K)
    with torch.cuda.device(xa.device):
        st = load().mmq_gemm_q4K_splitk_static(_ptr(w), _ptr(xa), _ptr(ds), _ptr(out), T, O, K, ksplit,
                                               _stream(xa.device))
    _check("mmq_gemm_q4K_splitk_static", st)
    return out


def gemm_subblock(fmt: str, w: torch.Tensor, xh: torch.Tensor, ds: torch.Tensor, O: int,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """Per-sub-block GEMM (exact integer sub-block dots + f32 fold) from the xh/ds planes;
    `fmt` q4_K, q5_K, q6_K or q8_0 (q8_0's only form)."""
    T, K = _check_gemm_args(fmt, w, xh, O, planes=1)
    _check_ds(ds, T, K)
    out = _out(out, T, O, xh.device)
    fn = {"q4_K": load().mmq_gemm_q4K_subblock, "q6_K": load().mmq_gemm_q6K_subblock,
          "q5_K": load().mmq_gemm_q5K_subblock, "q8_0": load().mmq_gemm_q8_0}[fmt]
    with torch.cuda.device(xh.device):
        st = fn(_ptr(w), _ptr(xh), _ptr(ds), _ptr(out), T, O, K, _stream(xh.device))
    _check(f"gemm_subblock({fmt})", st)
    return out


def debug_subdots(fmt: str, w: torch.Tensor, xh: torch.Tensor, O: int) -> torch.Tensor:
    """Per-sub-block integer dots: int32 [T][O][K/16] (q6_K) or [T][O][K/32] (the others)."""
    T, K = _check_gemm_args(fmt, w, xh, O, planes=1)
    nsub = K // 16 if fmt == "q6_K" else K // 32
    out = torch.empty((T, O, nsub), dtype=torch.int32, device=xh.device)
    fn = {"q4_K": load().mmq_debug_subdots_q4K, "q6_K": load().mmq_debug_subdots_q6K,
          "q5_K": load().mmq_debug_subdots_q5K, "q8_0": load().mmq_debug_subdots_q8_0}[fmt]
    with torch.cuda.device(xh.device):
        st = fn(_ptr(w), _ptr(xh), _ptr(out), T, O, K, _stream(xh.device))
    _check("mmq_debug_subdots", st)
    return out


def check_status(device: torch.device | None = None):
    """Synchronise the current stream and raise if a kernel reported an error."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    detail = (ctypes.c_int * 4)()
    with torch.cuda.device(dev):
        st = load().mmq_check_status(_stream(dev), detail)
    if st != 0:
        info = (ctypes.c_int * 4)()
        load().mmq_last_failure_info(info)
        raise MMQError(f"kernel (id {detail[1]}, site {detail[2]}, block {detail[3]}; waited {info[0]} us over "
                       f"{info[1]} polls for parity {info[2]} of the barrier at shared address {info[3]})", st)


def tensor_peak_tmacs(kind: str = "int8", device: torch.device | None = None) -> float:
    """Measured warp-level tensor throughput (TMAC/s) of the device: 'int8' or 'f16'."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    v = ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        st = load().mmq_probe_tensor_peak(0 if kind == "int8" else 1, ctypes.byref(v), _stream(dev))
    _check("mmq_probe_tensor_peak", st)
    return v.value


def mmq_forward(fmt: str, w: torch.Tensor, x: torch.Tensor, O: int) -> torch.Tensor:
    """Quantise x [T][K] to q8_1 and run the production GEMM: the whole hot path."""
    _, ds, _, xa = quantize_q8_1(x, want_qs=False, want_xh=False, want_xa=True)
    return gemm(fmt, w, xa, ds, O)
