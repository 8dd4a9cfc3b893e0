"""Seeded synthetic inputs for the k-quant MMQ prefill GEMM.

This module only draws random numbers and lays the drawn bytes out in the
storage formats; it performs none of the method's arithmetic (no dequant,
no quantisation, no dot products).  Both the CUDA path and the CPU oracle
consume the bytes produced here, so the two can be compared on identical
inputs.

Storage formats (little-endian):

* q4_K super-block, 144 bytes for 256 weights of one row:
  ``d`` f16 (bytes 0-1), ``dmin`` f16 (2-3), 12 bytes of packed 6-bit
  sub-block scales/mins (4-15), 128 bytes of 4-bit ``qs`` (16-143).
  The weight matrix is ``[O][K/256]`` blocks, row after row.
* q6_K super-block, 210 bytes: ``ql`` (0-127), ``qh`` (128-191),
  16 int8 ``scales`` (192-207), ``d`` f16 (208-209).

Distributions (the pages' 7B-class workload, redrawn synthetically):

* X ~ N(0, 1) in f64, stored f32; optionally 1 % of the channels (the
  first ``round(0.01*K)`` indices of a permutation drawn after X from the
  same generator) are scaled by 20 to mimic activation outliers.
* q4_K: ``qs`` bytes uniform 0..255 (both nibbles uniform 0..15); the 12
  scale bytes uniform 0..255, which makes every packed 6-bit scale and min
  uniform on 0..63 and independent; ``d`` and ``dmin`` are
  ``f16(|N(0, 1e-3)|)`` (round-to-nearest-even by NumPy; subnormals and
  zero allowed).
* q6_K: ``ql`` and ``qh`` bytes uniform (so every 6-bit q is uniform on
  0..63); scales uniform int8 on -64..63; ``d = f16(|N(0, 1e-3)|)``.
* q5_K (176 B: d, dmin, scales as q4_K, ``qh[32]``, ``qs[128]``): bytes
  uniform, so every 5-bit q is uniform on 0..31; q8_0 (34 B per 32: f16
  ``d``, 32 int8): values uniform on -127..127, ``d`` as above.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK_K = 256            # weights per k-quant super-block
QK8_1 = 32            # activations per q8_1 block
Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q5K_BLOCK_BYTES = 176
Q8_0_BLOCK_BYTES = 34


def _f16_bits(values: np.ndarray) -> np.ndarray:
    return values.astype(np.float16).view(np.uint16)


def _abs_normal_f16_bits(rng: np.random.Generator, shape, sigma: float = 1e-3) -> np.ndarray:
    return _f16_bits(np.abs(rng.standard_normal(shape) * sigma))


def make_x(T: int, K: int, seed: int, outliers: bool = True) -> np.ndarray:
    """Activations X[T][K] f32 ~ N(0,1), optional x20 outlier channels."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float32)
    if outliers:
        n_out = int(round(0.01 * K))
        idx = rng.permutation(K)[:n_out]
        x[:, idx] *= np.float32(20.0)
    return np.ascontiguousarray(x)


def make_q4K(O: int, K: int, seed: int) -> np.ndarray:
    """Random q4_K weight bytes, shape [O, K/256*144] uint8."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nsb = K // QK_K
    rng = np.random.default_rng(seed)
    d = _abs_normal_f16_bits(rng, (O, nsb))
    dmin = _abs_normal_f16_bits(rng, (O, nsb))
    scales = rng.integers(0, 256, size=(O, nsb, 12), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(O, nsb, 128), dtype=np.uint8)
    blk = np.empty((O, nsb, Q4K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(O, nsb, 2)
    blk[:, :, 2:4] = dmin.view(np.uint8).reshape(O, nsb, 2)
    blk[:, :, 4:16] = scales
    blk[:, :, 16:144] = qs
    return blk.reshape(O, nsb * Q4K_BLOCK_BYTES)


def make_q6K(O: int, K: int, seed: int) -> np.ndarray:
    """Random q6_K weight bytes, shape [O, K/256*210] uint8."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nsb = K // QK_K
    rng = np.random.default_rng(seed)
    ql = rng.integers(0, 256, size=(O, nsb, 128), dtype=np.uint8)
    qh = rng.integers(0, 256, size=(O, nsb, 64), dtype=np.uint8)
    sc = rng.integers(-64, 64, size=(O, nsb, 16), dtype=np.int8)
    d = _abs_normal_f16_bits(rng, (O, nsb))
    blk = np.empty((O, nsb, Q6K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, :, 0:128] = ql
    blk[:, :, 128:192] = qh
    blk[:, :, 192:208] = sc.view(np.uint8)
    blk[:, :, 208:210] = d.view(np.uint8).reshape(O, nsb, 2)
    return blk.reshape(O, nsb * Q6K_BLOCK_BYTES)


def make_q5K(O: int, K: int, seed: int) -> np.ndarray:
    """Random q5_K weight bytes, shape [O, K/256*176] uint8: d, dmin and the
    12 scale bytes as make_q4K, qh and qs bytes uniform (every 5-bit q uniform
    on 0..31)."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nsb = K // QK_K
    rng = np.random.default_rng(seed)
    d = _abs_normal_f16_bits(rng, (O, nsb))
    dmin = _abs_normal_f16_bits(rng, (O, nsb))
    scales = rng.integers(0, 256, size=(O, nsb, 12), dtype=np.uint8)
    qh = rng.integers(0, 256, size=(O, nsb, 32), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(O, nsb, 128), dtype=np.uint8)
    blk = np.empty((O, nsb, Q5K_BLOCK_BYTES), dtype=np.uint8)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(O, nsb, 2)
    blk[:, :, 2:4] = dmin.view(np.uint8).reshape(O, nsb, 2)
    blk[:, :, 4:16] = scales
    blk[:, :, 16:48] = qh
    blk[:, :, 48:176] = qs
    return blk.reshape(O, nsb * Q5K_BLOCK_BYTES)


def make_q8_0(O: int, K: int, seed: int) -> np.ndarray:
    """Random q8_0 weight bytes, shape [O, K/32*34] uint8: d = f16(|N(0, 1e-3)|),
    32 int8 values uniform on -127..127 per block."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // 32
    rng = np.random.default_rng(seed)
    d = _abs_normal_f16_bits(rng, (O, nb))
    q = rng.integers(-127, 128, size=(O, nb, 32)).astype(np.int8)
    blk = np.empty((O, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(O, nb, 2)
    blk[:, :, 2:34] = q.view(np.uint8)
    return blk.reshape(O, nb * Q8_0_BLOCK_BYTES)


def make_weights(fmt: str, O: int, K: int, seed: int) -> np.ndarray:
    if fmt == "q4_K":
        return make_q4K(O, K, seed)
    if fmt == "q6_K":
        return make_q6K(O, K, seed)
    if fmt == "q5_K":
        return make_q5K(O, K, seed)
    if fmt == "q8_0":
        return make_q8_0(O, K, seed)
    raise ValueError(f"unknown weight format {fmt!r}")


@dataclass(frozen=True)
class Gemm:
    """One GEMM of a workload: Y[T][O] = X[T][K] . W[O][K]^T."""
    name: str
    fmt: str          # "q4_K" or "q6_K"
    T: int
    K: int
    O: int
    w_seed: int
    x_seed: int
    outliers: bool = True

    @property
    def macs(self) -> int:
        return self.T * self.K * self.O

    def weights(self) -> np.ndarray:
        return make_weights(self.fmt, self.O, self.K, self.w_seed)

    def x(self) -> np.ndarray:
        return make_x(self.T, self.K, self.x_seed, self.outliers)


@dataclass(frozen=True)
class Workload:
    name: str
    gemms: tuple = field(default_factory=tuple)

    @property
    def macs(self) -> int:
        return sum(g.macs for g in self.gemms)


def _w_seed(cfg: int, m: int) -> int:
    return 100 + 10 * cfg + m


def _x_seed(cfg: int, j: int) -> int:
    return 10 * cfg + j


def config(cfg: int, T: int | None = None) -> Workload:
    """The five workload configurations, by index.

    0: tiny q4_K (T=64, K=512, O=256), no outliers.
    1: 7B attention projection q4_K (T=512, K=O=4096).
    2: 7B FFN q4_K: gate and up (K=4096, O=11008, shared X) and down
       (K=11008, O=4096).
    3: 7B attn_v q6_K (T=512, K=O=4096).
    4: q4_K token sweep; ``T`` picks the token count, the two shapes are
       K=4096/O=4096 and K=11008/O=4096.
    """
    if cfg == 0:
        return Workload("tiny_q4K_T64_K512_O256",
                        (Gemm("tiny", "q4_K", 64, 512, 256, _w_seed(0, 0), _x_seed(0, 0), False),))
    if cfg == 1:
        return Workload("attn_proj_q4K_T512_K4096_O4096",
                        (Gemm("attn_proj", "q4_K", 512, 4096, 4096, _w_seed(1, 0), _x_seed(1, 0)),))
    if cfg == 2:
        return Workload("ffn_q4K_T512",
                        (Gemm("gate", "q4_K", 512, 4096, 11008, _w_seed(2, 0), _x_seed(2, 0)),
                         Gemm("up", "q4_K", 512, 4096, 11008, _w_seed(2, 1), _x_seed(2, 0)),
                         Gemm("down", "q4_K", 512, 11008, 4096, _w_seed(2, 2), _x_seed(2, 1))))
    if cfg == 3:
        return Workload("attn_v_q6K_T512_K4096_O4096",
                        (Gemm("attn_v", "q6_K", 512, 4096, 4096, _w_seed(3, 0), _x_seed(3, 0)),))
    if cfg == 4:
        if T is None:
            raise ValueError("config 4 needs T")
        return Workload(f"sweep_q4K_T{T}",
                        (Gemm("sweep_k4096", "q4_K", T, 4096, 4096, _w_seed(4, 0), _x_seed(4, 0)),
                         Gemm("sweep_k11008", "q4_K", T, 11008, 4096, _w_seed(4, 1), _x_seed(4, 1))))
    raise ValueError(f"no config {cfg}")


SWEEP_T = (16, 64, 256, 1024, 4096)


def layer_7b(T: int = 512) -> Workload:
    """One LLaMA-7B-shaped decoder layer's seven projections at T tokens.

    q, k, o: q4_K 4096x4096; v: q6_K 4096x4096; gate, up: q4_K
    4096->11008; down: q4_K 11008->4096.  q/k/v share one activation input,
    gate/up share another, o and down each have their own: four q8_1
    quantisations per layer.
    """
    base = 500
    return Workload(f"layer7b_T{T}", (
        Gemm("q", "q4_K", T, 4096, 4096, base + 0, base + 0),
        Gemm("k", "q4_K", T, 4096, 4096, base + 1, base + 0),
        Gemm("v", "q6_K", T, 4096, 4096, base + 2, base + 0),
        Gemm("o", "q4_K", T, 4096, 4096, base + 3, base + 1),
        Gemm("gate", "q4_K", T, 4096, 11008, base + 4, base + 2),
        Gemm("up", "q4_K", T, 4096, 11008, base + 5, base + 2),
        Gemm("down", "q4_K", T, 11008, 4096, base + 6, base + 3),
    ))


def block_bytes(fmt: str) -> int:
    """Bytes per 256 weights of one row."""
    return {"q4_K": Q4K_BLOCK_BYTES, "q6_K": Q6K_BLOCK_BYTES, "q5_K": Q5K_BLOCK_BYTES,
            "q8_0": 8 * Q8_0_BLOCK_BYTES}[fmt]
