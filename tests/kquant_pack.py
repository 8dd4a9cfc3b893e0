"""Test-side packers: explicit field values -> k-quant block bytes.

These build blocks whose every element is known to the test, so the
oracle's decoding (and the CUDA path's) can be checked against values the
test chose rather than values it decoded.  They follow the layout
statements of the pages and the readings recorded in the design notes:

* q4_K (144 B): d f16, dmin f16, 12 bytes of packed 6-bit scales/mins,
  128 bytes qs.  Sub-block sg (32 weights) lives in qs bytes
  (sg>>1)*32 .. +31, low nibble for even sg, high nibble for odd sg
  ("31 . r28 -- Direction-A raw-nibble NB kernel", 3.2 Key code).
* 12-byte scale packing: GGUF k-quant packing (a reading; the pages elide it).
* q6_K (210 B): ql[128], qh[64], int8 scales[16], d f16 (GGUF order, a
  reading; the pages list the fields only).
* q5_K (176 B): d, dmin, the q4_K scale packing, qh[32], qs[128] (GGUF
  order, a reading: the pages name only the k-quant family); q8_0 (34 B):
  f16 d and 32 int8 values.
"""
from __future__ import annotations

import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def pack_q4K_scales(sc, m) -> np.ndarray:
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert len(sc) == 8 and len(m) == 8
    assert all(0 <= v < 64 for v in sc + m)
    s = np.zeros(12, np.uint8)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[4 + j] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[8 + j] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return s


def pack_q4K_qs(q) -> np.ndarray:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 16
    qs = np.zeros(128, np.uint8)
    for p in range(4):
        lo = q[64 * p: 64 * p + 32]
        hi = q[64 * p + 32: 64 * p + 64]
        qs[32 * p: 32 * p + 32] = (lo | (hi << 4)).astype(np.uint8)
    return qs


def pack_q4K_block(d: float, dmin: float, sc, m, q) -> np.ndarray:
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    blk[2:4] = np.array([f16_bits(dmin)], np.uint16).view(np.uint8)
    blk[4:16] = pack_q4K_scales(sc, m)
    blk[16:144] = pack_q4K_qs(q)
    return blk


def pack_q6K_block(d: float, sc, q) -> np.ndarray:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 64
    sc = np.asarray(sc, dtype=np.int64)
    assert sc.shape == (16,) and sc.min() >= -128 and sc.max() < 128
    blk = np.zeros(210, np.uint8)
    for h in range(2):
        base = 128 * h
        for l in range(32):
            q0, q1, q2, q3 = (int(q[base + l]), int(q[base + 32 + l]),
                              int(q[base + 64 + l]), int(q[base + 96 + l]))
            blk[64 * h + l] = (q0 & 15) | ((q2 & 15) << 4)
            blk[64 * h + 32 + l] = (q1 & 15) | ((q3 & 15) << 4)
            blk[128 + 32 * h + l] = (q0 >> 4) | ((q1 >> 4) << 2) | ((q2 >> 4) << 4) | ((q3 >> 4) << 6)
    blk[192:208] = sc.astype(np.int8).view(np.uint8)
    blk[208:210] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    return blk


def pack_q5K_block(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """One 176-byte q5_K block (d, dmin, the q4_K scale packing, qh[32], qs[128])
    from 8 scales, 8 mins and 256 values q in 0..31: the low 4 bits go where
    q4_K keeps its nibble, bit 4 of element 32j+i into bit j of qh[i]."""
    q = np.asarray(q, np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 31
    blk = np.zeros(176, np.uint8)
    blk[0:2] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    blk[2:4] = np.array([f16_bits(dmin)], np.uint16).view(np.uint8)
    blk[4:16] = pack_q4K_scales(sc, m)
    qh = np.zeros(32, np.int64)
    for e in range(256):
        j, i = divmod(e, 32)
        qh[i] |= ((q[e] >> 4) & 1) << j
    blk[16:48] = qh.astype(np.uint8)
    blk[48:176] = pack_q4K_qs(q & 15)
    return blk


def pack_q8_0_block(d: float, q) -> np.ndarray:
    """One 34-byte q8_0 block: f16 d, then 32 int8 values."""
    q = np.asarray(q, np.int64)
    assert q.shape == (32,) and q.min() >= -128 and q.max() <= 127
    blk = np.zeros(34, np.uint8)
    blk[0:2] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    blk[2:34] = q.astype(np.int8).view(np.uint8)
    return blk
