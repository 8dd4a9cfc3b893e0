"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, not against the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped fold
term, a wrong sign, a swapped scale/min, a wrong nibble or byte index, a
transposed operand, a wrong rounding rule) fails at least one of them.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

from tests.kquant_pack import (f16_bits, pack_q4K_block, pack_q4K_qs, pack_q4K_scales, pack_q5K_block, pack_q8_0_block,
                               pack_q6K_block)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ f16 (P-c) --

def test_f16_to_f32_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _check_f32_to_f16(orc, bits: np.ndarray):
    f = bits.view(np.float32)
    got = orc.f32_to_f16(f)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    # any NaN maps to a NaN
    g = got[nan]
    assert np.all(((g & 0x7c00) == 0x7c00) & ((g & 0x03ff) != 0))


def test_f32_to_f16_strided_sweep(orc):
    # every 4099th f32 bit pattern over the whole space, both signs
    bits = (np.arange(0, 1 << 32, 4099, dtype=np.uint64)).astype(np.uint32)
    _check_f32_to_f16(orc, bits)


@pytest.mark.parametrize("exp", [-26, -25, -24, -15, -14, -13, 0, 15])
def test_f32_to_f16_full_binades(orc, exp):
    # every mantissa in binades around the subnormal boundary, 1.0 and overflow
    man = np.arange(1 << 23, dtype=np.uint32)
    bits = (np.uint32(exp + 127) << np.uint32(23)) | man
    _check_f32_to_f16(orc, bits)
    _check_f32_to_f16(orc, bits | np.uint32(0x80000000))


# ----------------------------------------------------- block layout (P-c) --

def test_q4K_nibbles_every_byte_value(orc):
    # each byte value at each qs position decodes to (lo, hi) in sub-blocks (2p, 2p+1)
    rng = np.random.default_rng(1)
    for trial in range(4):
        q = rng.integers(0, 16, 256)
        blk = pack_q4K_block(1.0, 1.0, [0] * 8, [0] * 8, q)
        assert np.array_equal(orc.q4K_quants(blk), q)
    for b in range(256):
        blk = np.zeros(144, np.uint8)
        blk[16:] = b
        got = orc.q4K_quants(blk)
        for sg in range(8):
            want = (b & 15) if sg % 2 == 0 else (b >> 4)
            assert np.all(got[32 * sg: 32 * sg + 32] == want)


def test_q4K_nibble_positions(orc):
    # one nonzero byte: exactly one element in each of the two sub-blocks it feeds
    for pos in range(128):
        blk = np.zeros(144, np.uint8)
        blk[16 + pos] = 0xA5   # lo = 5, hi = 10
        got = orc.q4K_quants(blk)
        p, i = divmod(pos, 32)
        want = np.zeros(256, np.int64)
        want[64 * p + i] = 5
        want[64 * p + 32 + i] = 10
        assert np.array_equal(got, want), pos


def test_q4K_scale_packing_exhaustive_per_field(orc):
    rng = np.random.default_rng(2)
    for field in range(16):
        for v in range(64):
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            if field < 8:
                sc[field] = v
            else:
                m[field - 8] = v
            s = pack_q4K_scales(sc, m)
            for j in range(8):
                assert orc.q4K_scale_min(s, j) == (sc[j], m[j])


def test_q4K_scale_packing_is_a_bijection(orc):
    # 16 six-bit fields fill the 96 bits exactly: decode then re-pack is the identity
    rng = np.random.default_rng(3)
    for _ in range(2000):
        s = rng.integers(0, 256, 12).astype(np.uint8)
        f = [orc.q4K_scale_min(s, j) for j in range(8)]
        assert np.array_equal(pack_q4K_scales([a for a, _ in f], [b for _, b in f]), s)


def test_q6K_values_every_position(orc):
    rng = np.random.default_rng(4)
    for v in range(64):
        q = rng.integers(0, 64, 256)
        q[rng.integers(0, 256, 64)] = v
        blk = pack_q6K_block(1.0, np.zeros(16), q)
        assert np.array_equal(orc.q6K_quants(blk), q)
    for e in range(256):
        q = np.zeros(256, np.int64)
        q[e] = 63
        got = orc.q6K_quants(pack_q6K_block(1.0, np.zeros(16), q))
        assert np.array_equal(got, q), e


def test_q6K_layout_is_a_bijection(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        raw = rng.integers(0, 256, 210).astype(np.uint8)
        q = orc.q6K_quants(raw)
        sc = raw[192:208].view(np.int8).astype(np.int64)
        d = float(raw[208:210].view(np.float16)[0])
        if not np.isfinite(d):
            continue
        again = pack_q6K_block(d, sc, q)
        assert np.array_equal(again[:208], raw[:208])


# ------------------------------------------------ closed forms (P-a) ----

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "q4K_single_superblock.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, sc, m, y = [p.strip() for p in line.split("|")]
            rows.append((name, [int(v) for v in sc.split()], [int(v) for v in m.split()], float(y)))
    return rows


@pytest.mark.parametrize("name,sc,m,y", _golden_rows())
def test_q4K_single_superblock_closed_form(orc, name, sc, m, y):
    q = np.array([(i % 32) % 16 for i in range(256)])      # byte i holds 0x11*(i mod 16)
    blk = pack_q4K_block(1.0, 1.0, sc, m, q)
    assert np.all(blk[16:] == np.array([0x11 * (i % 16) for i in range(128)], np.uint8))
    x = np.full((1, 256), 127.0, np.float32)
    qs, ds = orc.quantize_q8_1(x)
    assert np.all(qs == 127) and np.all(ds == (0x3C00 | (4064 << 16)))
    assert np.all(orc.subdots("q4_K", blk, qs, 1) == 30480)
    got = orc.gemm("q4_K", blk, qs, ds, 1)
    assert got[0, 0] == y
    assert orc.gemm_dequant("q4_K", blk, qs, ds, 1)[0, 0] == y


# ------------------------------------------------ one-hot read-back (P-b) --

def test_q4K_one_hot_reads_back_weights(orc):
    rng = np.random.default_rng(6)
    q = rng.integers(0, 16, 256)
    sc = rng.integers(0, 64, 8)
    m = rng.integers(0, 64, 8)
    blk = pack_q4K_block(1.0, 1.0, sc, m, q)
    x = 127.0 * np.eye(256, dtype=np.float32)      # token t has 127 at k = t
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm("q4_K", blk, qs, ds, 1)[:, 0]
    want = np.array([sc[k // 32] * q[k] - m[k // 32] for k in range(256)], np.float64)
    assert np.array_equal(y / 127.0, want)
    assert np.array_equal(orc.dequant("q4_K", blk, 1, 256)[0], want)


def test_q6K_one_hot_reads_back_weights(orc):
    rng = np.random.default_rng(7)
    q = rng.integers(0, 64, 256)
    sc = rng.integers(-128, 128, 16)
    blk = pack_q6K_block(1.0, sc, q)
    x = 127.0 * np.eye(256, dtype=np.float32)
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm("q6_K", blk, qs, ds, 1)[:, 0]
    want = np.array([sc[k // 16] * (q[k] - 32) for k in range(256)], np.float64)
    assert np.array_equal(y / 127.0, want)
    assert np.array_equal(orc.dequant("q6_K", blk, 1, 256)[0], want)


def test_q4K_multi_superblock_one_hot(orc):
    # K=512: the second super-block's header and qs are used for k >= 256
    rng = np.random.default_rng(8)
    blocks, want = [], []
    for _ in range(2):
        q = rng.integers(0, 16, 256)
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        dd = float(rng.choice([0.5, 1.0, 2.0]))
        dm = float(rng.choice([0.25, 1.0, 4.0]))
        blocks.append(pack_q4K_block(dd, dm, sc, m, q))
        want += [dd * sc[k // 32] * q[k] - dm * m[k // 32] for k in range(256)]
    w = np.concatenate(blocks)
    x = 127.0 * np.eye(512, dtype=np.float32)
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm("q4_K", w, qs, ds, 1)[:, 0]
    assert np.array_equal(y / 127.0, np.array(want))


# ------------------------------------------------- q8_1 cases (P-d) ----

def test_q8_1_zero_block(orc):
    x = np.zeros((1, 64), np.float32)
    x[0, 32:] = np.linspace(-1, 1, 32)
    qs, ds = orc.quantize_q8_1(x)
    assert np.all(qs[0, :32] == 0) and ds[0, 0] == 0


def test_q8_1_ties_and_extremes(orc):
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0                 # amax = 127 -> d32 = 1
    x[0, 1:6] = [2.5, -2.5, 0.5, -0.5, 1.5]
    x[0, 6] = -127.0
    x[0, 7] = 126.49
    qs, ds = orc.quantize_q8_1(x)
    assert list(qs[0, :8]) == [127, 3, -3, 1, -1, 2, -127, 126]
    assert ds[0, 0] & 0xFFFF == 0x3C00
    assert np.int16(ds[0, 0] >> 16) == int(qs[0].astype(np.int64).sum())


def test_q8_1_single_max_maps_to_127(orc):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((200, 32)).astype(np.float32)
    qs, ds = orc.quantize_q8_1(x)
    amax_idx = np.abs(x).argmax(axis=1)
    picked = qs[np.arange(200), amax_idx].astype(np.int64)
    assert np.array_equal(np.abs(picked), np.full(200, 127))
    assert np.array_equal(np.sign(picked), np.sign(x[np.arange(200), amax_idx]).astype(np.int64))


def test_q8_1_invariants_random(orc):
    rng = np.random.default_rng(10)
    x = (rng.standard_normal((64, 1024)) * rng.choice([1e-6, 1e-3, 1.0, 30.0], (64, 1))).astype(np.float32)
    x[:, ::97] *= 20
    qs, ds = orc.quantize_q8_1(x)
    xb = x.reshape(64, 32, 32).astype(np.float64)
    qb = qs.reshape(64, 32, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    assert np.abs(qb).max() <= 127
    # |x - d32*q| <= d32/2 up to the f32 rounding of x/d32
    assert np.all(np.abs(xb - d32[..., None] * qb) <= 0.5 * d32[..., None] * (1 + 1e-5) + 1e-30)
    ssum = (ds >> 16).astype(np.uint16).view(np.int16).astype(np.int64)
    assert np.array_equal(ssum, qb.sum(axis=2))
    assert np.abs(ssum).max() <= 32 * 127
    d16 = (ds & 0xFFFF).astype(np.uint16)
    assert np.array_equal(d16, d32.astype(np.float32).astype(np.float16).view(np.uint16))


# ------------------------------------------- fold identity (P-e) ----

@pytest.mark.parametrize("fmt", ["q4_K", "q6_K", "q5_K", "q8_0"])
@pytest.mark.parametrize("T,O,K", [(3, 5, 256), (7, 4, 768), (16, 9, 1024)])
def test_method_form_matches_full_dequant(orc, fmt, T, O, K):
    from quantized_prefill_gemm_mmq_gb300 import synth
    w = synth.make_weights(fmt, O, K, seed=T * 1000 + O)
    x = synth.make_x(T, K, seed=K + O)
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm(fmt, w, qs, ds, O).astype(np.float64)
    y2 = orc.gemm_dequant(fmt, w, qs, ds, O)
    scale = np.abs(y2).max()
    assert scale > 0
    assert np.abs(y - y2).max() <= 1e-6 * scale
    # the unquantised product is close too (q8_1 error only), for information
    x_w = x.astype(np.float64) @ orc.dequant(fmt, w, O, K).T
    assert np.abs(y - x_w).max() <= 0.05 * np.abs(x_w).max()


# ----------------------------------------------- brute force (P-f) ----

@pytest.mark.parametrize("T", [1, 2, 3])
@pytest.mark.parametrize("O", [1, 2, 3])
@pytest.mark.parametrize("K", [256, 512])
def test_subdots_brute_force(orc, T, O, K):
    rng = np.random.default_rng(T * 100 + O * 10 + K)
    nsb = K // 256
    q4 = rng.integers(0, 16, (O, K))
    q6 = rng.integers(0, 64, (O, K))
    w4 = np.concatenate([pack_q4K_block(1.0, 1.0, rng.integers(0, 64, 8), rng.integers(0, 64, 8),
                                        q4[o, 256 * s: 256 * s + 256])
                         for o in range(O) for s in range(nsb)])
    w6 = np.concatenate([pack_q6K_block(1.0, rng.integers(-128, 128, 16), q6[o, 256 * s: 256 * s + 256])
                         for o in range(O) for s in range(nsb)])
    a = rng.integers(-127, 128, (T, K)).astype(np.int8)
    got4 = orc.subdots("q4_K", w4, a, O)
    got6 = orc.subdots("q6_K", w6, a, O)
    for t in range(T):
        for o in range(O):
            for b in range(K // 32):
                c = 0
                for i in range(32):
                    c += int(q4[o, 32 * b + i]) * int(a[t, 32 * b + i])
                assert got4[t, o, b] == c
            for u in range(K // 16):
                c = 0
                for i in range(16):
                    c += (int(q6[o, 16 * u + i]) - 32) * int(a[t, 16 * u + i])
                assert got6[t, o, u] == c


def test_gemm_points_match_full(orc):
    from quantized_prefill_gemm_mmq_gb300 import synth
    for fmt in ("q4_K", "q6_K"):
        w = synth.make_weights(fmt, 13, 512, seed=11)
        x = synth.make_x(9, 512, seed=12)
        qs, ds = orc.quantize_q8_1(x)
        y = orc.gemm(fmt, w, qs, ds, 13)
        ti, oi = np.meshgrid(np.arange(9), np.arange(13), indexing="ij")
        pts = orc.gemm_points(fmt, w, qs, ds, 13, ti.ravel(), oi.ravel())
        assert np.array_equal(pts, y.ravel())


def test_f16_bits_helper_matches_oracle(orc):
    for v in [0.0, 1.0, 1e-3, 6e-5, 65504.0, -2.5]:
        assert f16_bits(v) == int(orc.f32_to_f16(np.array([v], np.float32))[0])


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K"])
def test_oracle_threads_do_not_change_results(orc, fmt):
    """The OpenMP form divides output columns among threads; each output is the
    same single-thread computation, so the result must be identical bit for bit
    to the single-thread loop (also with more threads than columns)."""
    from quantized_prefill_gemm_mmq_gb300 import synth
    T, O, K = 9, 37, 768
    w = synth.make_weights(fmt, O, K, seed=5)
    qs, ds = orc.quantize_q8_1(synth.make_x(T, K, seed=6))
    y1 = orc.gemm(fmt, w, qs, ds, O, threads=1)
    for nt in (None, 3, 64):
        assert np.array_equal(orc.gemm(fmt, w, qs, ds, O, threads=nt).view(np.uint32), y1.view(np.uint32))


# ------------------------------------------------------------ SwiGLU ----

def _silu(orc, x):
    x = np.asarray(x, np.float32)
    return orc.swiglu(x, np.ones_like(x))


def test_swiglu_identities(orc):
    """silu pinned by identities of the function, not by its formula:
    silu(0) = 0; silu(x) - silu(-x) = x (odd part); silu(x) = x once e^-x is
    below half an f32 ulp of 1 (x >= 17); silu(x) = -0 where e^-x overflows;
    h is linear in u (times 2 is exact)."""
    assert _silu(orc, [0.0])[0] == 0.0
    x = np.linspace(-30.0, 30.0, 6001, dtype=np.float32)
    d = _silu(orc, x).astype(np.float64) - _silu(orc, -x).astype(np.float64)
    assert np.all(np.abs(d - x) <= 4 * np.spacing(np.maximum(np.abs(x), 1.0).astype(np.float32)))
    big = np.array([17.0, 20.0, 100.0, 1e4, 3e38], np.float32)
    assert np.array_equal(_silu(orc, big), big)
    neg = np.array([-89.0, -100.0, -1e4], np.float32)
    out = _silu(orc, neg)
    assert np.all(out == 0.0) and np.all(np.signbit(out))
    rng = np.random.default_rng(3)
    g = rng.standard_normal(1000).astype(np.float32) * 8
    u = rng.standard_normal(1000).astype(np.float32)
    assert np.array_equal(orc.swiglu(g, 2 * u), 2 * orc.swiglu(g, u))
    # sign: silu(x) > 0 for x > 0 and < 0 for x < 0, |silu(x)| < |x| below 17
    s = _silu(orc, x)
    assert np.all(s[x > 0] > 0) and np.all(s[x < 0] < 0)
    mid = (np.abs(x) < 16) & (x != 0)
    assert np.all(np.abs(s[mid]) < np.abs(x[mid]))


def test_swiglu_against_closed_form_values(orc):
    """silu(x) = x / (1 + e^-x) against values of the same function evaluated in
    f64 by Python's math.exp: within 2 f32 ulps (expf and the f32 division each
    round once)."""
    import math
    xs = np.array([-8.0, -2.5, -1.0, -0.5, 0.25, 1.0, 3.0, 7.5], np.float32)
    ref = np.array([float(v) / (1.0 + math.exp(-float(v))) for v in xs])
    got = _silu(orc, xs).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * np.spacing(np.abs(ref).astype(np.float32)))



# ------------------------------------------------------- q5_K and q8_0 ----

def test_q5K_values_every_position(orc):
    """Every 5-bit value at every position reads back (the fifth bit of element
    32j+i is bit j of qh[i]); the low nibbles sit where q4_K keeps them."""
    rng = np.random.default_rng(21)
    for rep in range(40):
        q = (np.arange(256) * 7 + rep) % 32 if rep < 32 else rng.integers(0, 32, 256)
        blk = pack_q5K_block(1.0, 0.0, [1] * 8, [0] * 8, q)
        assert np.array_equal(orc.q5K_quants(blk), q)
        assert np.array_equal(blk[48:], pack_q4K_qs(np.asarray(q) & 15))


def test_q5K_high_bits_one_at_a_time(orc):
    """Setting one bit of qh moves exactly one element up by 16."""
    base = pack_q5K_block(1.0, 0.0, [1] * 8, [0] * 8, np.zeros(256, np.int64))
    for i in range(32):
        for j in range(8):
            blk = base.copy()
            blk[16 + i] = 1 << j
            want = np.zeros(256, np.int64)
            want[32 * j + i] = 16
            assert np.array_equal(orc.q5K_quants(blk), want)


def test_q5K_one_hot_reads_back_weights(orc):
    rng = np.random.default_rng(22)
    q = rng.integers(0, 32, 256)
    sc = rng.integers(0, 64, 8)
    m = rng.integers(0, 64, 8)
    blk = pack_q5K_block(1.0, 1.0, sc, m, q)
    x = 127.0 * np.eye(256, dtype=np.float32)
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm("q5_K", blk, qs, ds, 1)[:, 0]
    want = np.array([sc[k // 32] * q[k] - m[k // 32] for k in range(256)], np.float64)
    assert np.array_equal(y / 127.0, want)
    assert np.array_equal(orc.dequant("q5_K", blk, 1, 256)[0], want)


def test_q5K_single_superblock_closed_form(orc):
    """All 5-bit values 17 (both the low nibble and the fifth bit in use), d =
    dmin = 1, X = 127: C = 127*17*32 = 69088 per sub-block, so
    Y = 69088*sum(sc) - 4064*sum(m) = 69088*259 - 4064*261 = 16,833,088 (even,
    so exact in f32 above 2^24)."""
    sc = [63, 1, 32, 17, 48, 5, 60, 33]
    m = [0, 63, 16, 47, 31, 62, 2, 40]
    blk = pack_q5K_block(1.0, 1.0, sc, m, np.full(256, 17))
    x = np.full((1, 256), 127.0, np.float32)
    qs, ds = orc.quantize_q8_1(x)
    assert np.all(orc.subdots("q5_K", blk, qs, 1) == 69088)
    assert orc.gemm("q5_K", blk, qs, ds, 1)[0, 0] == 16833088.0
    assert orc.gemm_dequant("q5_K", blk, qs, ds, 1)[0, 0] == 16833088.0


def test_q8_0_every_byte_value(orc):
    """Every int8 value at every position of a block reads back, with its d."""
    for shift in range(0, 256, 32):
        q = ((np.arange(32) + shift) % 256) - 128
        blk = pack_q8_0_block(0.5, q)
        d, got = orc.q8_0_block(blk)
        assert d == 0.5 and np.array_equal(got, q)


def test_q8_0_one_hot_reads_back_weights(orc):
    """K = 256 (8 blocks with different d): Y/127 = d_b * q for every k."""
    rng = np.random.default_rng(23)
    ds_w = [0.25, 0.5, 1.0, 2.0, 0.125, 4.0, 1.5, 0.75]
    qv = rng.integers(-128, 128, (8, 32))
    blk = np.concatenate([pack_q8_0_block(ds_w[b], qv[b]) for b in range(8)])
    x = 127.0 * np.eye(256, dtype=np.float32)
    qs, ds = orc.quantize_q8_1(x)
    y = orc.gemm("q8_0", blk, qs, ds, 1)[:, 0]
    want = np.array([ds_w[k // 32] * qv[k // 32, k % 32] for k in range(256)], np.float64)
    assert np.array_equal(y / 127.0, want)
    assert np.array_equal(orc.dequant("q8_0", blk, 1, 256)[0], want)


@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (2, 3, 256), (3, 2, 512)])
def test_q5K_q8_0_subdots_brute_force(orc, T, O, K):
    rng = np.random.default_rng(T * 100 + O * 10 + K + 1)
    nsb = K // 256
    q5 = rng.integers(0, 32, (O, K))
    q8 = rng.integers(-128, 128, (O, K))
    w5 = np.concatenate([pack_q5K_block(1.0, 1.0, rng.integers(0, 64, 8), rng.integers(0, 64, 8),
                                        q5[o, 256 * s: 256 * s + 256]) for o in range(O) for s in range(nsb)])
    w8 = np.concatenate([pack_q8_0_block(1.0, q8[o, 32 * b: 32 * b + 32]) for o in range(O) for b in range(K // 32)])
    a = rng.integers(-127, 128, (T, K)).astype(np.int8)
    got5 = orc.subdots("q5_K", w5, a, O)
    got8 = orc.subdots("q8_0", w8, a, O)
    for t in range(T):
        for o in range(O):
            for b in range(K // 32):
                sl = slice(32 * b, 32 * b + 32)
                assert got5[t, o, b] == int(np.dot(q5[o, sl], a[t, sl].astype(np.int64)))
                assert got8[t, o, b] == int(np.dot(q8[o, sl], a[t, sl].astype(np.int64)))
