"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: q8_1 values, scale words and per-sub-block integer dots bit-exact;
Y within max|Y_gpu - Y_ref| <= 2e-4 * max|Y_ref| (f32 accumulation order
differs from the oracle's f64 sum; f32 rounding alone stays near 1e-6).
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from quantized_prefill_gemm_mmq_gb300 import synth  # noqa: E402
from tests.kquant_pack import pack_q4K_block, pack_q5K_block, pack_q6K_block, pack_q8_0_block  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 2e-4


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_prefill_gemm_mmq_gb300 import ops as _ops
    from quantized_prefill_gemm_mmq_gb300 import _lib
    _lib.load()
    return _ops


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu_quant(ops, x):
    qs, ds, xh, xa = ops.quantize_q8_1(_dev(x))
    return qs, ds, xh, xa


def _to_np_ds(ds):
    return ds.cpu().numpy().view(np.uint32)


def _rel_err(y, ref):
    scale = float(np.abs(ref).max())
    return float(np.abs(y.astype(np.float64) - ref.astype(np.float64)).max()) / max(scale, 1e-30)


# -------------------------------------------------------------- q8_1 ----

@pytest.mark.parametrize("T,K,seed,outl", [(64, 512, 0, False), (37, 256, 1, True), (512, 4096, 10, True),
                                           (3, 11008, 21, True), (130, 768, 5, True)])
def test_quantize_bit_exact(ops, orc, T, K, seed, outl):
    x = synth.make_x(T, K, seed, outl)
    qs_r, ds_r = orc.quantize_q8_1(x)
    qs, ds, xh, xa = _gpu_quant(ops, x)
    ops.check_status()
    assert np.array_equal(qs.cpu().numpy(), qs_r)
    assert np.array_equal(_to_np_ds(ds), ds_r)
    assert np.array_equal(xh.cpu().numpy().astype(np.float32), qs_r.astype(np.float32))
    # xa: hi + lo reproduces the dequantised value f32(d16)*q exactly
    xa_np = xa.cpu().numpy().astype(np.float64)
    assert np.array_equal(xa_np[0] + xa_np[1], orc.dequant_q8_1(qs_r, ds_r))


def test_quantize_special_blocks(ops, orc):
    x = np.zeros((4, 128), np.float32)
    x[1, :32] = 127.0
    x[1, 1:6] = [2.5, -2.5, 0.5, -0.5, 1.5]
    x[2, 32:64] = np.float32(3e-7)              # tiny: d rounds into f16 subnormals
    x[2, 64] = -1e-30
    x[3, :] = np.linspace(-1000, 1000, 128, dtype=np.float32)
    qs_r, ds_r = orc.quantize_q8_1(x)
    qs, ds, xh, xa = _gpu_quant(ops, x)
    assert np.array_equal(qs.cpu().numpy(), qs_r)
    assert np.array_equal(_to_np_ds(ds), ds_r)
    xa_np = xa.cpu().numpy().astype(np.float64)
    assert np.array_equal(xa_np[0] + xa_np[1], orc.dequant_q8_1(qs_r, ds_r))


def test_quantize_near_half_integers(ops, orc):
    """Quotients x / d32 within ~2^-20 (relative) of half-integers, with block
    scales that are not powers of two, and blocks of tiny scale (d32 subnormal):
    the q8_1 codes and scale words must match the oracle's IEEE division and
    half-away rounding bit for bit."""
    rng = np.random.default_rng(7)
    T, nb = 64, 64
    x = np.zeros((T, nb * 32), np.float32)
    for t in range(T):
        for b in range(nb):
            amax = np.float32(rng.uniform(0.01, 1000.0)) if t < T - 4 else np.float32(rng.uniform(1e-43, 1e-37))
            d32 = np.float32(amax / np.float32(127.0))
            n = rng.integers(-127, 127, 31).astype(np.float64) + 0.5
            # half of the values inside the exact-division margin, half around it
            eps = rng.integers(-16, 17, 31) * np.where(rng.random(31) < 0.5, 2.0 ** -24, 2.0 ** -16)
            vals = (n * (1.0 + eps) * np.float64(d32)).astype(np.float32)
            vals = np.clip(vals, -amax, amax)
            blk = np.concatenate([[amax], vals]).astype(np.float32)
            rng.shuffle(blk)
            x[t, 32 * b:32 * b + 32] = blk
    qs_r, ds_r = orc.quantize_q8_1(x)
    qs, ds, _, _ = _gpu_quant(ops, x)
    assert np.array_equal(qs.cpu().numpy(), qs_r)
    assert np.array_equal(_to_np_ds(ds), ds_r)


def test_quantize_strided_rows(ops, orc):
    xfull = synth.make_x(50, 1024 + 64, 3)
    xt = _dev(xfull)[:, :1024]
    qs, ds, xh, xa = ops.quantize_q8_1(xt)
    qs_r, ds_r = orc.quantize_q8_1(xfull[:, :1024])
    assert np.array_equal(qs.cpu().numpy(), qs_r)
    assert np.array_equal(_to_np_ds(ds), ds_r)


# ---------------------------------------------------- sub-block dots ----

@pytest.mark.parametrize("fmt", ["q4_K", "q6_K", "q5_K", "q8_0"])
@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (64, 256, 512), (130, 200, 768), (200, 129, 256)])
def test_subdots_bit_exact(ops, orc, fmt, T, O, K):
    w = synth.make_weights(fmt, O, K, seed=T + O + K)
    x = synth.make_x(T, K, seed=O)
    qs_r, _ = orc.quantize_q8_1(x)
    _, _, xh, _ = _gpu_quant(ops, x)
    got = ops.debug_subdots(fmt, _dev(w), xh, O)
    ops.check_status()
    ref = orc.subdots(fmt, w, qs_r, O)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_subdots_extremes(ops, orc):
    # all-15 nibbles against all +-127 activations: the largest sub-block dots
    O, K, T = 3, 256, 4
    q = np.full(256, 15)
    w4 = np.concatenate([pack_q4K_block(1.0, 1.0, [63] * 8, [63] * 8, q)] * O)
    w6 = np.concatenate([pack_q6K_block(1.0, [-128] * 16, np.full(256, 63 if o % 2 else 0)) for o in range(O)])
    x = np.full((T, K), 127.0, np.float32)
    x[1] *= -1
    x[2, ::2] *= -1
    x[3, :] = 127.0 * ((np.arange(K) % 3) - 1)
    qs_r, _ = orc.quantize_q8_1(x)
    _, _, xh, _ = _gpu_quant(ops, x)
    assert np.array_equal(ops.debug_subdots("q4_K", _dev(w4), xh, O).cpu().numpy(), orc.subdots("q4_K", w4, qs_r, O))
    assert np.array_equal(ops.debug_subdots("q6_K", _dev(w6), xh, O).cpu().numpy(), orc.subdots("q6_K", w6, qs_r, O))


# -------------------------------------------------------------- GEMM ----

def _run_gemm(ops, fmt, w, x, O, kernel="production"):
    qs, ds, xh, xa = _gpu_quant(ops, x)
    if kernel == "production":
        y = ops.gemm(fmt, _dev(w), xa, ds, O)
    else:
        y = ops.gemm_subblock(fmt, _dev(w), xh, ds, O)
    ops.check_status()
    return y.cpu().numpy()


KERNELS = [("q4_K", "production"), ("q4_K", "subblock"), ("q6_K", "production"), ("q6_K", "subblock"),
           ("q5_K", "production"), ("q5_K", "subblock"), ("q8_0", "subblock")]


@pytest.mark.parametrize("fmt,kernel", KERNELS)
@pytest.mark.parametrize("T,O,K", [(64, 256, 512), (1, 1, 256), (130, 300, 768), (129, 129, 1280),
                                   (256, 512, 2048), (300, 200, 1024), (640, 136, 512)])
def test_gemm_full_small(ops, orc, fmt, kernel, T, O, K):
    """Whole outputs against the oracle, ragged T and O; T = 300 and 640 give
    an odd number of 128-token tiles."""
    w = synth.make_weights(fmt, O, K, seed=7 * T + O)
    x = synth.make_x(T, K, seed=K + T, outliers=T > 1)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm(fmt, w, qs_r, ds_r, O)
    y = _run_gemm(ops, fmt, w, x, O, kernel)
    assert y.shape == ref.shape
    assert _rel_err(y, ref) <= TOL


@pytest.mark.parametrize("kernel", ["production", "subblock"])
def test_gemm_config0_tiny(ops, orc, kernel):
    g = synth.config(0).gemms[0]
    w, x = g.weights(), g.x()
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm(g.fmt, w, qs_r, ds_r, g.O)
    y = _run_gemm(ops, g.fmt, w, x, g.O, kernel)
    assert _rel_err(y, ref) <= TOL


@pytest.mark.parametrize("kernel", ["production", "subblock"])
def test_gemm_closed_form_superblock(ops, kernel):
    sc = [63, 1, 32, 17, 48, 5, 60, 33]
    m = [0, 63, 16, 47, 31, 62, 2, 40]
    q = np.array([(i % 32) % 16 for i in range(256)])
    w = pack_q4K_block(1.0, 1.0, sc, m, q)
    x = np.full((1, 256), 127.0, np.float32)
    y = _run_gemm(ops, "q4_K", w, x, 1, kernel)
    assert y[0, 0] == 6833616.0


@pytest.mark.parametrize("cfg,T", [(1, None), (2, None), (3, None), (4, 16), (4, 64), (4, 256), (4, 1024), (4, 4096)])
def test_gemm_full_size(ops, oracle_ref, cfg, T):
    """Every output of every GEMM of the 7B configurations and of the token
    sweep, production kernels (and the per-sub-block kernels on configs 1-3),
    element by element against the oracle."""
    wl = synth.config(cfg, T)
    for g in wl.gemms:
        qs_r, ds_r, ref = oracle_ref(g)
        qs, ds, xh, xa = _gpu_quant(ops, g.x())
        assert np.array_equal(qs.cpu().numpy(), qs_r)
        assert np.array_equal(_to_np_ds(ds), ds_r)
        wd = _dev(g.weights())
        outs = [("production", ops.gemm(g.fmt, wd, xa, ds, g.O))]
        if cfg in (1, 2, 3):
            outs.append(("subblock", ops.gemm_subblock(g.fmt, wd, xh, ds, g.O)))
        ops.check_status()
        for kernel, y in outs:
            err = _rel_err(y.cpu().numpy(), ref)
            assert err <= TOL, (g.name, kernel, err)


@pytest.mark.parametrize("T,O,K,ksplit", [(16, 256, 1024, 4), (1, 129, 2816, 3), (130, 300, 1280, 2),
                                          (64, 512, 4096, 16), (200, 128, 768, 7), (300, 256, 2048, 3)])
def test_gemm_splitk_small(ops, orc, T, O, K, ksplit):
    w = synth.make_weights("q4_K", O, K, seed=3 * T + O)
    x = synth.make_x(T, K, seed=K + T + 1, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    _, ds, _, xa = _gpu_quant(ops, x)
    ws = ops.SplitKWorkspace(xa.device, *ops.splitk_sizes(T, O, K, ksplit))
    y1 = ops.gemm_splitk(_dev(w), xa, ds, O, ksplit=ksplit, workspace=ws)
    y2 = ops.gemm_splitk(_dev(w), xa, ds, O, ksplit=ksplit, workspace=ws)
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)                       # fixed summation order
    assert int(ws.counters.abs().sum()) == 0         # counters left at zero


@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (16, 256, 1024), (5, 131, 2816), (17, 200, 768), (33, 512, 4096),
                                   (64, 8, 11008), (40, 1000, 512), (3, 20000, 512), (64, 4096, 256),
                                   (16, 384, 4352), (1, 2048, 11008)])
def test_gemm_small_t(ops, orc, T, O, K):
    """Weight-stationary small-T kernel: token tiles of 16, 32 and 64, clusters of
    1 to 8 CTAs per row tile (O = 20000: one CTA per tile), ragged T and O."""
    w = synth.make_weights("q4_K", O, K, seed=5 * T + O)
    x = synth.make_x(T, K, seed=K + 2 * T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    _, ds, _, xa = _gpu_quant(ops, x)
    y1 = ops.gemm_small(_dev(w), xa, ds, O)
    y2 = ops.gemm_small(_dev(w), xa, ds, O)
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)                       # fixed summation order


@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (16, 256, 1024), (5, 131, 2816), (13, 200, 768), (16, 512, 4096),
                                   (9, 8, 11008), (2, 1000, 512)])
def test_gemm_small_t_imma(ops, orc, T, O, K):
    w = synth.make_weights("q4_K", O, K, seed=5 * T + O)
    x = synth.make_x(T, K, seed=K + 2 * T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    qs, ds, _, _ = ops.quantize_q8_1(_dev(x), want_xh=False, want_xa=False)
    y1 = ops.gemm_small_imma(_dev(w), qs, ds, O)
    y2 = ops.gemm_small_imma(_dev(w), qs, ds, O)
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (8, 256, 1024), (9, 131, 2816), (16, 200, 768), (3, 17, 512),
                                   (16, 512, 4096), (5, 8, 11008), (1, 1000, 512), (12, 4096, 256), (7, 33, 3072)])
def test_gemv(ops, orc, T, O, K):
    """Decode-shaped kernel: one and two 8-token MMA tiles, ragged T and O
    (token slots past T and rows past O), K from 1 to 43 super-blocks (fewer
    super-blocks than ring stages, and more)."""
    w = synth.make_weights("q4_K", O, K, seed=3 * T + O)
    x = synth.make_x(T, K, seed=K + 5 * T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    _, ds, xh, _ = ops.quantize_q8_1(_dev(x), want_qs=False, want_xa=False)
    y1 = ops.gemv(_dev(w), xh, ds, O)
    y2 = ops.gemv(_dev(w), xh, ds, O)
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)                       # fixed summation order


@pytest.mark.parametrize("T", [1, 8, 16])
def test_gemv_full_size(ops, oracle_ref, T):
    """The token-sweep shapes (K = 4096 and 11008, O = 4096) at decode sizes,
    every output against the oracle."""
    for g in synth.config(4, T).gemms:
        _, _, ref = oracle_ref(g)
        _, ds, xh, _ = ops.quantize_q8_1(_dev(g.x()), want_qs=False, want_xa=False)
        y = ops.gemv(_dev(g.weights()), xh, ds, g.O)
        ops.check_status()
        assert _rel_err(y.cpu().numpy(), ref) <= TOL, g.name


@pytest.mark.parametrize("fmt", ["q4_K", "q6_K"])
@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (1, 7, 768), (2, 300, 512), (3, 33, 2816), (4, 64, 4096),
                                   (1, 5000, 256), (4, 9, 11008), (2, 1, 32768), (3, 257, 1280), (1, 2047, 4096),
                                   (1, 131, 2816), (2, 17, 512)])
def test_gemv_f32(ops, orc, fmt, T, O, K):
    """Decode product with the quantisation built in: every output against the
    oracle's quantise-then-GEMM; ragged O (partial last warp pass, more rows
    than resident warps at O = 5000), short last chunks (K = 11008: 43
    super-blocks), odd super-block counts, the largest K, T = 1..4 (T = 3 runs
    the 4-token instantiation with a padded token).  For q6_K the byte size of
    W, O*(K/256)*210, is 2, 4, 6, 8, 10, 12 or 14 mod 16 in most cases, so the
    last chunk's 16-byte window ends past W and its last bytes are read one by
    one."""
    w = synth.make_weights(fmt, O, K, seed=3 * T + O)
    x = synth.make_x(T, K, seed=K + 5 * T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm(fmt, w, qs_r, ds_r, O)
    y1 = ops.gemv_f32(_dev(w), _dev(x), O, fmt=fmt)
    y2 = ops.gemv_f32(_dev(w), _dev(x), O, fmt=fmt)
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)                       # fixed summation order


def test_gemv_f32_chained_launches(ops, orc):
    """Decode launches back to back on one stream, each reading the previous
    launch's output as its token: with programmatic dependent launch the next
    kernel starts before the previous one has finished and may read its
    weights early, but x only after the previous kernel has completed, and it
    writes y only then.  The chain must equal the same chain with a device
    synchronisation after every launch, bit for bit, and every link the
    oracle's product of the link's input."""
    O = K = 4096
    fmts = ["q4_K", "q6_K", "q4_K", "q4_K", "q6_K", "q4_K"]

    def tame(w, f):
        # the f16 scales of every block / 16 (exact), so that a link's output is of the
        # order of its input and six links stay in the f16 range of the q8_1 scales
        size, at = (144, (0, 4)) if f == "q4_K" else (210, (208, 210))
        b = w.reshape(-1, size)
        d = b[:, at[0]:at[1]].copy().view(np.float16) / np.float16(16)
        b[:, at[0]:at[1]] = d.astype(np.float16).view(np.uint8).reshape(b.shape[0], -1)
        return w

    ws = [_dev(tame(synth.make_weights(f, O, K, seed=500 + i), f)) for i, f in enumerate(fmts)]
    x0 = _dev(synth.make_x(1, K, seed=499))

    def chain(sync):
        y, outs = x0, []
        for w, f in zip(ws, fmts):
            y = ops.gemv_f32(w, y, O, fmt=f)
            outs.append(y)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return outs

    a, b = chain(False), chain(True)
    ops.check_status()
    for ya, yb in zip(a, b):
        assert torch.isfinite(ya).all() and ya.abs().max() > 0
        assert torch.equal(ya, yb)
    # every link against the oracle on the link's own input (its predecessor's output)
    prev = x0.cpu().numpy()
    for y, w, f in zip(a, ws, fmts):
        qs_r, ds_r = orc.quantize_q8_1(prev)
        ref = orc.gemm(f, w.cpu().numpy(), qs_r, ds_r, O)
        assert _rel_err(y.cpu().numpy(), ref) <= TOL
        prev = y.cpu().numpy()


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_q6K_f32_full_size(ops, orc, T):
    """The 7B attn_v shape (q6_K, K = O = 4096) with full-range int8 sub-block
    scales (-128..127), every output against the oracle."""
    rng = np.random.default_rng(6262 + T)
    O, K = 4096, 4096
    w = synth.make_weights("q6_K", O, K, seed=35 + T).reshape(O * (K // 256), 210)
    w[:, 192:208] = rng.integers(0, 256, size=(w.shape[0], 16), dtype=np.uint8)
    w = w.reshape(-1)
    x = synth.make_x(T, K, seed=36 + T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q6_K", w, qs_r, ds_r, O)
    y = ops.gemv_f32(_dev(w), _dev(x), O, fmt="q6_K")
    ops.check_status()
    assert _rel_err(y.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_f32_full_size(ops, orc, oracle_ref, T):
    """The 7B decode shapes: K = 4096 and 11008 at O = 4096 (config 4's GEMMs),
    and the chained gate+up rows (O = 22016, K = 4096), every output against
    the oracle; the built-in quantisation against mmq_quantize_q8_1 through the
    unfused path (the same sub-block dots, so the two agree to f32 rounding)."""
    for g in synth.config(4, T).gemms:
        _, _, ref = oracle_ref(g)
        y = ops.gemv_f32(_dev(g.weights()), _dev(g.x()), g.O)
        _, ds, xh, _ = ops.quantize_q8_1(_dev(g.x()), want_qs=False, want_xa=False)
        y_unfused = ops.gemv(_dev(g.weights()), xh, ds, g.O)
        ops.check_status()
        assert _rel_err(y.cpu().numpy(), ref) <= TOL, g.name
        assert _rel_err(y.cpu().numpy(), y_unfused.cpu().numpy()) <= 1e-6, g.name
    O, K = 22016, 4096
    w = synth.make_weights("q4_K", O, K, seed=71)
    x = synth.make_x(T, K, seed=72, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    y = ops.gemv_f32(_dev(w), _dev(x), O)
    ops.check_status()
    assert _rel_err(y.cpu().numpy(), ref) <= TOL


def test_gemv_f32_zero_and_extreme_tokens(ops, orc):
    """An all-zero token (q8_1 d = 0: every term 0), a token with one nonzero
    element per 32-block, and a token at +-1e4 (codes +-127): bit-exact codes
    through the built-in quantisation show up as exact agreement with the
    unfused path where every sub-block term is an exact f32 number."""
    O, K = 130, 1024
    w = synth.make_weights("q4_K", O, K, seed=81)
    x = np.zeros((4, K), np.float32)
    x[1, ::32] = np.arange(K // 32, dtype=np.float32) - 16.0
    x[2] = np.where(np.arange(K) % 2 == 0, 1e4, -1e4).astype(np.float32)
    x[3] = synth.make_x(1, K, seed=82)[0]
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q4_K", w, qs_r, ds_r, O)
    y = ops.gemv_f32(_dev(w), _dev(x), O).cpu().numpy()
    ops.check_status()
    assert np.all(y[0] == 0.0)
    assert _rel_err(y, ref) <= TOL


@pytest.mark.parametrize("T,O,K", [(1, 1, 256), (8, 256, 1024), (9, 131, 2816), (16, 200, 768), (3, 17, 512),
                                   (16, 512, 4096), (5, 8, 11008), (1, 1000, 512), (12, 33, 3072), (2, 7, 256)])
def test_gemv_q6K(ops, orc, T, O, K):
    """Decode-shaped q6_K kernel: one and two 8-token tiles, ragged T and O, K
    from 1 to 43 super-blocks; O*K/256*210 mod 16 takes the values 0, 2, 4, 8
    and 14, so in most cases the buffer ends inside the last block's
    16-byte-aligned window (its tail bytes copied one by one)."""
    w = synth.make_weights("q6_K", O, K, seed=7 * T + O)
    x = synth.make_x(T, K, seed=K + 11 * T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q6_K", w, qs_r, ds_r, O)
    _, ds, xh, _ = ops.quantize_q8_1(_dev(x), want_qs=False, want_xa=False)
    y1 = ops.gemv(_dev(w), xh, ds, O, fmt="q6_K")
    y2 = ops.gemv(_dev(w), xh, ds, O, fmt="q6_K")
    ops.check_status()
    assert _rel_err(y1.cpu().numpy(), ref) <= TOL
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T", [1, 16])
def test_gemv_q6K_full_size(ops, orc, T):
    """The 7B attn_v shape (q6_K, K = O = 4096) at decode sizes, full-range
    int8 sub-block scales (-128..127) as well as the synthetic -64..63, every
    output against the oracle."""
    rng = np.random.default_rng(6161 + T)
    O, K = 4096, 4096
    x = synth.make_x(T, K, seed=33 + T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    _, ds, xh, _ = ops.quantize_q8_1(_dev(x), want_qs=False, want_xa=False)
    w = synth.make_weights("q6_K", O, K, seed=34 + T)
    wf = w.reshape(O, K // 256, 210).copy()
    wf[: O // 2, :, 192:208] = rng.integers(0, 256, size=(O // 2, K // 256, 16), dtype=np.uint8)
    for wt in (w, wf.reshape(w.shape)):
        y = ops.gemv(_dev(wt), xh, ds, O, fmt="q6_K")
        ops.check_status()
        ref = orc.gemm("q6_K", wt, qs_r, ds_r, O)
        assert _rel_err(y.cpu().numpy(), ref) <= TOL


def test_gemv_closed_form_and_limits(ops):
    """The closed-form super-block (exact 6,833,616), and T = 17 refused."""
    from quantized_prefill_gemm_mmq_gb300._lib import MMQError
    sc = [63, 1, 32, 17, 48, 5, 60, 33]
    m = [0, 63, 16, 47, 31, 62, 2, 40]
    q = np.array([(i % 32) % 16 for i in range(256)])
    w = pack_q4K_block(1.0, 1.0, sc, m, q)
    x = np.full((1, 256), 127.0, np.float32)
    _, ds, xh, _ = ops.quantize_q8_1(_dev(x), want_qs=False, want_xa=False)
    assert float(ops.gemv(_dev(w), xh, ds, 1)[0, 0]) == 6833616.0
    x17 = synth.make_x(17, 256, seed=1)
    _, ds17, xh17, _ = ops.quantize_q8_1(_dev(x17), want_qs=False, want_xa=False)
    with pytest.raises(MMQError) as e:
        ops.gemv(_dev(w), xh17, ds17, 1)
    assert e.value.status == -1


@pytest.mark.parametrize("T", [16, 64])
def test_gemm_small_t_full_size(ops, oracle_ref, T):
    """The small-T kernels on the token-sweep shapes, every output against the oracle."""
    for g in synth.config(4, T).gemms:
        _, _, ref = oracle_ref(g)
        qs, ds, _, xa = ops.quantize_q8_1(_dev(g.x()), want_xh=False)
        w = _dev(g.weights())
        outs = [("small", ops.gemm_small(w, xa, ds, g.O))]
        if T <= ops.SMALL_IMMA_T_MAX:
            outs.append(("small_imma", ops.gemm_small_imma(w, qs, ds, g.O)))
        ops.check_status()
        for kernel, y in outs:
            assert _rel_err(y.cpu().numpy(), ref) <= TOL, (g.name, kernel)


def test_gemm_small_t_closed_form(ops):
    sc = [63, 1, 32, 17, 48, 5, 60, 33]
    m = [0, 63, 16, 47, 31, 62, 2, 40]
    q = np.array([(i % 32) % 16 for i in range(256)])
    w = pack_q4K_block(1.0, 1.0, sc, m, q)
    x = np.full((1, 256), 127.0, np.float32)
    qs, ds, _, xa = ops.quantize_q8_1(_dev(x), want_xh=False)
    assert float(ops.gemm_small(_dev(w), xa, ds, 1)[0, 0]) == 6833616.0
    assert float(ops.gemm_small_imma(_dev(w), qs, ds, 1)[0, 0]) == 6833616.0


@pytest.mark.parametrize("T", [16, 64, 256])
def test_gemm_splitk_full_size(ops, oracle_ref, T):
    """Split-K on the token-sweep shapes, every output against the oracle."""
    for g in synth.config(4, T).gemms:
        _, _, ref = oracle_ref(g)
        _, ds, _, xa = ops.quantize_q8_1(_dev(g.x()), want_qs=False, want_xh=False)
        y = ops.gemm_splitk(_dev(g.weights()), xa, ds, g.O)
        ops.check_status()
        assert _rel_err(y.cpu().numpy(), ref) <= TOL, g.name


@pytest.mark.parametrize("kernel", ["production", "subblock"])
@pytest.mark.parametrize("T,O,K", [(64, 256, 512), (130, 300, 768), (512, 128, 4096)])
def test_gemm_q6K_full_range_scales(ops, orc, kernel, T, O, K):
    # int8 sub-block scales over the whole -128..127 range (as real q6_K data
    # has), so that sc*(q-32) reaches +-4096 and needs the weight lo plane
    w = synth.make_weights("q6_K", O, K, seed=11 * T + O).reshape(O, K // 256, 210).copy()
    rng = np.random.default_rng(T + O + K)
    w[:, :, 192:208] = rng.integers(-128, 128, size=(O, K // 256, 16), dtype=np.int64).astype(np.int8).view(np.uint8)
    w[:, 0, 192] = np.uint8(0x80)                 # -128 in every row
    w = w.reshape(-1)
    x = synth.make_x(T, K, seed=K - T, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q6_K", w, qs_r, ds_r, O)
    y = _run_gemm(ops, "q6_K", w, x, O, kernel)
    assert _rel_err(y, ref) <= TOL


def test_gemm_repeatable(ops):
    g = synth.config(1).gemms[0]
    w = _dev(g.weights())
    _, ds, xh, xa = ops.quantize_q8_1(_dev(g.x()))
    y1 = ops.gemm(g.fmt, w, xa, ds, g.O)
    y2 = ops.gemm(g.fmt, w, xa, ds, g.O)
    g6 = synth.config(3).gemms[0]
    w6 = _dev(g6.weights())
    _, ds6, _, xa6 = ops.quantize_q8_1(_dev(g6.x()))
    v1 = ops.gemm(g6.fmt, w6, xa6, ds6, g6.O)
    v2 = ops.gemm(g6.fmt, w6, xa6, ds6, g6.O)
    z1 = ops.gemm_subblock(g.fmt, w, xh, ds, g.O)
    z2 = ops.gemm_subblock(g.fmt, w, xh, ds, g.O)
    ops.check_status()
    assert torch.equal(y1, y2) and torch.equal(z1, z2) and torch.equal(v1, v2)


def test_pipelines_repeatable_under_graph_replay(ops):
    """Many back-to-back launches of the production q4_K GEMM and of the
    small-T GEMM (tiles of 16, 32 and 64 tokens), replayed from a CUDA graph
    with timing events between the launches: no pipeline wait may give up and
    every launch must reproduce the first result bit for bit (the kernels
    fix their accumulation order).  Guards the barrier-phase bookkeeping of
    the rings shared by alternating MMA issuers."""
    g = synth.config(1).gemms[0]
    w = _dev(g.weights())
    _, ds, _, xa = ops.quantize_q8_1(_dev(g.x()))
    cases = [(w, xa, ds, g.O, ops.gemm("q4_K", w, xa, ds, g.O), "prod")]
    for i, T in enumerate((16, 32, 64)):
        ws = _dev(synth.make_q4K(1024, 4096, 40 + i))
        _, dss, _, xas = ops.quantize_q8_1(_dev(synth.make_x(T, 4096, 50 + i)))
        cases.append((ws, xas, dss, 1024, ops.gemm_small(ws, xas, dss, 1024), "small"))
    outs = [[torch.empty_like(c[4]) for _ in range(4)] for c in cases]
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * len(cases) * 4)]

    def body():
        e = 0
        for j in range(4):
            for c, o in zip(cases, outs):
                evs[e].record()
                if c[5] == "prod":
                    ops.gemm("q4_K", c[0], c[1], c[2], c[3], out=o[j])
                else:
                    ops.gemm_small(c[0], c[1], c[2], c[3], out=o[j])
                evs[e + 1].record()
                e += 2

    body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            body()
    torch.cuda.current_stream().wait_stream(st)
    for r in range(200):
        graph.replay()
        if r % 50 == 49:
            torch.cuda.synchronize()
            ops.check_status()
            for c, o in zip(cases, outs):
                assert all(torch.equal(c[4], oj) for oj in o), c[5]


def test_gpu_argument_errors(ops):
    from quantized_prefill_gemm_mmq_gb300._lib import MMQError
    w = torch.zeros(144 * 2, dtype=torch.uint8, device="cuda")
    xa = torch.zeros((2, 4, 512), dtype=torch.float16, device="cuda")
    ds = torch.zeros((4, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        ops.gemm("q4_K", w, xa, ds, 2)        # wrong weight size for O=2, K=512 is 576 bytes
    w2 = torch.zeros(144 * 4 + 4, dtype=torch.uint8, device="cuda")[4:]
    with pytest.raises(MMQError) as e:
        ops.gemm("q4_K", w2, xa, ds, 2)       # misaligned weight pointer
    assert e.value.status == -2


def test_gemm_concatenated_rows_equal_separate(ops):
    """One GEMM over the concatenated rows of two weight matrices that share an
    input gives, column block for column block, exactly the two GEMMs' outputs
    (each 128 x 128 output tile depends only on its own weight rows); the
    benchmark's gate/up projections run this way."""
    T, K = 512, 4096
    O1, O2 = 11008, 11008
    w1 = synth.make_weights("q4_K", O1, K, seed=71)
    w2 = synth.make_weights("q4_K", O2, K, seed=72)
    x = synth.make_x(T, K, seed=73, outliers=True)
    _, ds, _, xa = ops.quantize_q8_1(_dev(x), want_qs=False, want_xh=False)
    y1 = ops.gemm("q4_K", _dev(w1), xa, ds, O1)
    y2 = ops.gemm("q4_K", _dev(w2), xa, ds, O2)
    y12 = ops.gemm("q4_K", _dev(np.concatenate([w1, w2])), xa, ds, O1 + O2)
    ops.check_status()
    assert torch.equal(y12[:, :O1], y1)
    assert torch.equal(y12[:, O1:], y2)


def _full_check(orc, fmt, w, x, O, ys):
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm(fmt, w, qs_r, ds_r, O)
    for name, y in ys:
        assert torch.isfinite(y).all(), name
        assert _rel_err(y.cpu().numpy(), ref) <= TOL, (name, _rel_err(y.cpu().numpy(), ref))


def test_gemm_max_k(ops, orc):
    """K at the library's limit (2^20: 4096 super-blocks per row): long
    accumulation in every q4_K and q6_K GEMM form, every output against the
    oracle."""
    T, O, K = 4, 128, 1 << 20
    x = synth.make_x(T, K, seed=91, outliers=True)
    qs, ds, xh, xa = _gpu_quant(ops, x)
    qs_r, ds_r = orc.quantize_q8_1(x)
    assert np.array_equal(qs.cpu().numpy(), qs_r)
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_r)
    w4 = synth.make_weights("q4_K", O, K, seed=92)
    wd = _dev(w4)
    ys = [("production", ops.gemm("q4_K", wd, xa, ds, O)),
          ("splitk", ops.gemm_splitk(wd, xa, ds, O, ksplit=8)),
          ("small", ops.gemm_small(wd, xa, ds, O)),
          ("small_imma", ops.gemm_small_imma(wd, qs, ds, O)),
          ("gemv", ops.gemv(wd, xh, ds, O))]
    ops.check_status()
    _full_check(orc, "q4_K", w4, x, O, ys)
    w6 = synth.make_weights("q6_K", O, K, seed=93)
    y6 = ops.gemm("q6_K", _dev(w6), xa, ds, O)
    y6v = ops.gemv(_dev(w6), xh, ds, O, fmt="q6_K")
    ops.check_status()
    _full_check(orc, "q6_K", w6, x, O, [("q6_K production", y6), ("q6_K gemv", y6v)])


def test_gemm_large_o(ops, orc):
    """2^18 output rows (2048 row tiles, 37.7 MB of q4_K weights at K = 256):
    tile indexing and 64-bit offsets, every output against the oracle."""
    T, O, K = 3, 1 << 18, 256
    x = synth.make_x(T, K, seed=94, outliers=True)
    qs, ds, xh, xa = _gpu_quant(ops, x)
    w = synth.make_weights("q4_K", O, K, seed=95)
    wd = _dev(w)
    ys = [("production", ops.gemm("q4_K", wd, xa, ds, O)),
          ("small", ops.gemm_small(wd, xa, ds, O)),
          ("small_imma", ops.gemm_small_imma(wd, qs, ds, O)),
          ("gemv", ops.gemv(wd, xh, ds, O))]
    ops.check_status()
    _full_check(orc, "q4_K", w, x, O, ys)


# ------------------------------------------------ chained FFN (SwiGLU) ----

def _swiglu_gpu(ops, w_gate, w_up, x, F):
    w_gu = ops.interleave_gate_up(_dev(w_gate), _dev(w_up), F)
    _, ds, _, xa = ops.quantize_q8_1(_dev(x), want_qs=False, want_xh=False)
    hq, hd, hx = ops.gemm_swiglu(w_gu, xa, ds, F)
    ops.check_status()
    return hq.cpu().numpy(), hd.cpu().numpy().view(np.uint32), hx.cpu().numpy()


def _f16_scale(ds):
    return (ds & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)


def test_swiglu_exact_integers(ops, orc):
    """Gate and up outputs that are exact on both sides (power-of-two weight
    scales, integer activations with amax 127 in every block so that q = x,
    every partial sum an integer below 2^24 times the scale) and gate values
    >= 17, where e^-g is below half an f32 ulp of 1 and silu(g) = g exactly:
    h = g*u is then the same f32 on both sides, so the fused q8_1 codes, scale
    words and operand planes must equal the oracle's bit for bit.  Two 128-row
    tiles, ragged T."""
    rng = np.random.default_rng(11)
    T, F, K = 9, 128, 512
    nsb = K // 256
    w_gate = np.concatenate([pack_q4K_block(2.0 ** -12, 0.0, rng.integers(1, 8, 8), [0] * 8,
                                            rng.integers(1, 16, 256)) for _ in range(F * nsb)])
    w_up = np.concatenate([pack_q4K_block(2.0 ** -12, 2.0 ** -12, rng.integers(0, 8, 8), rng.integers(0, 64, 8),
                                          rng.integers(0, 16, 256)) for _ in range(F * nsb)])
    x = rng.integers(1, 128, (T, K)).astype(np.float32)
    x[:, ::32] = 127.0
    qs, ds = orc.quantize_q8_1(x)
    G = orc.gemm("q4_K", w_gate, qs, ds, F)
    U = orc.gemm("q4_K", w_up, qs, ds, F)
    assert G.min() >= 17 and np.array_equal(G * 4096, np.round(G * 4096)) and \
        np.array_equal(U * 4096, np.round(U * 4096))
    assert np.abs(G * U).max() < 65504            # the xa planes hold |v| within the f16 range
    qs_r, ds_r = orc.quantize_q8_1(orc.swiglu(G, U))
    hq, hd, hx = _swiglu_gpu(ops, w_gate, w_up, x, F)
    assert np.array_equal(hq, qs_r)
    assert np.array_equal(hd, ds_r)
    hx64 = hx.astype(np.float64)
    assert np.array_equal(hx64[0] + hx64[1], orc.dequant_q8_1(qs_r, ds_r))


def test_swiglu_config2_chain(ops, orc, oracle_ref):
    """The 7B FFN of config 2 (T = 512, K = 4096, F = 11008) through the fused
    gate/up + SwiGLU + q8_1 launch and then the down projection, against the
    oracle's gate and up GEMMs, its SwiGLU and its quantiser.
    Tolerance rule for the codes: the GPU's gate/up sums differ from the
    oracle's by at most the GEMM tolerance (TOL * max|G|, TOL * max|U|), which
    bounds |h_gpu - h_ref| per element by dh = 1.1 TOL max|G| |u| + |g| TOL max|U|
    (|silu'| <= 1.1, |silu(g)| <= |g|) plus an ulp.  A block's f16 scale may
    then differ by one f16 step, and a code may differ from the oracle's by one
    only where the oracle's quotient h/d lies within dh/d of a rounding
    boundary (n + 1/2); elsewhere codes are equal.  The down projection on the
    fused operands must match the oracle's down projection on its own codes
    within TOL."""
    gg, gu, gd = synth.config(2).gemms
    _, _, G = oracle_ref(gg)
    _, _, U = oracle_ref(gu)
    F = gg.O
    h = orc.swiglu(G, U)
    qs_r, ds_r = orc.quantize_q8_1(h)
    hq, hd, hx = _swiglu_gpu(ops, gg.weights(), gu.weights(), gg.x(), F)
    hx64 = hx.astype(np.float64)
    assert np.array_equal(hx64[0] + hx64[1], orc.dequant_q8_1(hq, hd))     # the planes match the codes
    d16_g, d16_r = (hd & 0xFFFF).astype(np.int64), (ds_r & 0xFFFF).astype(np.int64)
    assert np.all(np.abs(d16_g - d16_r) <= 1)
    same = np.repeat(d16_g == d16_r, 32, axis=1)
    d_r = np.repeat(_f16_scale(ds_r), 32, axis=1)
    dh = 1.1 * TOL * np.abs(G).max() * np.abs(U) + np.abs(G) * TOL * np.abs(U).max() + np.spacing(np.abs(h))
    qg, qr = hq.astype(np.int64), qs_r.astype(np.int64)
    diff = qg != qr
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = np.abs(h.astype(np.float64) / d_r)
        near = np.abs(quot - np.floor(quot) - 0.5) <= dh / d_r + 1e-6
    assert np.all(np.abs(qg - qr)[same] <= 1)
    assert np.all(near[diff & same])
    assert diff.mean() < 1e-3, diff.mean()
    yd = ops.gemm("q4_K", _dev(gd.weights()), _dev(hx), _dev(hd.view(np.int32)), gd.O)
    ops.check_status()
    ref_down = orc.gemm("q4_K", gd.weights(), qs_r, ds_r, gd.O)
    assert _rel_err(yd.cpu().numpy(), ref_down) <= TOL



# -------------------------------------------------------- q5_K, q8_0 ----

def test_subdots_extremes_q5K_q8_0(ops, orc):
    """The largest dots: 5-bit 31 everywhere, int8 -128 and 127, against +-127."""
    O, K, T = 3, 256, 4
    w5 = np.concatenate([pack_q5K_block(1.0, 1.0, [63] * 8, [63] * 8, np.full(256, 31))] * O)
    w8 = np.concatenate([pack_q8_0_block(1.0, np.full(32, -128 if o % 2 else 127)) for o in range(O) for _ in range(8)])
    x = np.full((T, K), 127.0, np.float32)
    x[1] *= -1
    x[2, ::2] *= -1
    x[3, :] = 127.0 * ((np.arange(K) % 3) - 1)
    qs_r, _ = orc.quantize_q8_1(x)
    _, _, xh, _ = _gpu_quant(ops, x)
    for fmt, w in (("q5_K", w5), ("q8_0", w8)):
        assert np.array_equal(ops.debug_subdots(fmt, _dev(w), xh, O).cpu().numpy(), orc.subdots(fmt, w, qs_r, O))


def test_q5K_closed_form_superblock(ops):
    """All 5-bit values 17, d = dmin = 1, X = 127: Y = 16,833,088 exactly."""
    sc = [63, 1, 32, 17, 48, 5, 60, 33]
    m = [0, 63, 16, 47, 31, 62, 2, 40]
    w = pack_q5K_block(1.0, 1.0, sc, m, np.full(256, 17))
    x = np.full((1, 256), 127.0, np.float32)
    assert float(_run_gemm(ops, "q5_K", w, x, 1, "production")[0, 0]) == 16833088.0
    assert float(_run_gemm(ops, "q5_K", w, x, 1, "subblock")[0, 0]) == 16833088.0


@pytest.mark.parametrize("fmt,kernel", [("q5_K", "production"), ("q5_K", "subblock"), ("q8_0", "subblock")])
def test_gemm_q5K_q8_0_7b_shape(ops, orc, fmt, kernel):
    """A 7B projection shape (T = 512, K = O = 4096) and the FFN down shape
    (K = 11008) with q5_K and q8_0 weights, every output against the oracle."""
    for (T, K, O, seed) in ((512, 4096, 4096, 61), (512, 11008, 4096, 62)):
        w = synth.make_weights(fmt, O, K, seed)
        x = synth.make_x(T, K, seed + 1, outliers=True)
        qs_r, ds_r = orc.quantize_q8_1(x)
        ref = orc.gemm(fmt, w, qs_r, ds_r, O)
        y = _run_gemm(ops, fmt, w, x, O, kernel)
        assert _rel_err(y, ref) <= TOL, (fmt, kernel, K)


def test_gemm_q8_0_buffer_end_and_zero_scales(ops, orc):
    """q8_0 rows whose last block ends the buffer (ragged O), blocks with d = 0,
    and full-range int8 values (-128 included)."""
    T, O, K = 33, 131, 768
    w = synth.make_weights("q8_0", O, K, 64).reshape(O, K // 32, 34).copy()
    rng = np.random.default_rng(65)
    w[:, :, 2:] = rng.integers(0, 256, size=(O, K // 32, 32), dtype=np.uint8)
    w[::3, 1, 0:2] = 0                                   # d = 0 in one block of every third row
    w = w.reshape(-1)
    x = synth.make_x(T, K, 66, outliers=True)
    qs_r, ds_r = orc.quantize_q8_1(x)
    ref = orc.gemm("q8_0", w, qs_r, ds_r, O)
    assert _rel_err(_run_gemm(ops, "q8_0", w, x, O, "subblock"), ref) <= TOL
