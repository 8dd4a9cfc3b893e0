/*
 * mmq.h -- C ABI of libmmq: the k-quant "MMQ" prefill GEMM on GB300 (sm_103a)
 *
 *     Y[T x O] = X[T x K] . W[O x K]^T
 *
 * with W stored in a k-quant format (q4_K, q6_K, q5_K) or q8_0 and X quantised per
 * 32-element block to q8_1.  The method is the one described on the
 * "minfer" CUDA optimisation pages for the q4_K MMQ line:
 *   - "31 . r28 -- Direction-A raw-nibble NB kernel, 2 blocks/SM", section
 *     2.3 "The numerics contract": the integer dot of unsigned 4-bit weights
 *     with int8 activations over each 32-weight sub-block, followed by the
 *     f32 two-term fold  sum += dx*(d*sc)*C + (dx*ssum)*(-(dmin*m)),
 *     stored f32 with no f16 between the dot and the store;
 *   - "19 . r14 -- B fragments via ldmatrix + widened scale reads", 3.2(d):
 *     the q8_1 activation scale pair (f16 d | int16 block sum);
 *   - "43 . r40 -- __launch_bounds__(256,3) third resident block", 5:
 *     q6_K, w = d*sc*(q-32) on 16-weight sub-blocks.
 *
 * Which call for which job
 * ------------------------
 *   prefill, T >= ~256 ....... mmq_gemm_q4K / mmq_gemm_q5K / mmq_gemm_q6K
 *                              (whole-super-block accumulation on the tensor
 *                              core; Y to the f32 tolerance, the sub-block
 *                              dots are never formed as numbers)
 *   FFN gate + up + SwiGLU ... mmq_gemm_q4K_swiglu (writes the down
 *                              projection's q8_1 operands)
 *   few output tiles ......... mmq_gemm_q4K_splitk (caller scratch) or
 *                              mmq_gemm_q4K_splitk_static (no allocation)
 *   17 <= T <= 64 ............ mmq_gemm_q4K_small
 *   T <= 4 (decode), f32 in .. mmq_gemv_q4K_f32 / mmq_gemv_q6K_f32 (q8_1
 *                              quantisation built in; per-sub-block integer
 *                              dots on the SIMT cores)
 *   T <= 16 (decode) ......... mmq_gemv_q4K / mmq_gemv_q6K (per-sub-block
 *                              integer dots, exact); mmq_gemm_q4K_small_imma
 *                              takes qs + ds as the pages' q8_1 does, at the
 *                              int8 warp-MMA rate
 *   the pages' literal form .. mmq_gemm_q4K_subblock / _q5K_subblock /
 *                              _q6K_subblock / mmq_gemm_q8_0 (one exact
 *                              integer dot per sub-block, folded in f32 per
 *                              sub-block); slower, kept as the reference form
 *                              on the GPU and for q8_0
 *   diagnostics .............. mmq_debug_subdots_* (the int32 dots themselves),
 *                              mmq_probe_tensor_peak, mmq_debug_fault_inject
 *                              (test-only)
 *
 * Conventions for every call
 * --------------------------
 *   - All array arguments are DEVICE pointers allocated and owned by the
 *     caller (for example PyTorch tensors).  The library allocates no
 *     device memory per call, keeps no pointer after the call returns and
 *     writes only the output arrays named below.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) on the current device.  A return value of
 *     MMQ_OK means the work was validated and launched, not that it has
 *     finished.  Kernel-side failures (a pipeline wait that exceeded its
 *     time limit) are reported by mmq_check_status().
 *   - Every pointer must be 16-byte aligned.  Inputs must be finite; the
 *     result for NaN or Inf inputs is unspecified.
 *   - The device must be compute capability 10.3 (GB300).
 *   - Return value: MMQ_OK (0) or a negative MMQ_ERR_* code; on error
 *     nothing is launched and no output is written.
 *
 * Storage formats (little-endian, rows contiguous)
 * ------------------------------------------------
 *   q4_K super-block, 144 bytes per 256 weights of one row: f16 d (bytes
 *     0-1), f16 dmin (2-3), 12 bytes of packed 6-bit sub-block scales and
 *     mins (4-15, GGUF k-quant packing), 128 bytes of 4-bit quants (16-143);
 *     sub-block j (weights 32j..32j+31) is the low nibble (j even) or high
 *     nibble (j odd) of quant bytes 32*(j/2) .. 32*(j/2)+31.
 *     w = d*sc_j*q - dmin*m_j.
 *   q6_K super-block, 210 bytes: ql[128], qh[64], int8 scales[16], f16 d
 *     (GGUF order); w = d*sc_(e/16)*(q-32), q in 0..63.
 *   W: [O][K/256] super-blocks, O*(K/256)*bytes_per_block bytes in total.
 *   q8_1 activations, split-plane form of the pages' 40-byte block:
 *     qs  int8     [T][K]     quantised values, -127..127;
 *     xh  uint16   [T][K]     the same values as IEEE f16 (exact integers):
 *                             the operand of the per-sub-block kernels;
 *     xa  uint16   [2][T][K]  the dequantised value v = f32(d)*q as two f16
 *                             planes, hi = f16(v) then lo = f16(v - hi); both
 *                             are exact and hi + lo == v (v is a multiple of
 *                             2^-24 with at most 18 significant bits) as long
 *                             as |v| <= 65504, the f16 range (activations of
 *                             larger magnitude overflow the hi plane): the
 *                             operand of the production GEMMs;
 *     ds  uint32   [T][K/32]  low 16 bits: f16 d of the 32-block,
 *                             high 16 bits: int16 sum of its 32 values.
 *   Y: f32 [T][O], row-major, overwritten.
 */
#ifndef MMQ_H
#define MMQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *mmq_stream_t;   /* == cudaStream_t */

enum {
    MMQ_OK = 0,
    MMQ_ERR_SHAPE = -1,     /* a size is out of range (see each call)              */
    MMQ_ERR_ALIGN = -2,     /* a pointer or leading dimension is misaligned        */
    MMQ_ERR_ARCH = -3,      /* current device is not compute capability 10.3      */
    MMQ_ERR_LAUNCH = -4,    /* the CUDA runtime refused the launch                 */
    MMQ_ERR_TIMEOUT = -5,   /* (mmq_check_status) a kernel pipeline wait timed out */
    MMQ_ERR_NULL = -6,      /* a required pointer is NULL                          */
    MMQ_ERR_DRIVER = -7,    /* the driver could not build a TMA tensor map         */
    MMQ_ERR_CUDA = -8,      /* (mmq_check_status) a CUDA error is pending          */
    MMQ_ERR_SCRATCH = -9,   /* the call needs more than the library's static scratch */
    MMQ_ERR_DEVICE = -10    /* current device index >= 64 (the library's per-device tables) */
};

/* Library ABI version; bumped on any signature or format change. */
int mmq_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *mmq_status_str(int status);

/*
 * q8_1 quantisation of activations ("31 . r28", 3.2: the q8_1 blocks
 * carrying int8 values and the (f16 d | int16 ssum) pair).
 * For every token t and 32-block b of x[t][0..K):
 *   amax = max |x|;  d32 = amax/127 (IEEE f32 division);
 *   q = clamp(round_half_away_from_zero(x/d32), -127, 127) (IEEE division);
 *   ssum = sum of the 32 q;  stored d = f16(d32), round to nearest even.
 *   An all-zero block stores d = 0, q = 0, ssum = 0.
 * x:   f32, T rows of leading dimension ldx elements (ldx >= K, ldx % 4 == 0).
 * qs:  int8 [T][K] or NULL.   xh: f16 bits [T][K] or NULL.
 * xa:  f16 bits [2][T][K] or NULL.   (at least one of qs, xh, xa)
 * ds:  uint32 [T][K/32], required.
 * T >= 0 (T == 0 is a no-op), 32 <= K <= 2^20, K % 32 == 0.
 */
int mmq_quantize_q8_1(const float *x, int64_t ldx, int T, int K,
                      int8_t *qs, uint32_t *ds, uint16_t *xh, uint16_t *xa, mmq_stream_t stream);

/*
 * q4_K x q8_1 GEMM ("31 . r28", 2.3):  y[t][o] = sum over 32-weight
 * sub-blocks b of  dx_b*(d*sc_b)*C_b + (dx_b*ssum_b)*(-(dmin*m_b)),
 * C_b the exact integer dot of the 32 unsigned quants with the 32 int8
 * activations, i.e. sum_k dequant(W)[o][k]*dequant(X)[t][k]; accumulation
 * in f32 (rounding order unspecified).
 * Production form: the tensor core accumulates each 256-weight super-block
 * from the exact operands v = f32(d)*q (xa, hi + lo) and sc*q; d and the
 * dmin*m term are applied per super-block.
 * w: O*(K/256)*144 bytes.  xa, ds: as written by mmq_quantize_q8_1.
 * y: f32 [T][O], overwritten.
 * T >= 0, O >= 1, 256 <= K <= 2^20, K % 256 == 0.
 */
int mmq_gemm_q4K(const void *w, const uint16_t *xa, const uint32_t *ds,
                 float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * Split-K form of mmq_gemm_q4K for outputs with few 128 x 128 tiles (small T):
 * the super-blocks of each row are divided among up to `ksplit` CTAs per
 * output tile (ceil(K/256 / ksplit) each).  Every CTA writes its partial sums
 * to `part` [splits][T][O] f32; the last CTA of a tile to finish (counted in
 * counters[tile], tile = (t/128) * ceil(O/128) + o/128) adds the splits in
 * split order and writes y, so the result is the same on every call.  The
 * sum is the same mathematical Y as mmq_gemm_q4K's; only the f32 summation
 * order differs.
 * part, counters: caller-owned device scratch; mmq_splitk_sizes gives their
 * sizes.  counters (int32, 4-byte aligned) must be all zero before the first
 * call and are left all zero by every call whose kernel ran, one that timed
 * out included; after a call whose mmq_check_status is not MMQ_OK, y from that
 * call is undefined.  Two calls that use
 * the same part/counters at the same time (different streams) race.
 * ksplit == 1 is mmq_gemm_q4K (part and counters unused, may be NULL).
 * Limits as mmq_gemm_q4K; ksplit >= 1; part 16-byte aligned.
 */
int mmq_splitk_sizes(int T, int O, int K, int ksplit, int64_t *part_floats, int64_t *counters);
int mmq_gemm_q4K_splitk(const void *w, const uint16_t *xa, const uint32_t *ds, float *y,
                        int T, int O, int K, int ksplit, float *part, int *counters, mmq_stream_t stream);

/*
 * The 7B FFN's first half as one launch, chained into the down projection
 * (the pages' workload is whole-model prefill, "31 . r28", 5 "Results"; the
 * FFN activation is not printed there, so this follows the LLaMA-family
 * SwiGLU: h = silu(g) * u, silu(g) = g / (1 + e^-g)).
 *   g = X . W_gate^T and u = X . W_up^T are computed as mmq_gemm_q4K computes
 *   y; the epilogue then evaluates h in f32, one rounding per operation
 *   (expf, add, divide, multiply), and quantises h to q8_1 exactly as
 *   mmq_quantize_q8_1 quantises x: the outputs are the down projection's
 *   operands, ready for mmq_gemm_q4K with K = F.
 * w_gu: 2F q4_K rows, gate and up interleaved in groups of 64 rows: rows
 *   128j .. 128j+63 are gate rows 64j .. 64j+63 and rows 128j+64 .. 128j+127
 *   the up rows of the same features (O*(K/256)*144 bytes with O = 2F).
 * xa, ds: the input's planes as written by mmq_quantize_q8_1 (K columns).
 * h_xa: f16 bits [2][T][F] (hi, lo planes), h_ds: uint32 [T][F/32] (4-byte
 *   aligned), h_qs: int8 [T][F] or NULL; all written.
 * T >= 0, 64 <= F <= 2^20, F % 64 == 0, K as mmq_gemm_q4K.  Deterministic.
 */
int mmq_gemm_q4K_swiglu(const void *w_gu, const uint16_t *xa, const uint32_t *ds,
                        uint16_t *h_xa, uint32_t *h_ds, int8_t *h_qs,
                        int T, int F, int K, mmq_stream_t stream);

/*
 * q4_K GEMM for few tokens (1 <= T <= 64), where the GEMM is bound by
 * streaming W from HBM.  Same operands and result as mmq_gemm_q4K (xa, ds
 * from mmq_quantize_q8_1; y [T][O] f32, overwritten), computed with the
 * weight rows on the tensor core's 128-row side fed from tensor memory and
 * the (at most 64) tokens on the other; the per-super-block fold of
 * "31 . r28" (2.3), as in mmq_gemm_q4K.  Each 128-row tile is handled by a
 * cluster of up to 8 CTAs that split its super-blocks and add their partial
 * sums in a fixed order through distributed shared memory, so the result is
 * the same on every call.  Allocates nothing; no scratch.
 * T <= 64 (MMQ_ERR_SHAPE above), other limits as mmq_gemm_q4K.
 */
int mmq_gemm_q4K_small(const void *w, const uint16_t *xa, const uint32_t *ds, float *y,
                       int T, int O, int K, mmq_stream_t stream);

/*
 * q4_K GEMM for few tokens (1 <= T <= 16) on the int8 warp MMA: the pages'
 * per-sub-block form ("31 . r28", 2.3) with mma.sync m16n8k32 s8 (one
 * instruction per 32-weight sub-block, the nibbles used as int8 operands),
 * the exact integer dots C_b folded in f32 per sub-block.  qs: the int8 q8_1
 * values [T][K] and ds the scale words, both as written by
 * mmq_quantize_q8_1.  Result as mmq_gemm_q4K up to f32 summation order;
 * deterministic.  Allocates nothing.  Kept beside mmq_gemm_q4K_small as the
 * per-sub-block integer form of the same product.
 * T <= 16 (MMQ_ERR_SHAPE above), other limits as mmq_gemm_q4K.
 */
int mmq_gemm_q4K_small_imma(const void *w, const int8_t *qs, const uint32_t *ds, float *y,
                            int T, int O, int K, mmq_stream_t stream);

/*
 * Decode-shaped q4_K product for 1 <= T <= 16 tokens, where the whole cost is
 * reading W from HBM once.  The pages' per-sub-block form ("31 . r28", 2.3):
 * for every 32-weight sub-block the exact integer dot C_b of the 4-bit
 * quants with the int8 activations, folded in f32 as
 * (dx*(d*sc))*C_b + (dx*ssum)*(-(dmin*m)).  The dots run on the f16 warp MMA
 * with exact integer operands (every product and partial sum is an integer
 * below 2^24); one CTA per 16 weight rows streams the rows' super-blocks
 * through a shared-memory ring.
 * xh: the int8 q8_1 values as f16 [T][K] and ds the scale words [T][K/32],
 * both as written by mmq_quantize_q8_1.  y: f32 [T][O], overwritten.  Result
 * as mmq_gemm_q4K up to f32 summation order; the same on every call.
 * Allocates nothing.
 * Launched with programmatic stream serialisation: the kernel may start
 * while the previous kernel on `stream` is still running and reads the first
 * super-blocks of W before that kernel has completed (xh, ds and y are
 * touched only after it has).  So W must not be written by the kernel
 * launched immediately before on the same stream (weights written by a copy,
 * or by any earlier kernel, are fine).  The same holds for mmq_gemv_q6K.
 * T <= 16 (MMQ_ERR_SHAPE above), other limits as mmq_gemm_q4K.
 */
int mmq_gemv_q4K(const void *w, const uint16_t *xh, const uint32_t *ds, float *y,
                 int T, int O, int K, mmq_stream_t stream);

/*
 * Decode-shaped q4_K product for 1 <= T <= 4 tokens with the q8_1
 * quantisation of the f32 tokens built in: y = mmq_gemm_q4K applied to
 * mmq_quantize_q8_1(x), without the separate quantise launch.  Every CTA
 * quantises the tokens into shared memory with the same arithmetic as
 * mmq_quantize_q8_1 (bit-identical codes, scales and sums), then forms the
 * pages' per-sub-block exact integer dots ("31 . r28", 2.3) with __dp4a on
 * the SIMT cores and folds them in f32 as (dx*(d*sc))*C_b + (dx*ssum)*
 * (-(dmin*m)); one warp per weight row, the rows dealt over the CTAs so that
 * every SM streams the same share of W.  Result as mmq_gemm_q4K up to f32
 * summation order; the same on every call.  Allocates nothing.
 * x: f32 [T][ldx] (ldx >= K, ldx % 4 == 0), finite.  w: as mmq_gemm_q4K.
 * y: f32 [T][O], overwritten.  T <= 4, 256 <= K <= 32768, K % 256 == 0
 * (MMQ_ERR_SHAPE otherwise), O >= 1.
 * Launched with programmatic stream serialisation like mmq_gemv_q4K: W must
 * not be written by the kernel launched immediately before on the same
 * stream; x and y are touched only after that kernel has completed.
 */
int mmq_gemv_q4K_f32(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K,
                     mmq_stream_t stream);

/*
 * The same for q6_K ("43 . r40", 5: w = d*sc_u*(q-32) on 16-weight
 * sub-blocks; the pages' per-16 fold y += (dx*(d*sc_u))*C16_u with C16_u the
 * exact integer dot of (q - 32) with the int8 activations, __dp4a).  The
 * 210-byte blocks are only 2-byte aligned: every chunk is copied as the
 * 16-byte-aligned window around it, and the bytes of a window past the end
 * of W are read one by one, never beyond it.  w: O*(K/256)*210 bytes; other
 * arguments, limits and launch behaviour as mmq_gemv_q4K_f32.
 */
int mmq_gemv_q6K_f32(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K,
                     mmq_stream_t stream);

/*
 * Decode-shaped q6_K product for 1 <= T <= 16 tokens ("43 . r40", 5:
 * w = d*sc_u*(q-32) on 16-weight sub-blocks u with signed 8-bit scales): for
 * every sub-block the exact integer dot C16_u of (q-32) with the int8
 * activations, folded in f32 as (dx_b*(d*sc_u))*C16_u, b = u/2 the q8_1
 * block.  The dots run on the f16 warp MMA with exact integer operands; the
 * 210-byte blocks are staged through 16-byte-aligned windows.
 * w: O*(K/256)*210 bytes.  xh, ds: as for mmq_gemv_q4K.  y: f32 [T][O],
 * overwritten.  Result as mmq_gemm_q6K up to f32 summation order; the same on
 * every call.  Allocates nothing.
 * T <= 16 (MMQ_ERR_SHAPE above), other limits as mmq_gemm_q6K.
 */
int mmq_gemv_q6K(const void *w, const uint16_t *xh, const uint32_t *ds, float *y,
                 int T, int O, int K, mmq_stream_t stream);

/*
 * mmq_gemm_q4K_splitk without caller scratch: this entry point allocates
 * nothing.  The partial sums and tile counters live in the library's own
 * statically allocated device arrays, 4 Mi f32 (16 MiB) of partial sums and
 * 8192 tile counters per device.  (The pages have no counterpart: their
 * kernel never splits K.)
 *   - The scratch address is obtained once per device, with that device
 *     current, on the first call for that device that needs scratch (under a
 *     lock: first calls from several host threads are safe).  Make that
 *     first call before any stream capture.  The address belongs to the
 *     device's CUDA context of that moment: after cudaDeviceReset of the
 *     device, do not call this entry point again in the same process.
 *   - Calls with one split (ksplit == 1, or K == 256) need no scratch and
 *     run as mmq_gemm_q4K whatever their size.  Calls whose
 *     mmq_splitk_sizes exceed the scratch return MMQ_ERR_SCRATCH and
 *     launch nothing.
 *   - What must start at zero: the tile counters.  They are zero when the
 *     library is loaded, and every call that launched leaves them at zero
 *     when its kernel ends (a kernel that timed out included).  After a call
 *     whose mmq_check_status is not MMQ_OK, y from that call is undefined
 *     (an aborted split may have skipped its partial sums); the counters
 *     are still valid for the next call.
 *   - The scratch is shared by every call on the device: calls that may
 *     overlap in time (different streams, no ordering between them) race
 *     and give wrong results.  Order them on one stream.
 * Arguments, limits and result as mmq_gemm_q4K_splitk.
 */
int mmq_gemm_q4K_splitk_static(const void *w, const uint16_t *xa, const uint32_t *ds, float *y,
                               int T, int O, int K, int ksplit, mmq_stream_t stream);

/*
 * The same q4_K GEMM in the pages' per-sub-block form: the tensor core forms
 * every 32-weight sub-block's exact integer dot (times its 6-bit scale) in
 * its own TMEM accumulator and the f32 fold dx_b*C'_b runs per sub-block
 * ("31 . r28", 2.3 and 3.2).  xh: the int8 values as f16 (mmq_quantize_q8_1).
 * Same limits and result (up to f32 summation order) as mmq_gemm_q4K.
 */
int mmq_gemm_q4K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds,
                          float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * q6_K x q8_1 GEMM ("43 . r40", 5: w = d*sc_u*(q-32) on 16-weight
 * sub-blocks u):  y[t][o] = sum_k dequant(W)[o][k]*dequant(X)[t][k], i.e.
 * the pages' per-16 fold sum_u dx_(u/2)*(d*sc_u)*C16_u with C16_u the exact
 * integer dot of (q-32) with the int8 activations; accumulation in f32
 * (rounding order unspecified).
 * Production form: the tensor core accumulates each 256-weight super-block
 * from the exact activation planes xa (hi + lo) and the weight values
 * sc*(q-32) as exact f16 hi + lo planes (two MMAs per 16-k step, weight hi
 * and weight lo against both activation planes: every product exact in f32);
 * d is applied per super-block.
 * w: O*(K/256)*210 bytes.  xa: as written by mmq_quantize_q8_1.  ds: not
 * read (q6_K has no min term; may be NULL).  y: f32 [T][O], overwritten.
 * T >= 0, O >= 1, 256 <= K <= 2^20, K % 256 == 0.
 */
int mmq_gemm_q6K(const void *w, const uint16_t *xa, const uint32_t *ds,
                 float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * The same q6_K GEMM in the pages' per-sub-block form: the tensor core forms
 * every 16-weight half's exact integer dot C16_u = sum (q-32)*a (operand xh,
 * the int8 values as f16) in its own TMEM accumulator and the f32 fold
 * dx*(d*sc_u)*C16_u runs per 16-weight half.  Same limits and result (up to
 * f32 summation order) as mmq_gemm_q6K.
 */
int mmq_gemm_q6K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds,
                          float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * q5_K x q8_1 GEMM, the sibling of q4_K in the same k-quant family (the pages
 * run the "q4_K line" and "q6_K line" of one skeleton, "43 . r40", 6; the
 * q5_K bytes are the GGUF layout, a reading): 176-byte super-blocks of 256
 * weights, d and dmin (f16) and the 12 scale/min bytes exactly as q4_K,
 * qh[32] at bytes 16-47, qs[128] at 48-175; weight 32j+i of a super-block
 * has q = (q4_K's nibble of qs for element 32j+i) + 16 * (bit j of qh[i]),
 * 0..31, and w = d*sc_j*q - dmin*m_j.
 * The q4_K fold and the production form of mmq_gemm_q4K (sc*q <= 1953 is
 * exact in f16).  w: O*(K/256)*176 bytes; xa, ds, y, limits as mmq_gemm_q4K.
 * mmq_gemm_q5K_subblock: the pages' per-sub-block form (exact integer dots
 * C_b, f32 fold per 32-weight sub-block) from xh, as mmq_gemm_q4K_subblock.
 */
int mmq_gemm_q5K(const void *w, const uint16_t *xa, const uint32_t *ds,
                 float *y, int T, int O, int K, mmq_stream_t stream);
int mmq_gemm_q5K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds,
                          float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * q8_0 x q8_1 GEMM: 34-byte blocks of 32 weights (f16 d, then 32 int8 values,
 * w = d*q; GGUF's q8_0, a reading), rows of K/32 blocks.  The pages' fold
 * with the weight block's scale in place of d*sc and no min term:
 * y[t][o] = sum_b (dx_b*d_b)*C_b, C_b the exact integer dot of the 32 int8
 * weights with the 32 int8 activations, formed by the tensor core (exact f16
 * operands) per block and folded in f32.  xh, ds: as written by
 * mmq_quantize_q8_1.  w: O*(K/32)*34 bytes, K % 256 == 0; other limits as
 * mmq_gemm_q4K.
 */
int mmq_gemm_q8_0(const void *w, const uint16_t *xh, const uint32_t *ds,
                  float *y, int T, int O, int K, mmq_stream_t stream);

/*
 * Diagnostic: the per-sub-block exact integer dots the GEMMs fold, through
 * the same tensor-core pipeline.  out: int32 [T][O][K/32] for q4_K
 * (C_b = sum q*a over 32 weights) or [T][O][K/16] for q6_K
 * (C16_u = sum (q-32)*a over 16 weights).  Same shape limits as the GEMMs.
 * Meant for small shapes (the output is K/32 or K/16 times larger than y).
 */
int mmq_debug_subdots_q4K(const void *w, const uint16_t *xh, int32_t *out,
                          int T, int O, int K, mmq_stream_t stream);
int mmq_debug_subdots_q6K(const void *w, const uint16_t *xh, int32_t *out,
                          int T, int O, int K, mmq_stream_t stream);
/* The same for q5_K and q8_0: int32 [T][O][K/32]. */
int mmq_debug_subdots_q5K(const void *w, const uint16_t *xh, int32_t *out,
                          int T, int O, int K, mmq_stream_t stream);
int mmq_debug_subdots_q8_0(const void *w, const uint16_t *xh, int32_t *out,
                           int T, int O, int K, mmq_stream_t stream);

/*
 * Diagnostic: measured warp-level tensor throughput of the current device,
 * in TMAC/s (10^12 multiply-accumulates per second), for kind 0 = int8
 * (mma.sync m16n8k32 s8*s8->s32, the only int8 tensor path on sm_103a) or
 * kind 1 = f16 (mma.sync m16n8k16, f32 accumulate).  Synchronous: runs a
 * few hundred microseconds of probe kernels on `stream` and waits for them.
 * The reported figure is the denominator of "fraction of int8 peak".
 */
int mmq_probe_tensor_peak(int kind, double *tmacs, mmq_stream_t stream);

/*
 * Waits for `stream`, then reports and clears the library's device status
 * word for the current device: MMQ_OK, MMQ_ERR_TIMEOUT (a kernel's pipeline
 * wait ran past its limit; the kernel stopped early and its output is
 * invalid) or MMQ_ERR_CUDA (the stream reported a CUDA error).  If
 * `detail` is non-NULL it receives 4 ints: code, kernel id, wait site,
 * linear block index of the first failure.
 */
int mmq_check_status(mmq_stream_t stream, int *detail);

/*
 * Test-only: exercises the bounded pipeline waits (the pages' launcher never
 * runs over its limits silently, "31 . r28", 3.3 Pitfalls; the waits and
 * this knob are the library's own).  Sets, for the current device, the time a
 * kernel's pipeline wait may take before it gives up (wait_limit_us > 0; <= 0
 * restores the default of 2 s) and a mode: 0 = off; 1 = the production q4_K
 * kernels (mmq_gemm_q4K, mmq_gemm_q4K_splitk*, mmq_gemm_q5K) withhold the raw
 * weight copy of their second super-block (K >= 512), so the waits for it run
 * out: the kernel records MMQ_ERR_TIMEOUT (see mmq_check_status), stops every
 * role, drains the work it issued, frees its tensor memory and returns; its y
 * is undefined.  Synchronous with respect to the host.  Returns MMQ_OK,
 * MMQ_ERR_SHAPE (unknown mode) or MMQ_ERR_CUDA.  Leave it at mode 0 outside
 * tests.
 */
int mmq_debug_fault_inject(int mode, int wait_limit_us);

/*
 * More detail on the last failure that mmq_check_status reported (no
 * counterpart on the pages; a diagnostic of the library's own bounded waits): info
 * receives 4 ints: the time the failed wait had waited (microseconds), its
 * poll count, the phase parity it waited for and the waited barrier's
 * shared-memory address.  All zero if no failure was reported yet.  Returns
 * MMQ_OK, or MMQ_ERR_NULL for a NULL `info`.
 */
int mmq_last_failure_info(int *info);

#ifdef __cplusplus
}
#endif

#endif /* MMQ_H */
