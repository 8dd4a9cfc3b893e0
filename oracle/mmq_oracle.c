/*
 * mmq_oracle.c -- plain, slow CPU oracle for the k-quant MMQ prefill GEMM
 *                 Y[T x O] = X[T x K] . W[O x K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code with the CUDA library: every format
 * rule below is written out again here from the pages' statements.
 *
 * Sources (the "minfer" CUDA optimisation pages on the q4_K MMQ line):
 *   [r28]  "31 . r28 -- Direction-A raw-nibble NB kernel, 2 blocks/SM"
 *   [r14]  "19 . r14 -- B fragments via ldmatrix + widened scale reads"
 *   [r40]  "43 . r40 -- __launch_bounds__(256,3) third resident block"
 *
 * What is computed, and where it comes from:
 *   - q4_K element decode: [r28] 3.2 "Key code" (raw qs plane at byte +16
 *     of a 144-byte super-block, sub-block sg reads byte (sg>>1)*32+i, low
 *     nibble for even sg, high for odd, unsigned 0..15) and [r14] 3.2(b).
 *   - q4_K weight value w = d*sc*q - dmin*m: [r28] 2.3 "numerics contract".
 *   - two-term fold  sum += dx*dsv*C + (dx*ssum)*dmv  with dsv = d*sc,
 *     dmv = -(dmin*m): [r28] 2.3 and 3.2 (the SDS plane and the fold).
 *   - q8_1 activation block (int8 values, f16 d, int16 block sum):
 *     [r28] 3.2 (sda_q "d f16 | ssum i16") and [r14] 3.2(d).
 *   - q6_K: w = d*sc*(q-32) on 16-weight sub-blocks, two k16 halves per
 *     32-k chunk: [r40] 5 "Results" (item 4).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 q4_K header: d f16 at bytes 0-1, dmin f16 at 2-3, scales at 4-15.
 *   R2 6-bit scale/min packing of the 12 scale bytes: the GGUF k-quant
 *      packing (see q4K_scale_min below).  Parity unpinned with respect to
 *      GGUF interoperability: no GGUF sample exists to check against.
 *   R4 q6_K byte layout: the GGUF order ql[128], qh[64], scales[16], d.
 *      Parity unpinned with respect to GGUF interoperability, as R2.
 *   R5 q8_1 block sum is the exact integer sum of the int8 values.
 *   R6 q8_1 rounding: d32 = amax/127 (IEEE f32 division), q =
 *      round-half-away(x/d32) clamped to [-127,127] (IEEE f32 division),
 *      stored d = f16 round-to-nearest-even of d32; an all-zero block gets
 *      d = 0, q = 0, ssum = 0.
 *   R8 q6_K sub-block dot is taken on the centred value q-32.
 *   R15 q5_K layout (a sibling of q4_K in the same k-quant family; the pages
 *      name the family, not this member's bytes): the GGUF order, 176 bytes
 *      = d, dmin (f16), the 12 scale/min bytes packed as q4_K's (R2), qh[32]
 *      at +16 and qs[128] at +48; element 32j+i takes q4_K's nibble of qs
 *      (R3) as its low 4 bits and bit j of qh[i] as bit 4, so q is 0..31 and
 *      w = d*sc_j*q - dmin*m_j.  Parity unpinned w.r.t. GGUF interoperability.
 *   R16 q8_0 layout: 34 bytes per 32 weights, f16 d then 32 int8 values,
 *      w = d*q; blocks of a row contiguous.  Its dot follows the pages' fold
 *      with the scale d_w of the weight block in place of d*sc and no min
 *      term: y += (dx*d_w)*C_b, C_b the exact integer dot of the 32 int8
 *      weights with the 32 int8 activations.
 *   R14 FFN activation between the gate/up and down projections of the pages'
 *      7B workload ([r28] 5 "Results": whole-model prefill): the pages print
 *      none; the reading is the LLaMA-family SwiGLU h = silu(g) * u with
 *      silu(g) = g / (1 + e^-g), evaluated in f32 (the kernel's precision)
 *      one operation at a time, h then quantised to q8_1 like any activation.
 *   Method-form rounding: each fold term is evaluated in f32 exactly as
 *   written (no contraction: build with -ffp-contract=off), the terms are
 *   summed in f64 in sub-block order, and the result is rounded to f32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_QK 256
#define ORC_QK8 32
#define ORC_Q4K_BYTES 144
#define ORC_Q6K_BYTES 210
#define ORC_Q5K_BYTES 176
#define ORC_Q8_0_BYTES 34

/* ---------------------------------------------------------------- f16 -- */

/* IEEE binary16 -> binary32, from the encoding's definition:
 * exponent field 0: value = mantissa * 2^-24 (zero and subnormals);
 * 1..30: value = (1024 + mantissa) * 2^(exponent - 25); 31: inf / nan. */
float orc_f16_to_f32(uint16_t h)
{
    const int e = (h >> 10) & 31;
    const int m = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);
    return (h & 0x8000) ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even.  The magnitude is
 * divided by the f16 quantum of its binade (an exact power-of-two scaling
 * in f64), rounded to an integer with ties-to-even, and re-encoded; a carry
 * into the next binade falls out of the encoding by itself. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, 4);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    const uint32_t mag = bits & 0x7fffffffu;
    if (mag > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);   /* nan */
    if (mag == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);  /* inf */
    const double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);      /* rounds past 65504 */
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = r * 2^e2, r in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -14) {                /* subnormal range: quantum 2^-24 */
        const double n = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n);        /* n == 1024 -> min normal */
    }
    const double n = nearbyint(ldexp(a, 10 - E));     /* in [1024, 2048] */
    const uint32_t enc = ((uint32_t)(E + 15) << 10) + (uint32_t)n - 1024u;
    return (uint16_t)(sign | enc);
}

/* ------------------------------------------------------- q4_K decode -- */

/* Sub-block j (0..7) scale and min from the 12 packed bytes s[] (reading
 * R2, the GGUF k-quant packing):
 *   bytes 0..3 : low 6 bits = scale j (j<4);  top 2 bits = bits 4-5 of scale j+4
 *   bytes 4..7 : low 6 bits = min j   (j<4);  top 2 bits = bits 4-5 of min j+4
 *   bytes 8..11: low nibble = bits 0-3 of scale j+4, high nibble = bits 0-3
 *                of min j+4. */
void orc_q4K_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 0x3f;
        *m = s[4 + j] & 0x3f;
    } else {
        const int i = j - 4;
        *sc = (s[8 + i] & 0x0f) | ((s[i] >> 6) << 4);
        *m = (s[8 + i] >> 4) | ((s[4 + i] >> 6) << 4);
    }
}

/* Unsigned 4-bit quant of element e (0..255) of one 144-byte block. */
int orc_q4K_quant(const uint8_t *blk, int e)
{
    const int j = e / 32, i = e % 32;
    const uint8_t byte = blk[16 + 32 * (j / 2) + i];
    return (j % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
}

/* ------------------------------------------------------- q5_K decode -- */

/* 5-bit quant (0..31) of element e (0..255) of one 176-byte block (R15). */
int orc_q5K_quant(const uint8_t *blk, int e)
{
    const int j = e / 32, i = e % 32;
    const uint8_t byte = blk[48 + 32 * (j / 2) + i];
    const int lo = (j % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
    const int hi = (blk[16 + i] >> j) & 1;
    return lo | (hi << 4);
}

/* ------------------------------------------------------- q8_0 decode -- */

/* int8 quant of element i (0..31) of one 34-byte block (R16). */
int orc_q8_0_quant(const uint8_t *blk, int i)
{
    return (int)(int8_t)blk[2 + i];
}

float orc_q8_0_d(const uint8_t *blk)
{
    return orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
}

/* ------------------------------------------------------- q6_K decode -- */

/* 6-bit quant (0..63) of element e (0..255) of one 210-byte block
 * (reading R4).  Within half h (elements 128h..128h+127) with
 * L = ql + 64h and H = qh + 32h, element 128h + 32*g + l (l < 32) takes
 *   g=0: low nibble of L[l],     bits 0-1 of H[l]
 *   g=1: low nibble of L[l+32],  bits 2-3 of H[l]
 *   g=2: high nibble of L[l],    bits 4-5 of H[l]
 *   g=3: high nibble of L[l+32], bits 6-7 of H[l]
 * with the H bits as bits 4-5 of the result. */
int orc_q6K_quant(const uint8_t *blk, int e)
{
    const int h = e / 128, g = (e % 128) / 32, l = e % 32;
    const uint8_t *L = blk + 64 * h;
    const uint8_t *H = blk + 128 + 32 * h;
    const uint8_t lbyte = (g == 0 || g == 2) ? L[l] : L[l + 32];
    const int lo = (g < 2) ? (lbyte & 0x0f) : (lbyte >> 4);
    const int hi = (H[l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

int orc_q6K_scale(const uint8_t *blk, int u)
{
    return (int)(int8_t)blk[192 + u];
}

float orc_q6K_d(const uint8_t *blk)
{
    return orc_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8)));
}

/* d and dmin of a q4_K or q5_K block (the first four bytes, R1). */
static float q4K_d(const uint8_t *blk)
{
    return orc_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
}

static float q4K_dmin(const uint8_t *blk)
{
    return orc_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
}

/* ---------------------------------------------------------- dequant -- */

/* W[o][k] as f64: d*sc*q - dmin*m, every factor exact, so the product is
 * exact in f64 ([r28] 2.3). */
void orc_dequant_q4K(const uint8_t *w, int O, int K, double *out)
{
    const int nsb = K / ORC_QK;
    for (int o = 0; o < O; ++o)
        for (int sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = w + ((size_t)o * nsb + sb) * ORC_Q4K_BYTES;
            const double d = q4K_d(blk), dmin = q4K_dmin(blk);
            for (int e = 0; e < ORC_QK; ++e) {
                int sc, m;
                orc_q4K_scale_min(blk + 4, e / 32, &sc, &m);
                out[(size_t)o * K + (size_t)sb * ORC_QK + e] =
                    d * sc * orc_q4K_quant(blk, e) - dmin * m;
            }
        }
}

/* W[o][k] as f64: d*sc*q - dmin*m with 5-bit q (R15). */
void orc_dequant_q5K(const uint8_t *w, int O, int K, double *out)
{
    const int nsb = K / ORC_QK;
    for (int o = 0; o < O; ++o)
        for (int sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = w + ((size_t)o * nsb + sb) * ORC_Q5K_BYTES;
            const double d = q4K_d(blk), dmin = q4K_dmin(blk);
            for (int e = 0; e < ORC_QK; ++e) {
                int sc, m;
                orc_q4K_scale_min(blk + 4, e / 32, &sc, &m);
                out[(size_t)o * K + (size_t)sb * ORC_QK + e] = d * sc * orc_q5K_quant(blk, e) - dmin * m;
            }
        }
}

/* W[o][k] as f64: d*q (R16). */
void orc_dequant_q8_0(const uint8_t *w, int O, int K, double *out)
{
    const int nb = K / 32;
    for (int o = 0; o < O; ++o)
        for (int b = 0; b < nb; ++b) {
            const uint8_t *blk = w + ((size_t)o * nb + b) * ORC_Q8_0_BYTES;
            const double d = orc_q8_0_d(blk);
            for (int i = 0; i < 32; ++i)
                out[(size_t)o * K + (size_t)b * 32 + i] = d * orc_q8_0_quant(blk, i);
        }
}

/* W[o][k] as f64: d*sc*(q-32) ([r40] 5). */
void orc_dequant_q6K(const uint8_t *w, int O, int K, double *out)
{
    const int nsb = K / ORC_QK;
    for (int o = 0; o < O; ++o)
        for (int sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = w + ((size_t)o * nsb + sb) * ORC_Q6K_BYTES;
            const double d = orc_q6K_d(blk);
            for (int e = 0; e < ORC_QK; ++e)
                out[(size_t)o * K + (size_t)sb * ORC_QK + e] =
                    d * orc_q6K_scale(blk, e / 16) * (orc_q6K_quant(blk, e) - 32);
        }
}

/* ----------------------------------------------------------- q8_1 ---- */

/* Quantise X[T][ldx] (first K columns) to q8_1, reading R5/R6.
 * qs: [T][K] int8.  ds: [T][K/32], low 16 bits = f16 d, high 16 = int16
 * block sum. */
void orc_quantize_q8_1(const float *x, int64_t ldx, int T, int K,
                       int8_t *qs, uint32_t *ds)
{
    const int nb = K / ORC_QK8;
    for (int t = 0; t < T; ++t)
        for (int b = 0; b < nb; ++b) {
            const float *xb = x + (size_t)t * ldx + (size_t)b * ORC_QK8;
            int8_t *qb = qs + (size_t)t * K + (size_t)b * ORC_QK8;
            float amax = 0.0f;
            for (int i = 0; i < ORC_QK8; ++i)
                if (fabsf(xb[i]) > amax) amax = fabsf(xb[i]);
            int ssum = 0;
            float d32 = 0.0f;
            if (amax == 0.0f) {
                for (int i = 0; i < ORC_QK8; ++i) qb[i] = 0;
            } else {
                d32 = amax / 127.0f;
                for (int i = 0; i < ORC_QK8; ++i) {
                    long q = lroundf(xb[i] / d32);   /* ties away from zero */
                    if (q > 127) q = 127;
                    if (q < -127) q = -127;
                    qb[i] = (int8_t)q;
                    ssum += (int)q;
                }
            }
            const uint16_t d16 = orc_f32_to_f16(d32);
            ds[(size_t)t * nb + b] = (uint32_t)d16 | ((uint32_t)(uint16_t)(int16_t)ssum << 16);
        }
}

/* ------------------------------------------------- sub-block dots ---- */

/* C[j] = sum_i q(32j+i) * a(32j+i), the exact integer dot of one 32-weight
 * q4_K sub-block ([r28] 2.3: unsigned nibble times int8 activation). */
static int32_t subdot_q4K(const uint8_t *blk, int j, const int8_t *a)
{
    int32_t c = 0;
    for (int i = 0; i < 32; ++i)
        c += orc_q4K_quant(blk, 32 * j + i) * (int32_t)a[32 * j + i];
    return c;
}

/* C16[u] = sum_i (q(16u+i) - 32) * a(16u+i), reading R8. */
static int32_t subdot_q6K(const uint8_t *blk, int u, const int8_t *a)
{
    int32_t c = 0;
    for (int i = 0; i < 16; ++i)
        c += (orc_q6K_quant(blk, 16 * u + i) - 32) * (int32_t)a[16 * u + i];
    return c;
}

/* C[j] over a 32-weight q5_K sub-block: 5-bit quant times int8 activation. */
static int32_t subdot_q5K(const uint8_t *blk, int j, const int8_t *a)
{
    int32_t c = 0;
    for (int i = 0; i < 32; ++i)
        c += orc_q5K_quant(blk, 32 * j + i) * (int32_t)a[32 * j + i];
    return c;
}

/* C_b of a q8_0 block: int8 weight times int8 activation over 32 (R16). */
static int32_t subdot_q8_0(const uint8_t *blk, const int8_t *a)
{
    int32_t c = 0;
    for (int i = 0; i < 32; ++i) c += orc_q8_0_quant(blk, i) * (int32_t)a[i];
    return c;
}

/* out: [T][O][K/32] int32 (q5_K and q8_0: fmt 5 / 8). */
void orc_subdots_b32(int fmt, const uint8_t *w, const int8_t *qs, int T, int O, int K, int32_t *out)
{
    const int nb = K / 32;
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < O; ++o)
            for (int b = 0; b < nb; ++b) {
                const int8_t *a = qs + (size_t)t * K;
                int32_t c;
                if (fmt == 5) {
                    const uint8_t *blk = w + ((size_t)o * (K / ORC_QK) + b / 8) * ORC_Q5K_BYTES;
                    c = subdot_q5K(blk, b % 8, a + (size_t)(b / 8) * ORC_QK);
                } else {
                    const uint8_t *blk = w + ((size_t)o * nb + b) * ORC_Q8_0_BYTES;
                    c = subdot_q8_0(blk, a + (size_t)b * 32);
                }
                out[((size_t)t * O + o) * nb + b] = c;
            }
}

/* out: [T][O][K/32] int32. */
void orc_subdots_q4K(const uint8_t *w, const int8_t *qs, int T, int O, int K, int32_t *out)
{
    const int nsb = K / ORC_QK, nb = K / 32;
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < O; ++o)
            for (int b = 0; b < nb; ++b) {
                const uint8_t *blk = w + ((size_t)o * nsb + b / 8) * ORC_Q4K_BYTES;
                out[((size_t)t * O + o) * nb + b] =
                    subdot_q4K(blk, b % 8, qs + (size_t)t * K + (size_t)(b / 8) * ORC_QK);
            }
}

/* out: [T][O][K/16] int32. */
void orc_subdots_q6K(const uint8_t *w, const int8_t *qs, int T, int O, int K, int32_t *out)
{
    const int nsb = K / ORC_QK, nu = K / 16;
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < O; ++o)
            for (int u = 0; u < nu; ++u) {
                const uint8_t *blk = w + ((size_t)o * nsb + u / 16) * ORC_Q6K_BYTES;
                out[((size_t)t * O + o) * nu + u] =
                    subdot_q6K(blk, u % 16, qs + (size_t)t * K + (size_t)(u / 16) * ORC_QK);
            }
}

/* ----------------------------------------------- method-form GEMM ---- */

static float act_d(uint32_t ds) { return orc_f16_to_f32((uint16_t)(ds & 0xffffu)); }
static int act_ssum(uint32_t ds) { return (int)(int16_t)(uint16_t)(ds >> 16); }

/* One output of the q4_K GEMM in the method form ([r28] 2.3):
 *   for every super-block and sub-block j:
 *     dsv = f32(d)*sc,  dmv = -(f32(dmin)*m)
 *     t1  = (dx*dsv) * C          t2 = (dx*ssum) * dmv       (all f32)
 *     acc += t1 + t2              (f64)                                  */
static float point_q4K(const uint8_t *wrow, const int8_t *qrow, const uint32_t *dsrow, int K)
{
    const int nsb = K / ORC_QK;
    double acc = 0.0;
    for (int sb = 0; sb < nsb; ++sb) {
        const uint8_t *blk = wrow + (size_t)sb * ORC_Q4K_BYTES;
        const float d = q4K_d(blk), dmin = q4K_dmin(blk);
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            orc_q4K_scale_min(blk + 4, j, &sc, &m);
            const float dsv = d * (float)sc;
            const float dmv = -(dmin * (float)m);
            const uint32_t dsb = dsrow[sb * 8 + j];
            const float dx = act_d(dsb);
            const int ssum = act_ssum(dsb);
            const int32_t c = subdot_q4K(blk, j, qrow + (size_t)sb * ORC_QK);
            const float dxs = dx * dsv;
            const float t1 = dxs * (float)c;
            const float dma = dx * (float)ssum;
            const float t2 = dma * dmv;
            acc += (double)t1;
            acc += (double)t2;
        }
    }
    return (float)acc;
}

/* One output of the q5_K GEMM: the q4_K method form (above) with the 5-bit
 * quant (R15). */
static float point_q5K(const uint8_t *wrow, const int8_t *qrow, const uint32_t *dsrow, int K)
{
    const int nsb = K / ORC_QK;
    double acc = 0.0;
    for (int sb = 0; sb < nsb; ++sb) {
        const uint8_t *blk = wrow + (size_t)sb * ORC_Q5K_BYTES;
        const float d = q4K_d(blk), dmin = q4K_dmin(blk);
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            orc_q4K_scale_min(blk + 4, j, &sc, &m);
            const float dsv = d * (float)sc;
            const float dmv = -(dmin * (float)m);
            const uint32_t dsb = dsrow[sb * 8 + j];
            const float dx = act_d(dsb);
            const int ssum = act_ssum(dsb);
            const int32_t c = subdot_q5K(blk, j, qrow + (size_t)sb * ORC_QK);
            const float dxs = dx * dsv;
            const float t1 = dxs * (float)c;
            const float dma = dx * (float)ssum;
            const float t2 = dma * dmv;
            acc += (double)t1;
            acc += (double)t2;
        }
    }
    return (float)acc;
}

/* One output of the q8_0 GEMM (R16): per 32-block b, t = (dx_b*d_w)*C_b in
 * f32, acc += t in f64. */
static float point_q8_0(const uint8_t *wrow, const int8_t *qrow, const uint32_t *dsrow, int K)
{
    const int nb = K / 32;
    double acc = 0.0;
    for (int b = 0; b < nb; ++b) {
        const uint8_t *blk = wrow + (size_t)b * ORC_Q8_0_BYTES;
        const float dw = orc_q8_0_d(blk);
        const float dx = act_d(dsrow[b]);
        const int32_t c = subdot_q8_0(blk, qrow + (size_t)b * 32);
        const float dxs = dx * dw;
        const float t = dxs * (float)c;
        acc += (double)t;
    }
    return (float)acc;
}

/* One output of the q6_K GEMM in the method form ([r40] 5): per 32-k chunk
 * b and each of its 16-weight halves u, t = (dx*dsv_u) * C16_u in f32 with
 * dsv_u = f32(d)*sc_u; acc += t in f64. */
static float point_q6K(const uint8_t *wrow, const int8_t *qrow, const uint32_t *dsrow, int K)
{
    const int nsb = K / ORC_QK;
    double acc = 0.0;
    for (int sb = 0; sb < nsb; ++sb) {
        const uint8_t *blk = wrow + (size_t)sb * ORC_Q6K_BYTES;
        const float d = orc_q6K_d(blk);
        for (int u = 0; u < 16; ++u) {
            const float dsv = d * (float)orc_q6K_scale(blk, u);
            const float dx = act_d(dsrow[sb * 8 + u / 2]);
            const int32_t c = subdot_q6K(blk, u, qrow + (size_t)sb * ORC_QK);
            const float dxs = dx * dsv;
            const float t = dxs * (float)c;
            acc += (double)t;
        }
    }
    return (float)acc;
}

/* Y[t*ldy + o] for all t < T, o < O.  w holds O rows of K/256 blocks. */
void orc_gemm_q4K(const uint8_t *w, const int8_t *qs, const uint32_t *ds,
                  int T, int O, int K, float *y, int64_t ldy)
{
    const size_t row_bytes = (size_t)(K / ORC_QK) * ORC_Q4K_BYTES;
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < O; ++o)
            y[(size_t)t * ldy + o] = point_q4K(w + (size_t)o * row_bytes, qs + (size_t)t * K,
                                               ds + (size_t)t * (K / 32), K);
}

void orc_gemm_q6K(const uint8_t *w, const int8_t *qs, const uint32_t *ds,
                  int T, int O, int K, float *y, int64_t ldy)
{
    const size_t row_bytes = (size_t)(K / ORC_QK) * ORC_Q6K_BYTES;
    for (int t = 0; t < T; ++t)
        for (int o = 0; o < O; ++o)
            y[(size_t)t * ldy + o] = point_q6K(w + (size_t)o * row_bytes, qs + (size_t)t * K,
                                               ds + (size_t)t * (K / 32), K);
}

/* Selected outputs only: out[i] = Y[ti[i]][oi[i]]; fmt 4 = q4_K, 6 = q6_K. */
void orc_gemm_points(int fmt, const uint8_t *w, const int8_t *qs, const uint32_t *ds,
                     int K, int n, const int32_t *ti, const int32_t *oi, float *out)
{
    const size_t bb = (fmt == 6) ? ORC_Q6K_BYTES : ORC_Q4K_BYTES;
    const size_t row_bytes = (size_t)(K / ORC_QK) * bb;
    for (int i = 0; i < n; ++i) {
        const uint8_t *wrow = w + (size_t)oi[i] * row_bytes;
        const int8_t *qrow = qs + (size_t)ti[i] * K;
        const uint32_t *dsrow = ds + (size_t)ti[i] * (K / 32);
        out[i] = (fmt == 6) ? point_q6K(wrow, qrow, dsrow, K) : point_q4K(wrow, qrow, dsrow, K);
    }
}

/* Dequantised activations X^[t][k] = f32(d16) * q, as f64 (exact). */
void orc_dequant_q8_1(const int8_t *qs, const uint32_t *ds, int T, int K, double *out)
{
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            out[(size_t)t * K + k] =
                (double)act_d(ds[(size_t)t * (K / 32) + k / 32]) * qs[(size_t)t * K + k];
}

/* --------------------------------------------------------- SwiGLU ---- */

/* h[i] = silu(g[i]) * u[i], silu(g) = g / (1 + e^-g), in f32 with every
 * operation rounded on its own (reading R14; built without contraction). */
void orc_swiglu(const float *g, const float *u, int64_t n, float *h)
{
    for (int64_t i = 0; i < n; ++i) {
        const float e = expf(-g[i]);
        const float den = 1.0f + e;
        const float s = g[i] / den;
        h[i] = s * u[i];
    }
}

/* ------------------------------------------- all host cores (OpenMP) -- */

/* The same outputs as orc_gemm_q4K / orc_gemm_q6K, with the output columns o
 * (weight rows) shared among `nthreads` OpenMP threads (<= 0: the runtime's
 * default, i.e. every core the process may use).  Every output is still
 * computed by one call of the plain per-output function above, so the result
 * is bit-identical to the single-thread form; only the work is divided.
 * fmt 4 = q4_K, 6 = q6_K. */
void orc_gemm_mt(int fmt, const uint8_t *w, const int8_t *qs, const uint32_t *ds,
                 int T, int O, int K, float *y, int64_t ldy, int nthreads)
{
    const size_t bb = (fmt == 6) ? ORC_Q6K_BYTES : (fmt == 5) ? ORC_Q5K_BYTES : (fmt == 8) ? 8 * ORC_Q8_0_BYTES
                                                                                  : ORC_Q4K_BYTES;
    const size_t row_bytes = (size_t)(K / ORC_QK) * bb;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (int o = 0; o < O; ++o) {
        const uint8_t *wrow = w + (size_t)o * row_bytes;
        for (int t = 0; t < T; ++t) {
            const int8_t *qrow = qs + (size_t)t * K;
            const uint32_t *dsrow = ds + (size_t)t * (K / 32);
            y[(size_t)t * ldy + o] = (fmt == 6)   ? point_q6K(wrow, qrow, dsrow, K)
                                     : (fmt == 5) ? point_q5K(wrow, qrow, dsrow, K)
                                     : (fmt == 8) ? point_q8_0(wrow, qrow, dsrow, K)
                                                  : point_q4K(wrow, qrow, dsrow, K);
        }
    }
    (void)nthreads;
}

/* Threads orc_gemm_mt uses by default (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int orc_version(void) { return 2; }

/* Array forms of the f16 conversions, for exhaustive checks. */
void orc_f16_to_f32_array(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(h[i]);
}

void orc_f32_to_f16_array(const float *f, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(f[i]);
}
