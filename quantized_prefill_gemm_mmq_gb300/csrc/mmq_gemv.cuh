// mmq_gemv.cuh -- decode-shaped q4_K x q8_1 product (1 <= T <= 16 tokens).
// Included by mmq_gemm.cu: it shares that unit's bounded mbarrier waits and
// the device status word that mmq_check_status reads.
//
// With a handful of tokens the product reads every weight byte once and does
// little arithmetic per byte, so its time is the time to stream W from HBM.
// The arithmetic is the pages' per-sub-block form ("31 . r28 -- Direction-A
// raw-nibble NB kernel, 2 blocks/SM", 2.3): for every 32-weight sub-block b
// the exact integer dot C_b of the unsigned 4-bit quants with the int8
// activations, folded in f32 as
//     y += (dx_b * (d*sc_b)) * C_b + (dx_b * ssum_b) * (-(dmin*m_b)).
//
// GB300 design:
//   * One CTA per 16 weight rows, the whole K range, two CTAs per SM; nine
//     warps: one TMA producer (warp 8) and two groups of four consumer warps
//     (warps 0-3 and 4-7) that take alternate super-blocks.
//   * A ring of 12 (T <= 8) or 8 (T <= 16) stages, one super-block column
//     each, filled by three TMA copies per stage: the 16 rows' raw 144-byte
//     blocks (one 2-D box), the tokens' 256 activations (f16 copies of the
//     int8 values) and their 8 scale words.  Token rows past T and weight
//     rows past O arrive zero-filled from the tensor maps' bounds.  Each slot
//     has a full barrier (the copies' bytes) and an empty barrier (the four
//     consumer warps of its group); the ring length is a multiple of the
//     group count, so each slot's barriers are waited on by one agent
//     through consecutive phases.  No CTA-wide barrier inside the loop.
//     (Per-thread 16-byte cp.async copies of the same stages, and TMA with a
//     CTA barrier per stage, were measured first: both were bound by the
//     per-stage chain, not by HBM.)
//   * Consumer warp w takes sub-block pair p = w % 4 (sub-blocks 2p, 2p + 1)
//     of the 16 rows; each lane decodes the scale terms of its two rows and
//     the scale words of its two tokens itself.
//   * The dots run on the f16 warp MMA (m16n8k16, f32 accumulate) with the
//     weight rows on M and the tokens on N (one or two 8-token tiles).  The
//     weight operand is 1024 + q (low nibbles) or 1024 + 16q (high nibbles),
//     made by OR-ing the masked nibbles into the f16 exponent of 1024; the
//     activation operand is the int8 value as f16.  Every product is an
//     integer below 2^18 and every partial sum an integer below 2^24, so the
//     f32 accumulator is exact.  The accumulator starts at -1024*ssum, which
//     removes the 1024 offset: the result is C_b (low) or 16*C_b (high; its
//     scale d*sc/16 is pre-divided, an exact power-of-two scaling).
//   * Each consumer warp adds its super-blocks in order and the eight warps'
//     partial sums are added in warp order (deterministic).
//   * Every wait is bounded: after a timeout all warps leave their loops,
//     the copies still in flight are waited for (bounded) and nothing is
//     stored.

namespace mmq {
namespace {

namespace gv {

constexpr int GROUPS = 2;                 // consumer groups, taking alternate stages
constexpr int CWARPS = 4 * GROUPS;        // consumer warps: group w / 4, sub-block pair w % 4
constexpr int NTHREADS = (CWARPS + 1) * 32;   // + one TMA producer warp
constexpr int ROWS = 16;                  // weight rows per CTA (the MMA's M)
constexpr int MAXT = 16;                  // tokens: at most two 8-token MMA N tiles
constexpr int KID = 12;                   // kernel id in the status word

template <int NT>
struct Cfg {
    static constexpr int TOK = 8 * NT;                      // token slots (TMA box rows)
    static constexpr int X_OFF = ROWS * 144;                // activations within a stage ([TOK][256] f16)
    static constexpr int D_OFF = X_OFF + TOK * 512;         // scale words within a stage ([TOK][8] u32)
    static constexpr int STAGE = D_OFF + TOK * 32;          // bytes per stage, all counted by the barrier
    static constexpr int S = NT == 1 ? 12 : 8;              // ring stages; a multiple of GROUPS, so that
                                                            // every slot is consumed by one group only
    static constexpr int BAR_OFF = S * STAGE;               // S full, then S empty barriers
    static constexpr int ABORT_OFF = BAR_OFF + 16 * S;
    static constexpr int RED_OFF = ABORT_OFF + 16;          // [CWARPS][TOK][ROWS] f32 partial sums
    static constexpr int SMEM = RED_OFF + CWARPS * TOK * ROWS * 4 + 128;   // + alignment slack of the base
};
static_assert(Cfg<1>::S % GROUPS == 0 && Cfg<2>::S % GROUPS == 0, "slots map to one consumer group");
static_assert(Cfg<1>::X_OFF % 128 == 0 && Cfg<1>::D_OFF % 128 == 0 && Cfg<1>::STAGE % 128 == 0 &&
                  Cfg<2>::D_OFF % 128 == 0 && Cfg<2>::STAGE % 128 == 0,
              "TMA destinations are 128-byte aligned");
static_assert(2 * (Cfg<1>::SMEM + 1024) <= 233472 && 2 * (Cfg<2>::SMEM + 1024) <= 233472, "two CTAs per SM");

__device__ __forceinline__ float f16_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }

// Exact float of an integer 0 <= v < 2^23 (v | 2^23 read as a float is 2^23 + v).
__device__ __forceinline__ float small_u2f(uint32_t v) { return __int_as_float((int)(0x4B000000u | v)) - 8388608.0f; }
// Exact float of the signed 16-bit value in the high half of w (2^23 + 2^22 + v
// for |v| < 2^22 has the integer v in its low mantissa bits).
__device__ __forceinline__ float hi16_s2f(uint32_t w)
{
    return __int_as_float(((int)w >> 16) + 0x4B400000) - 12582912.0f;
}

// {d*sc_j (divided by 16 if j is odd), -(dmin*m_j)} of sub-block j = 2p + e of
// one row from its 16-byte block header (f16 d, f16 dmin, 12 scale bytes in
// the GGUF k-quant packing: sub-block j < 4 keeps its scale / min in the low 6
// bits of byte j / j + 4; j >= 4 takes its low 4 bits from the low / high
// nibble of byte j + 4 and its high 2 bits from the top bits of byte j - 4 /
// j).  p is warp-uniform, e may differ between lanes.
__device__ __forceinline__ float2 sub_scales(const uint4 &h, int p, int e)
{
    uint32_t sc, m;
    if (p < 2) {
        const int b = 16 * p + 8 * e;
        sc = (h.y >> b) & 63u;
        m = (h.z >> b) & 63u;
    } else {
        const int b = 16 * (p - 2) + 8 * e;
        sc = ((h.w >> b) & 15u) | (((h.y >> (b + 6)) & 3u) << 4);
        m = ((h.w >> (b + 4)) & 15u) | (((h.z >> (b + 6)) & 3u) << 4);
    }
    const float d = f16_bits(h.x & 0xFFFFu), dmin = f16_bits(h.x >> 16);
    return make_float2(d * small_u2f(sc) * (e ? 0.0625f : 1.0f), -(dmin * small_u2f(m)));
}

// Quant bytes b0..b3 of one word -> f16 pairs {1024+lo(b0), 1024+lo(b1)},
// {1024+lo(b2), 1024+lo(b3)} and the same with 1024 + 16*hi(b).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&lo)[2], uint32_t (&hi)[2])
{
    const uint32_t t = __byte_perm(w, 0u, 0x3120);   // bytes b0 b2 b1 b3
    const uint32_t t8 = t >> 8;                       // bytes b2 b1 b3 0
    lo[0] = (t & 0x000F000Fu) | 0x64006400u;
    lo[1] = (t8 & 0x000F000Fu) | 0x64006400u;
    hi[0] = (t & 0x00F000F0u) | 0x64006400u;
    hi[1] = (t8 & 0x00F000F0u) | 0x64006400u;
}

// pdl_launch_dependents / pdl_wait: mmq_pdl.cuh

// D = A (16 x 16, f16, row) * B (16 x 8, f16, col) + D, f32
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace gv

template <int NT>
__global__ void __launch_bounds__(gv::NTHREADS, 2)
    mmq_q4K_gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmD, float *__restrict__ y, int T, int O, int K)
{
    using namespace gv;
    using C = Cfg<NT>;
    extern __shared__ uint8_t sm_raw[];
    // TMA destinations: 128-byte aligned base
    uint8_t *sm = sm_raw + ((128u - (smem_u32(sm_raw) & 127u)) & 127u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int o0 = blockIdx.x * ROWS;
    const int nsb = K >> 8;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t full0 = sbase + C::BAR_OFF;      // slot s: full0 + 8 s (TMA bytes landed)
    const uint32_t empty0 = full0 + 8 * C::S;       // slot s: empty0 + 8 s (its four consumer warps done)
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + C::ABORT_OFF);
    float *red = reinterpret_cast<float *>(sm + C::RED_OFF);   // [CWARPS][TOK][ROWS]

    if (tid == 0) {
        *abort_flag = 0u;
        for (int s = 0; s < C::S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 4);
        }
        fence_mbar_init();
    }
    pdl_launch_dependents();
    __syncthreads();

    int issued = 0;   // producer: stages issued
    if (warp == CWARPS) {
        // producer: stage i -> slot i % S, the rows' blocks of super-block i and
        // the tokens' activations and scale words of k = 256 i .. 256 i + 255
        if (lane == 0) {
            tma_prefetch(&tmW);
            tma_prefetch(&tmX);
            tma_prefetch(&tmD);
            // the weights do not depend on the previous kernel: the first ring's
            // worth of weight copies go out before waiting for it, the
            // activations and scale words after
            const int first = nsb < C::S ? nsb : C::S;
            for (int i = 0; i < first; ++i) {
                const uint32_t bar = full0 + 8 * i;
                mbar_arrive_expect_tx(bar, C::STAGE);
                tma_load_2d(sbase + i * C::STAGE, &tmW, bar, i * 144, o0);
            }
            pdl_wait();
            for (int i = 0; i < first; ++i) {
                const uint32_t dst = sbase + i * C::STAGE, bar = full0 + 8 * i;
                tma_load_2d(dst + C::X_OFF, &tmX, bar, i * 256, 0);
                tma_load_2d(dst + C::D_OFF, &tmD, bar, i * 8, 0);
            }
            issued = first;
            int slot = first == C::S ? 0 : first;
            for (; issued < nsb; ++issued) {
                if (!mbar_wait(empty0 + 8 * slot, (uint32_t)((issued / C::S - 1) & 1), abort_flag, KID, SITE_P_STAGE))
                    break;
                const uint32_t dst = sbase + slot * C::STAGE, bar = full0 + 8 * slot;
                mbar_arrive_expect_tx(bar, C::STAGE);
                tma_load_2d(dst, &tmW, bar, issued * 144, o0);
                tma_load_2d(dst + C::X_OFF, &tmX, bar, issued * 256, 0);
                tma_load_2d(dst + C::D_OFF, &tmD, bar, issued * 8, 0);
                if (++slot == C::S) slot = 0;
            }
        }
    } else {
        // consumer warp: group w / 4 takes stages w / 4, w / 4 + GROUPS, ...;
        // sub-block pair p = w % 4 (sub-blocks 2p, 2p + 1) of the 16 rows
        const int p = warp & 3;
        const int g = lane >> 2, tig = lane & 3;
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[n][i] = 0.0f;
        int slot = warp >> 2;
        uint32_t phase = 0u;
        for (int i = warp >> 2; i < nsb; i += GROUPS) {
            const bool landed = mbar_wait(full0 + 8 * slot, phase, abort_flag, KID, SITE_U_STAGE);
            if (!__all_sync(0xffffffffu, landed)) break;
            const uint8_t *st = sm + slot * C::STAGE;
            // quant bytes 8 tig .. 8 tig + 7 of pair p in rows g and g + 8; element
            // e of either sub-block is byte e (low / high nibble), so word h holds
            // elements 8 tig + 4h .. + 3: the lane's k of MMA half h
            const uint2 wa = *reinterpret_cast<const uint2 *>(st + g * 144 + 16 + 32 * p + 8 * tig);
            const uint2 wb = *reinterpret_cast<const uint2 *>(st + (g + 8) * 144 + 16 + 32 * p + 8 * tig);
            // scale terms of sub-blocks 2p, 2p + 1 in rows g and g + 8
            const uint4 hA = *reinterpret_cast<const uint4 *>(st + g * 144);
            const uint4 hB = *reinterpret_cast<const uint4 *>(st + (g + 8) * 144);
            float sA[4], sB[4];
            {
                const float2 a0 = sub_scales(hA, p, 0), a1 = sub_scales(hA, p, 1);
                const float2 b0 = sub_scales(hB, p, 0), b1 = sub_scales(hB, p, 1);
                sA[0] = a0.x;
                sA[1] = a0.y;
                sA[2] = a1.x;
                sA[3] = a1.y;
                sB[0] = b0.x;
                sB[1] = b0.y;
                sB[2] = b1.x;
                sB[3] = b1.y;
            }
            uint32_t la[2][2], ha[2][2], lb[2][2], hb[2][2];
            unpack_word(wa.x, la[0], ha[0]);
            unpack_word(wa.y, la[1], ha[1]);
            unpack_word(wb.x, lb[0], hb[0]);
            unpack_word(wb.y, lb[1], hb[1]);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                // token 8n + g: elements 8 tig .. 8 tig + 7 of sub-blocks 2p and 2p + 1
                const uint8_t *xr = st + C::X_OFF + (8 * n + g) * 512 + 128 * p + 16 * tig;
                const uint4 xl = *reinterpret_cast<const uint4 *>(xr);
                const uint4 xu = *reinterpret_cast<const uint4 *>(xr + 64);
                // scale words of tokens t0, t0 + 1 for sub-blocks 2p, 2p + 1
                const int t0 = 8 * n + 2 * tig;
                const uint2 w0 = *reinterpret_cast<const uint2 *>(st + C::D_OFF + t0 * 32 + 8 * p);
                const uint2 w1 = *reinterpret_cast<const uint2 *>(st + C::D_OFF + (t0 + 1) * 32 + 8 * p);
                const float dxl0 = f16_bits(w0.x & 0xFFFFu), ssl0 = hi16_s2f(w0.x);
                const float dxu0 = f16_bits(w0.y & 0xFFFFu), ssu0 = hi16_s2f(w0.y);
                const float dxl1 = f16_bits(w1.x & 0xFFFFu), ssl1 = hi16_s2f(w1.x);
                const float dxu1 = f16_bits(w1.y & 0xFFFFu), ssu1 = hi16_s2f(w1.y);
                // c: rows (g, g+8) x tokens (t0, t0+1); starts at -1024*ssum
                float cl[4] = {-1024.0f * ssl0, -1024.0f * ssl1, -1024.0f * ssl0, -1024.0f * ssl1};
                mma_f16(cl, la[0][0], lb[0][0], la[0][1], lb[0][1], xl.x, xl.y);
                mma_f16(cl, la[1][0], lb[1][0], la[1][1], lb[1][1], xl.z, xl.w);
                float cu[4] = {-1024.0f * ssu0, -1024.0f * ssu1, -1024.0f * ssu0, -1024.0f * ssu1};
                mma_f16(cu, ha[0][0], hb[0][0], ha[0][1], hb[0][1], xu.x, xu.y);
                mma_f16(cu, ha[1][0], hb[1][0], ha[1][1], hb[1][1], xu.z, xu.w);
                const float ml0 = dxl0 * ssl0, ml1 = dxl1 * ssl1, mu0 = dxu0 * ssu0, mu1 = dxu1 * ssu1;
                acc[n][0] = fmaf(dxl0 * sA[0], cl[0], acc[n][0]);
                acc[n][1] = fmaf(dxl1 * sA[0], cl[1], acc[n][1]);
                acc[n][2] = fmaf(dxl0 * sB[0], cl[2], acc[n][2]);
                acc[n][3] = fmaf(dxl1 * sB[0], cl[3], acc[n][3]);
                acc[n][0] = fmaf(ml0, sA[1], acc[n][0]);
                acc[n][1] = fmaf(ml1, sA[1], acc[n][1]);
                acc[n][2] = fmaf(ml0, sB[1], acc[n][2]);
                acc[n][3] = fmaf(ml1, sB[1], acc[n][3]);
                acc[n][0] = fmaf(dxu0 * sA[2], cu[0], acc[n][0]);
                acc[n][1] = fmaf(dxu1 * sA[2], cu[1], acc[n][1]);
                acc[n][2] = fmaf(dxu0 * sB[2], cu[2], acc[n][2]);
                acc[n][3] = fmaf(dxu1 * sB[2], cu[3], acc[n][3]);
                acc[n][0] = fmaf(mu0, sA[3], acc[n][0]);
                acc[n][1] = fmaf(mu1, sA[3], acc[n][1]);
                acc[n][2] = fmaf(mu0, sB[3], acc[n][2]);
                acc[n][3] = fmaf(mu1, sB[3], acc[n][3]);
            }
            // release the slot: this lane's reads come before its refill by TMA
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            slot += GROUPS;
            if (slot >= C::S) {
                slot -= C::S;
                phase ^= 1u;
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int t0 = 8 * n + 2 * tig;
            red[(warp * C::TOK + t0) * ROWS + g] = acc[n][0];
            red[(warp * C::TOK + t0 + 1) * ROWS + g] = acc[n][1];
            red[(warp * C::TOK + t0) * ROWS + g + 8] = acc[n][2];
            red[(warp * C::TOK + t0 + 1) * ROWS + g + 8] = acc[n][3];
        }
    }
    __syncthreads();
    if (*abort_flag) {
        // a wait ran out of time: wait (bounded) for the copies still in flight
        // (the last S stages issued, one per slot), store nothing
        if (warp == CWARPS && lane == 0)
            for (int i = issued > C::S ? issued - C::S : 0; i < issued; ++i)
                if (!wait_drain(full0 + 8 * (i % C::S), (uint32_t)((i / C::S) & 1))) {
                    record_error(kStatusTimeout, KID, SITE_DRAIN);
                    break;
                }
        __syncthreads();
        return;
    }
    // partial sums of the eight consumer warps, added in warp order (y is
    // written only once the previous kernel in the stream has completed)
    pdl_wait();
    for (int i = tid; i < C::TOK * ROWS; i += NTHREADS) {
        const int t = i / ROWS, r = i % ROWS;
        if (t < T && o0 + r < O) {
            float s = red[t * ROWS + r];
#pragma unroll
            for (int v = 1; v < CWARPS; ++v) s += red[(v * C::TOK + t) * ROWS + r];
            y[(size_t)t * O + o0 + r] = s;
        }
    }
}

template <int NT>
int launch_gemv_nt(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                   mmq_stream_t stream)
{
    using C = gv::Cfg<NT>;
    const int nsb = K / 256;
    CUtensorMap tmW, tmX, tmD;
    // W as [O][nsb*144] bytes, box 144 B x 16 rows; rows past O read as zero
    int rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)nsb * 144, (uint64_t)O,
                          (uint64_t)nsb * 144, 144, gv::ROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    // xh as [T][K] 16-bit, box 256 x TOK; token rows past T read as zero
    rc = make_tmap_2d(&tmX, xh, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, 256,
                      C::TOK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    // ds as [T][K/32] words, box 8 x TOK
    rc = make_tmap_2d(&tmD, ds, CU_TENSOR_MAP_DATA_TYPE_UINT32, (uint64_t)(K / 32), (uint64_t)T, (uint64_t)(K / 8), 8,
                      C::TOK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    static bool attr_done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q4K_gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((O + gv::ROWS - 1) / gv::ROWS));
    cfg.blockDim = dim3(gv::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may overlap the previous kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mmq_q4K_gemv_kernel<NT>, tmW, tmX, tmD, y, T, O, K) != cudaSuccess)
        return launch_status();
    return launch_status();
}

int launch_gemv(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                mmq_stream_t stream)
{
    if (T < 0 || T > gv::MAXT || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !xh || !ds || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xh) || !aligned16(ds) || !aligned16(y)) return MMQ_ERR_ALIGN;
    const int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    return T <= 8 ? launch_gemv_nt<1>(w, xh, ds, y, T, O, K, stream)
                  : launch_gemv_nt<2>(w, xh, ds, y, T, O, K, stream);
}

}  // namespace
}  // namespace mmq

extern "C" int mmq_gemv_q4K(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_gemv(w, xh, ds, y, T, O, K, stream);
}
