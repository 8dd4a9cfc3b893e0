// mmq_gemv_q6.cuh -- decode-shaped q6_K x q8_1 product (1 <= T <= 16 tokens).
// Included by mmq_gemm.cu after mmq_gemv.cuh (it shares that unit's bounded
// waits, status word and the decode-shaped kernels' helpers).
//
// The pages' q6_K form ("43 . r40 -- __launch_bounds__(256,3) third resident
// block", 5): w = d * sc_u * (q - 32) on 16-weight sub-blocks u with signed
// 8-bit scales, and the per-16 fold  y += (dx_b * (d*sc_u)) * C16_u  with
// C16_u the exact integer dot of (q - 32) with the int8 activations of the
// 32-block b = u / 2.
//
// Same skeleton as the q4_K decode kernel (mmq_gemv.cuh): one CTA per 16
// weight rows over the whole K, a producer warp, two groups of four consumer
// warps on alternate super-blocks, full / empty barriers per slot.
//   * A 210-byte q6_K block starts on a 2-byte boundary, so a TMA box cannot
//     address it.  Each producer lane (one per row) copies the 16-byte-aligned
//     224-byte window holding its row's block with one bulk copy; past the
//     buffer's last full 16-byte granule the remaining bytes are copied one
//     by one before the lane's arrival on the full barrier.  Lane 0 also
//     requests the tokens' activations and scale words by TMA, as in q4_K.
//   * Consumer warp w takes quarter p = w % 4 of the super-block (weights
//     64p .. 64p + 63: q8_1 blocks 2p, 2p + 1, sub-blocks 4p .. 4p + 3).  Its
//     lanes read the ql / qh / scale bytes they need as aligned 32-bit words
//     of the window and shift them into place (the block's offset in the
//     window is even, 0..14).
//   * Each 16-weight sub-block is one m16n8k16 f16 MMA: weight operand q - 32
//     (the 6-bit value OR-ed into the f16 exponent of 1024, minus 1056: exact),
//     activation operand the int8 value as f16; |(q - 32) * a| <= 4064 and 16
//     of them stay far below 2^24, so the accumulator holds C16_u exactly.

namespace mmq {
namespace {

namespace gv6 {

constexpr int ROWS = 16;
constexpr int KID = 13;               // kernel id in the status word

template <int NT>
struct Cfg {
    static constexpr int TOK = 8 * NT;
    // super-blocks per stage: two at T <= 8 (half the producer's copies per
    // byte), one at T <= 16 (where the larger activation boxes leave room
    // for fewer stages)
    static constexpr int SB = NT == 1 ? 2 : 1;
    static constexpr int WROW = SB == 2 ? 448 : 224;         // 16-byte-aligned window per row
    static constexpr int GROUPS = 2;
    static constexpr int CWARPS = 4 * GROUPS;
    static constexpr int NTHREADS = (CWARPS + 1) * 32;      // + the producer warp
    static constexpr int X_OFF = ROWS * WROW;               // activations [SB][TOK][256] f16
    static constexpr int D_OFF = X_OFF + SB * TOK * 512;    // scale words [TOK][8 SB]
    static constexpr int STAGE = D_OFF + TOK * 32 * SB;
    static constexpr int S = NT == 1 ? 6 : 8;               // ring stages, a multiple of GROUPS
    static constexpr int BAR_OFF = S * STAGE;               // S full, then S empty barriers
    static constexpr int ABORT_OFF = BAR_OFF + 16 * S;
    static constexpr int RED_OFF = ABORT_OFF + 16;          // [CWARPS][TOK][ROWS] f32
    static constexpr int SMEM = RED_OFF + CWARPS * TOK * ROWS * 4 + 128;
};
static_assert(Cfg<1>::X_OFF % 128 == 0 && Cfg<1>::D_OFF % 128 == 0 && Cfg<1>::STAGE % 128 == 0 &&
                  Cfg<2>::D_OFF % 128 == 0 && Cfg<2>::STAGE % 128 == 0,
              "TMA destinations are 128-byte aligned");
static_assert(Cfg<1>::S % Cfg<1>::GROUPS == 0 && Cfg<2>::S % Cfg<2>::GROUPS == 0, "slots map to one group");
static_assert(2 * (Cfg<1>::SMEM + 1024) <= 233472 && 2 * (Cfg<2>::SMEM + 1024) <= 233472, "two CTAs per SM");

// the 32-bit little-endian word at byte offset `o` (any even offset) of a
// 4-byte-aligned shared-memory row, from the two aligned words around it
__device__ __forceinline__ uint32_t ld_u32_at(const uint8_t *row, int o)
{
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row) + (o >> 2);
    return __funnelshift_r(w[0], w[1], (o & 3) * 8);
}

// four 6-bit values (one per byte) -> two f16 pairs {q0-32, q1-32}, {q2-32, q3-32}
__device__ __forceinline__ void q6_pairs(uint32_t q, uint32_t &p01, uint32_t &p23)
{
    const __half2 off = __float2half2_rn(-1056.0f);
    uint32_t h01 = __byte_perm(q, 0x64646464u, 0x4140), h23 = __byte_perm(q, 0x64646464u, 0x4342);
    __half2 a = __hadd2(*reinterpret_cast<const __half2 *>(&h01), off);
    __half2 b = __hadd2(*reinterpret_cast<const __half2 *>(&h23), off);
    p01 = *reinterpret_cast<const uint32_t *>(&a);
    p23 = *reinterpret_cast<const uint32_t *>(&b);
}

}  // namespace gv6

template <int NT>
__global__ void __launch_bounds__(gv6::Cfg<NT>::NTHREADS, 2)
    mmq_q6K_gemv_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
                        const uint8_t *__restrict__ w, float *__restrict__ y, int T, int O, int K)
{
    using namespace gv6;
    using C = Cfg<NT>;
    constexpr int GROUPS = C::GROUPS, CWARPS = C::CWARPS, NTHREADS = C::NTHREADS;
    constexpr int SB = C::SB, WROW = C::WROW;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = sm_raw + ((128u - (smem_u32(sm_raw) & 127u)) & 127u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int o0 = blockIdx.x * ROWS;
    const int nsb = K >> 8;
    const int nst = (nsb + SB - 1) / SB;            // stages: SB super-blocks each (fewer at the end)
    const uint32_t sbase = smem_u32(sm);
    const uint32_t full0 = sbase + C::BAR_OFF;      // slot s: + 8 s (32 producer-lane arrivals + bytes)
    const uint32_t empty0 = full0 + 8 * C::S;       // slot s: + 8 s (its four consumer warps)
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + C::ABORT_OFF);
    float *red = reinterpret_cast<float *>(sm + C::RED_OFF);   // [CWARPS][TOK][ROWS]

    if (tid == 0) {
        *abort_flag = 0u;
        for (int s = 0; s < C::S; ++s) {
            mbar_init(full0 + 8 * s, 32);
            mbar_init(empty0 + 8 * s, 4);
        }
        fence_mbar_init();
    }
    pdl_launch_dependents();
    __syncthreads();

    int issued = 0;   // producer: stages issued
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.0f;

    if (warp == CWARPS) {
        // producer: stage j -> slot j % S holds super-blocks SB j .. SB j + SB - 1
        // (fewer at the end of the row): lane r < 16 copies row o0 + r's window
        // around them, lane 0 also requests the tokens' activations (one box
        // per super-block) and scale words
        const int nrows = min(ROWS, O - o0);
        const uint64_t nbytes = (uint64_t)O * nsb * 210;
        if (lane == 0) {
            tma_prefetch(&tmX);
            tma_prefetch(&tmD);
        }
        // row lane's window of stage j into the stage at dst, the lane's arrival
        // on the stage's full barrier with its bytes (lane 0: also the boxes'
        // bytes; the boxes are requested separately)
        auto stage_w = [&](int j, uint32_t dst, uint32_t bar, uint8_t *dst_gen) {
            const int nb = min(SB, nsb - SB * j);
            uint32_t mine = 0, sz = 0;
            uint64_t a = 0;
            if (lane < nrows) {
                const uint64_t start = ((uint64_t)(o0 + lane) * nsb + SB * j) * 210;
                a = start & ~15ull;
                sz = nb == SB ? WROW : 224;   // covers the blocks plus their <= 14-byte lead-in
                if (a + sz > nbytes) {
                    // the buffer ends inside this window (it holds the buffer's last
                    // block): bulk-copy its full 16-byte granules, the blocks'
                    // remaining bytes one by one
                    sz = (uint32_t)((nbytes - a) & ~15ull);
                    uint8_t *drow = dst_gen + lane * WROW;
                    for (uint64_t b = a + sz; b < start + 210 * nb; ++b) drow[b - a] = w[b];
                }
                mine = sz;
            }
            if (lane == 0) mine += nb * C::TOK * 512 + C::TOK * 32 * SB;
            mbar_arrive_expect_tx(bar, mine);
            if (sz) bulk_load(dst + lane * WROW, w + a, sz, bar);
        };
        auto stage_x = [&](int j, uint32_t dst, uint32_t bar) {
            const int nb = min(SB, nsb - SB * j);
            for (int q = 0; q < nb; ++q)
                tma_load_2d(dst + C::X_OFF + q * C::TOK * 512, &tmX, bar, (SB * j + q) * 256, 0);
            tma_load_2d(dst + C::D_OFF, &tmD, bar, SB * j * 8, 0);   // words past K/32 read as zero
        };
        // the weights do not depend on the previous kernel: the first ring's
        // worth of windows go out before waiting for it, the activations and
        // scale words after
        const int first = nst < C::S ? nst : C::S;
        for (int j = 0; j < first; ++j) stage_w(j, sbase + j * C::STAGE, full0 + 8 * j, sm + j * C::STAGE);
        pdl_wait();
        if (lane == 0)
            for (int j = 0; j < first; ++j) stage_x(j, sbase + j * C::STAGE, full0 + 8 * j);
        issued = first;
        int slot = first == C::S ? 0 : first;
        for (; issued < nst; ++issued) {
            if (!mbar_wait_warp(empty0 + 8 * slot, (uint32_t)((issued / C::S - 1) & 1), abort_flag, KID, SITE_P_RAW))
                break;
            const uint32_t dst = sbase + slot * C::STAGE, bar = full0 + 8 * slot;
            stage_w(issued, dst, bar, sm + slot * C::STAGE);
            if (lane == 0) stage_x(issued, dst, bar);
            if (++slot == C::S) slot = 0;
        }
    } else {
        // consumer warp: group w / 4 takes stages w / 4, w / 4 + GROUPS, ...;
        // quarter p = w % 4 of each super-block: 32-blocks 2p + e (e = 0, 1),
        // sub-blocks 4p + 2e + s
        const int p = warp & 3, h = p >> 1, pq = p & 1;
        const int g = lane >> 2, tig = lane & 3;
        int slot = warp >> 2;
        uint32_t phase = 0u;
        for (int j = warp >> 2; j < nst; j += GROUPS) {
            const bool landed = mbar_wait(full0 + 8 * slot, phase, abort_flag, KID, SITE_U_STAGE);
            if (!__all_sync(0xffffffffu, landed)) break;
            const uint8_t *st = sm + slot * C::STAGE;
            const int nb = min(SB, nsb - SB * j);
            for (int q = 0; q < nb; ++q) {
                // rows g (jr = 0) and g + 8 (jr = 1): the exact f16 operands (q - 32)
                // of elements 16 s + 4 tig .. + 3 of 32-block 2p + e of super-block
                // SB j + q, and the scale terms d*sc of its sub-blocks 4p + k, k = 2e + s
                uint32_t a01[2][2][2], a23[2][2][2];   // [jr][e][s]
                float dsv[2][4];
#pragma unroll
                for (int jr = 0; jr < 2; ++jr) {
                    const int r = g + 8 * jr;
                    const uint8_t *wr = st + r * WROW;
                    // the first block's offset in the window: start mod 16 (start =
                    // 210 * block index); the stage's next block follows it
                    const int off = (int)((((uint32_t)(o0 + r) * (uint32_t)nsb + (uint32_t)(SB * j)) & 7u) * 210u & 15u) +
                                    210 * q;
                    const uint32_t qh0 = ld_u32_at(wr, off + 128 + 32 * h + 4 * tig);
                    const uint32_t qh1 = ld_u32_at(wr, off + 128 + 32 * h + 16 + 4 * tig);
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            const uint32_t ql = ld_u32_at(wr, off + 64 * h + 32 * e + 16 * s + 4 * tig);
                            const uint32_t n4 = (ql >> (4 * pq)) & 0x0F0F0F0Fu;
                            const uint32_t h2 = (((s ? qh1 : qh0) >> (2 * (2 * pq + e))) & 0x03030303u) << 4;
                            gv6::q6_pairs(n4 | h2, a01[jr][e][s], a23[jr][e][s]);
                        }
                    const uint32_t scw = ld_u32_at(wr, off + 192 + 4 * p);
                    const float d = gv::f16_bits(*reinterpret_cast<const uint16_t *>(wr + off + 208));
#pragma unroll
                    for (int k = 0; k < 4; ++k) dsv[jr][k] = d * (float)(int)(int8_t)(uint8_t)(scw >> (8 * k));
                }
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int t0 = 8 * n + 2 * tig;
                    const uint8_t *xr = st + C::X_OFF + q * C::TOK * 512 + (8 * n + g) * 512;
                    const uint8_t *dw = st + C::D_OFF + 32 * SB * t0 + 32 * q;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int b = 2 * p + e;
                        const float dx0 = gv::f16_bits(*reinterpret_cast<const uint32_t *>(dw + b * 4) & 0xFFFFu);
                        const float dx1 = gv::f16_bits(*reinterpret_cast<const uint32_t *>(dw + 32 * SB + b * 4) & 0xFFFFu);
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            // token 8n + g: elements 16 s + 4 tig .. + 3 of 32-block b
                            const uint2 xv = *reinterpret_cast<const uint2 *>(xr + 2 * (32 * b + 16 * s + 4 * tig));
                            float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            gv::mma_f16(c, a01[0][e][s], a01[1][e][s], a23[0][e][s], a23[1][e][s], xv.x, xv.y);
                            const int k = 2 * e + s;
                            acc[n][0] = fmaf(dx0 * dsv[0][k], c[0], acc[n][0]);
                            acc[n][1] = fmaf(dx1 * dsv[0][k], c[1], acc[n][1]);
                            acc[n][2] = fmaf(dx0 * dsv[1][k], c[2], acc[n][2]);
                            acc[n][3] = fmaf(dx1 * dsv[1][k], c[3], acc[n][3]);
                        }
                    }
                }
            }
            // release the slot: this lane's reads come before its refill
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
    pdl_wait();   // y is written only once the previous kernel in the stream has completed
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
int launch_gemv_q6_nt(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                      mmq_stream_t stream)
{
    using C = gv6::Cfg<NT>;
    CUtensorMap tmX, tmD;
    // xh as [T][K] 16-bit, box 256 x TOK; ds as [T][K/32] words, box 8 SB x TOK;
    // token rows past T and words past K/32 read as zero
    int rc = make_tmap_2d(&tmX, xh, CU_TENSOR_MAP_DATA_TYPE_UINT16, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, 256,
                          C::TOK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    rc = make_tmap_2d(&tmD, ds, CU_TENSOR_MAP_DATA_TYPE_UINT32, (uint64_t)(K / 32), (uint64_t)T, (uint64_t)(K / 8),
                      8 * C::SB, C::TOK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    static bool attr_done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q6K_gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((O + gv6::ROWS - 1) / gv6::ROWS));
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may overlap the previous kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mmq_q6K_gemv_kernel<NT>, tmX, tmD, static_cast<const uint8_t *>(w), y, T, O, K) !=
        cudaSuccess)
        return launch_status();
    return launch_status();
}

int launch_gemv_q6(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                   mmq_stream_t stream)
{
    if (T < 0 || T > gv::MAXT || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !xh || !ds || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xh) || !aligned16(ds) || !aligned16(y)) return MMQ_ERR_ALIGN;
    const int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    return T <= 8 ? launch_gemv_q6_nt<1>(w, xh, ds, y, T, O, K, stream)
                  : launch_gemv_q6_nt<2>(w, xh, ds, y, T, O, K, stream);
}

}  // namespace
}  // namespace mmq

extern "C" int mmq_gemv_q6K(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_gemv_q6(w, xh, ds, y, T, O, K, stream);
}
