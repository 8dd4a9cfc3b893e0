// mmq_gemm.cu -- q4_K / q6_K x q8_1 prefill GEMM on sm_103a tensor cores.
//
// Y[t][o] = sum_k W[o][k] X[t][k] in the block-wise integer form of the
// "minfer" pages ("31 . r28 -- Direction-A raw-nibble NB kernel", 2.3):
// per 32-weight sub-block b the exact integer dot C_b of the unsigned
// 4-bit quants with the int8 activations, then the f32 two-term fold
//     y += dx_b*(d*sc_b)*C_b + (dx_b*ssum_b)*(-(dmin*m_b)).
// q6_K ("43 . r40 -- __launch_bounds__(256,3)", 5) uses 16-weight halves:
//     y += dx_(u/2)*(d*sc_u)*C16_u,  C16_u = sum (q-32)*a.
//
// GB300 design (prior art on the pages is warp-level IMMA on GB10; sm_103a
// has no int8 tcgen05 kind, so the dot runs as kind::f16 on exact integers):
//   * The q8_1 values arrive as f16 (exact for |q| <= 127), K-major [T][K];
//     TMA copies 128-token x 64-k tiles straight into the 128-byte-swizzled
//     operand layout (tensor-core operand A, M = tokens).
//   * Raw weight super-blocks are staged unmodified: q4_K with one 2-D TMA
//     box of 128 rows x 144 B; q6_K with one bulk copy per row of the
//     224-byte, 16-byte-aligned window around its 210-byte block (blocks
//     start on 2-byte boundaries; the last few bytes of the buffer, past its
//     final full 16-byte granule, are copied with byte loads instead).
//   * Four unpack warps turn the raw bytes into the f16 operand B tile
//     (N = 128 weight rows x 64 k, same swizzled layout) and decode the
//     per-row, per-sub-block scale terms into shared memory.
//   * One thread issues tcgen05.mma: every sub-block (32 k, or 16 k for
//     q6_K) goes into a fresh TMEM accumulator of 128 x 128 f32; the products
//     are integers and every partial sum stays below 2^24, so the f32
//     accumulator holds the exact integer dot.  Four accumulators rotate.
//   * Eight epilogue warps tcgen05.ld each accumulator and apply the fold in
//     f32 registers; Y is written once at the end (f32, no f16 on the way).
//   * Every pipeline wait is bounded: after a time limit the kernel records
//     MMQ_ERR_TIMEOUT in the device status word, all roles stop, the MMA
//     thread drains its tensor-core work and TMEM is freed.
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>
#include <cstring>
#include <mutex>

#include "mmq_dev.cuh"
#include "mmq_host.h"

namespace mmq {
namespace {

enum { kQ4K = 0, kQ6K = 1, kQ5K = 2, kQ8_0 = 3 };
enum { kFold = 0, kSubdots = 1 };

constexpr int BM = 128;           // tokens per tile: MMA M, TMEM lanes
constexpr int BN = 128;           // weight rows per tile: MMA N, columns per accumulator
constexpr int BK = 64;            // k per pipeline stage: one 128-byte swizzled f16 row
constexpr int STAGES = 4;         // operand ring depth
constexpr int RAW_STAGES = 2;     // raw super-block ring depth
constexpr int SDS_STAGES = 3;     // decoded scale ring depth
constexpr int ACC_SLOTS = 4;      // TMEM accumulators (BN columns each)
constexpr int TMEM_COLS = ACC_SLOTS * BN;
constexpr int NUM_THREADS = 448;  // 14 warps
constexpr int UNPACK_WARP0 = 2;   // warps 2..5
constexpr int EPI_WARP0 = 6;      // warps 6..13
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t A_BYTES = BM * 128;
constexpr uint32_t B_BYTES = BN * 128;

template <int FMT>
struct Fmt;
template <>
struct Fmt<kQ4K> {
    static constexpr int kBlockBytes = 144;
    static constexpr int kRawRow = 144;     // staged bytes per tile row
    static constexpr int kKSub = 32;        // k per accumulator
    static constexpr int kSdsEntry = 8;     // float2 (d*sc, -dmin*m)
};
template <>
struct Fmt<kQ6K> {
    static constexpr int kBlockBytes = 210;
    static constexpr int kRawRow = 224;     // 210 bytes + up to 14 bytes of lead-in
    static constexpr int kKSub = 16;
    static constexpr int kSdsEntry = 4;     // float d*sc
};
template <>
struct Fmt<kQ5K> {                          // d, dmin, scales as q4_K; qh[32] at +16, qs[128] at +48
    static constexpr int kBlockBytes = 176;
    static constexpr int kRawRow = 176;
    static constexpr int kKSub = 32;
    static constexpr int kSdsEntry = 8;     // float2 (d*sc, -dmin*m)
};
template <>
struct Fmt<kQ8_0> {                         // per 256 weights: eight 34-byte blocks (f16 d, 32 int8)
    static constexpr int kBlockBytes = 272;
    static constexpr int kRawRow = 272;
    static constexpr int kKSub = 32;
    static constexpr int kSdsEntry = 4;     // float d of the block
};

template <int FMT>
struct Layout {
    static constexpr int kSubPerSb = 256 / Fmt<FMT>::kKSub;          // accumulators per super-block
    static constexpr int kSubPerStage = BK / Fmt<FMT>::kKSub;         // accumulators per stage
    static constexpr uint32_t kRawBytes = BN * Fmt<FMT>::kRawRow;
    static constexpr uint32_t kSdsBytes = kSubPerSb * BN * Fmt<FMT>::kSdsEntry;
    static constexpr uint32_t oA = 0;
    static constexpr uint32_t oB = oA + STAGES * A_BYTES;
    static constexpr uint32_t oRaw = oB + STAGES * B_BYTES;
    static constexpr uint32_t oSds = oRaw + RAW_STAGES * kRawBytes;
    static constexpr uint32_t oBar = oSds + SDS_STAGES * kSdsBytes;
    // barriers: a_full, b_full, st_empty [STAGES]; r_full, r_empty [RAW];
    // s_full, s_empty [SDS]; acc_full, acc_empty [ACC]; mma_done
    static constexpr int kNumBars = 3 * STAGES + 2 * RAW_STAGES + 2 * SDS_STAGES + 2 * ACC_SLOTS + 1;
    static constexpr uint32_t oMisc = oBar + kNumBars * 8;
    static constexpr uint32_t kBytes = oMisc + 16;
    static constexpr uint32_t kDynSmem = kBytes + 1024;   // slack for 1024-byte alignment
    static_assert(kDynSmem <= 232448, "shared memory budget");
    static_assert(oRaw % 1024 == 0 && kRawBytes % 1024 == 0, "raw ring alignment");
};

struct Params {
    const uint8_t *w;     // raw weights (q6_K bulk copies)
    const uint32_t *ds;   // [T][K/32]
    float *y;             // [T][O]
    int32_t *sub;         // [T][O][K/kKSub] (subdots mode)
    int T, O, K;
    // split-K (production q4_K kernel): blockIdx.z handles super-blocks
    // [z*sb_per_split, min(nsb, (z+1)*sb_per_split)); with part != nullptr the
    // partial sums go to part[z][T][O] and the last CTA of each output tile
    // (counted in cnt[tile]) adds them in z order and writes y.
    int sb_per_split;
    float *part;
    int *cnt;
    // SwiGLU output (production q4_K kernel): with h_xa != nullptr the O = 2F weight
    // rows are gate and up rows interleaved in groups of 64 (tile j: gate rows
    // 64j..64j+63, then up rows 64j..64j+63), and instead of y the kernel writes
    // h = silu(gate)*up quantised to q8_1: h_xa [2][T][F] (hi, lo planes), h_ds
    // [T][F/32], h_qs [T][F] (optional)
    uint16_t *h_xa;
    uint32_t *h_ds;
    int8_t *h_qs;
};

// wait sites recorded with a timeout
enum { SITE_P_RAW = 1, SITE_P_STAGE, SITE_M_A, SITE_M_B, SITE_M_ACC, SITE_U_RAW, SITE_U_SDS,
       SITE_U_STAGE, SITE_E_SDS, SITE_E_ACC, SITE_DRAIN };

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity)
{
    // used on the way out: waits for work already in flight, which completes
    // on its own; bounded all the same, with the time waited counted as in
    // mbar_wait (positive global-timer steps of at most kPollCreditNs each),
    // so that a timer adjustment cannot end the drain early
    uint64_t prev = globaltimer(), waited = 0;
    while (!mbar_try_wait(bar, parity)) {
        const uint64_t now = globaltimer();
        const int64_t step = (int64_t)(now - prev);
        prev = now;
        if (step > 0) waited += (uint64_t)step < kPollCreditNs ? (uint64_t)step : kPollCreditNs;
        if (waited > g_wait_limit_ns) return false;
    }
    return true;
}

// two f16 values from the low nibbles of bytes (sel) of w, exact
__device__ __forceinline__ uint32_t nib_lo2(uint32_t w, uint32_t sel)
{
    const uint32_t p = __byte_perm(w, 0u, sel);                 // bytes -> [b, 0, b', 0]
    const uint32_t h = (p & 0x000F000Fu) | 0x64006400u;           // 1024 + q in each half
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), __half2half2(__ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// two f16 values from the high nibbles of bytes (sel) of w, exact
__device__ __forceinline__ uint32_t nib_hi2(uint32_t w, uint32_t sel)
{
    const uint32_t p = __byte_perm(w, 0u, sel);
    const uint32_t h = (p & 0x00F000F0u) | 0x64006400u;           // 1024 + 16 q
    const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&h),
                              __half2half2(__ushort_as_half(0x2C00)),      // 1/16
                              __half2half2(__ushort_as_half(0xD400)));     // -64
    return *reinterpret_cast<const uint32_t *>(&r);
}

// two f16 values from the low 5 bits of bytes (sel) of w (each byte 0..31), exact
__device__ __forceinline__ uint32_t u5_2(uint32_t w, uint32_t sel)
{
    const uint32_t p = __byte_perm(w, 0u, sel);
    const uint32_t h = (p & 0x001F001Fu) | 0x64006400u;           // 1024 + v in each half
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), __half2half2(__ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t pack_h2(int a, int b)
{
    const __half2 h = __halves2half2(__int2half_rn(a), __int2half_rn(b));
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    mmq_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                    const Params p)
{
    using F = Fmt<FMT>;
    using L = Layout<FMT>;
    constexpr int kKid = FMT < 2 ? 1 + FMT * 2 + MODE : 20 + (FMT - 2) * 2 + MODE;
    constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-byte aligned
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int T = p.T, O = p.O, K = p.K;
    const int nks = K / BK, nsb = K / 256;

    const uint32_t bar0 = sbase + L::oBar;
    auto a_full = [&](int s) { return bar0 + 8u * s; };
    auto b_full = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto st_empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto r_full = [&](int s) { return bar0 + 8u * (3 * STAGES + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (3 * STAGES + RAW_STAGES + s); };
    auto s_full = [&](int s) { return bar0 + 8u * (3 * STAGES + 2 * RAW_STAGES + s); };
    auto s_empty = [&](int s) { return bar0 + 8u * (3 * STAGES + 2 * RAW_STAGES + SDS_STAGES + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (3 * STAGES + 2 * RAW_STAGES + 2 * SDS_STAGES + s); };
    auto acc_empty = [&](int s) {
        return bar0 + 8u * (3 * STAGES + 2 * RAW_STAGES + 2 * SDS_STAGES + ACC_SLOTS + s);
    };
    const uint32_t mma_done = bar0 + 8u * (L::kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::oMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(a_full(s), 1);
            mbar_init(b_full(s), 128);
            mbar_init(st_empty(s), 1);
        }
        for (int s = 0; s < RAW_STAGES; ++s) {
            mbar_init(r_full(s), FMT == kQ6K ? 32 : 1);   // q6_K: every producer lane arrives
            mbar_init(r_empty(s), 128);
        }
        for (int s = 0; s < SDS_STAGES; ++s) {
            mbar_init(s_full(s), 128);
            mbar_init(s_empty(s), NUM_EPI_WARPS);
        }
        for (int s = 0; s < ACC_SLOTS; ++s) {
            mbar_init(acc_full(s), 1);
            mbar_init(acc_empty(s), NUM_EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer --
        if (lane == 0) {
            tma_prefetch(&tmA);
            if (FMT != kQ6K) tma_prefetch(&tmW);
        }
        int n_a = 0, n_r = 0;   // loads issued, for the drain on abort
        bool ok = true;
        for (int ks = 0; ks < nks && ok; ++ks) {
            if ((ks & 3) == 0) {
                const int sb = ks >> 2, rs = sb % RAW_STAGES;
                ok = mbar_wait_warp(r_empty(rs), ((sb / RAW_STAGES) & 1) ^ 1, abort_flag, kKid, SITE_P_RAW);
                if (!ok) break;
                const uint32_t dst = sbase + L::oRaw + rs * L::kRawBytes;
                if (FMT != kQ6K) {
                    // one 2-D box of 128 rows x the super-block's bytes (q8_0: counted in
                    // 16-bit elements, the box's inner extent being limited to 256 elements)
                    if (lane == 0) {
                        mbar_arrive_expect_tx(r_full(rs), L::kRawBytes);
                        tma_load_2d(dst, &tmW, r_full(rs), sb * (FMT == kQ8_0 ? F::kBlockBytes / 2 : F::kBlockBytes),
                                    o0);
                    }
                } else {
                    // one bulk copy per row: the 16-byte-aligned 224-byte window
                    // holding the row's 210-byte block (its lead-in is skipped
                    // by the unpack); past the buffer's last full 16-byte
                    // granule the bytes are copied one by one
                    const int nrows = min(BN, O - o0);
                    const long long nbytes = (long long)O * nsb * F::kBlockBytes;
                    uint32_t mine = 0;
                    for (int r = lane; r < nrows; r += 32) {
                        const long long start = ((long long)(o0 + r) * nsb + sb) * F::kBlockBytes;
                        const long long a = start & ~15ll;
                        uint32_t sz = F::kRawRow;
                        if (a + F::kRawRow > nbytes) {
                            sz = (uint32_t)((nbytes - a) & ~15ll);
                            uint8_t *drow = smem + L::oRaw + rs * L::kRawBytes + r * F::kRawRow;
                            for (long long i = a + sz; i < start + F::kBlockBytes; ++i) drow[i - a] = p.w[i];
                        }
                        mine += sz;
                    }
                    mbar_arrive_expect_tx(r_full(rs), mine);
                    for (int r = lane; r < nrows; r += 32) {
                        const long long start = ((long long)(o0 + r) * nsb + sb) * F::kBlockBytes;
                        const long long a = start & ~15ll;
                        uint32_t sz = F::kRawRow;
                        if (a + F::kRawRow > nbytes) sz = (uint32_t)((nbytes - a) & ~15ll);
                        bulk_load(dst + r * F::kRawRow, p.w + a, sz, r_full(rs));
                    }
                }
                ++n_r;
            }
            const int s = ks % STAGES;
            ok = mbar_wait_warp(st_empty(s), ((ks / STAGES) & 1) ^ 1, abort_flag, kKid, SITE_P_STAGE);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(a_full(s), A_BYTES);
                tma_load_2d(sbase + L::oA + s * A_BYTES, &tmA, a_full(s), ks * BK, t0);
            }
            ++n_a;
            __syncwarp();
        }
        if (!ok) {
            // let the copies already issued land before the block can exit
            for (int i = max(0, n_a - STAGES); i < n_a; ++i) wait_drain(a_full(i % STAGES), (i / STAGES) & 1);
            for (int i = max(0, n_r - RAW_STAGES); i < n_r; ++i)
                wait_drain(r_full(i % RAW_STAGES), (i / RAW_STAGES) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer --
        if (lane == 0) {
            bool ok = true;
            int acc = 0;
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % STAGES;
                const uint32_t par = (ks / STAGES) & 1;
                ok = mbar_wait(a_full(s), par, abort_flag, kKid, SITE_M_A) &&
                     mbar_wait(b_full(s), par, abort_flag, kKid, SITE_M_B);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_base = sbase + L::oA + s * A_BYTES;
                const uint32_t b_base = sbase + L::oB + s * B_BYTES;
#pragma unroll
                for (int g = 0; g < L::kSubPerStage; ++g, ++acc) {
                    const int slot = acc % ACC_SLOTS;
                    ok = mbar_wait(acc_empty(slot), ((acc / ACC_SLOTS) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < F::kKSub / 16; ++kk) {
                        const uint32_t koff = (uint32_t)(g * (F::kKSub / 16) + kk) * 32u;
                        umma_f16(tmem_base + slot * BN, sdesc_k_sw128(a_base + koff),
                                 sdesc_k_sw128(b_base + koff), kIdesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(acc_full(slot));
                }
                if (!ok) break;
                umma_commit(st_empty(s));
            }
            umma_commit(mma_done);
            if (!wait_drain(mma_done, 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        const int r = threadIdx.x - UNPACK_WARP0 * 32;   // tile row 0..127
        const int o = o0 + r;
        const bool row_ok = o < O;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RAW_STAGES, ss = sb % SDS_STAGES;
            ok = mbar_wait(r_full(rs), (sb / RAW_STAGES) & 1, abort_flag, kKid, SITE_U_RAW) &&
                 mbar_wait(s_empty(ss), ((sb / SDS_STAGES) & 1) ^ 1, abort_flag, kKid, SITE_U_SDS);
            if (!ok) break;
            const uint8_t *raw = smem + L::oRaw + rs * L::kRawBytes + r * F::kRawRow;
            uint8_t *sds = smem + L::oSds + ss * L::kSdsBytes;
            if (FMT == kQ8_0) {
                // the eight blocks' d (rows past O arrive zero-filled)
                float *sd1 = reinterpret_cast<float *>(sds);
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    sd1[g * BN + r] = __half2float(__ushort_as_half(
                        (unsigned short)(raw[34 * g] | (raw[34 * g + 1] << 8))));
            } else if (FMT == kQ4K || FMT == kQ5K) {
                // header: d, dmin (f16), 12 bytes of 6-bit scales / mins
                const uint4 hd = *reinterpret_cast<const uint4 *>(raw);
                const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                const uint32_t s0 = hd.y, s1 = hd.z, s2 = hd.w;
                float2 *sd2 = reinterpret_cast<float2 *>(sds);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int sc_lo = (s0 >> (8 * j)) & 63, m_lo = (s1 >> (8 * j)) & 63;
                    const int sc_hi = ((s2 >> (8 * j)) & 15) | (((s0 >> (8 * j + 6)) & 3) << 4);
                    const int m_hi = ((s2 >> (8 * j + 4)) & 15) | (((s1 >> (8 * j + 6)) & 3) << 4);
                    sd2[j * BN + r] = make_float2(d * (float)sc_lo, -(dmin * (float)m_lo));
                    sd2[(j + 4) * BN + r] = make_float2(d * (float)sc_hi, -(dmin * (float)m_hi));
                }
            } else {
                const int lead = (int)((((long long)o * nsb + sb) * F::kBlockBytes) & 15);
                const uint8_t *blk = raw + lead;
                float *sd1 = reinterpret_cast<float *>(sds);
                const float d = row_ok ? __half2float(__ushort_as_half((unsigned short)(blk[208] | (blk[209] << 8))))
                                       : 0.0f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    sd1[u * BN + r] = row_ok ? d * (float)(int8_t)blk[192 + u] : 0.0f;
            }
            mbar_arrive(s_full(ss));

            for (int p4 = 0; p4 < 4; ++p4) {
                const int ks = sb * 4 + p4, s = ks % STAGES;
                ok = mbar_wait(st_empty(s), ((ks / STAGES) & 1) ^ 1, abort_flag, kKid, SITE_U_STAGE);
                if (!ok) break;
                uint8_t *brow = smem + L::oB + s * B_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
                if (FMT == kQ8_0) {
                    // stage p4 = blocks 2*p4, 2*p4 + 1: 64 int8 values (2-byte aligned), exact in f16
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint8_t *qb = raw + 34 * (2 * p4 + (c >> 2)) + 2 + 8 * (c & 3);
                        int v[8];
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            const uint32_t two = *reinterpret_cast<const uint16_t *>(qb + i);
                            v[i] = (int)(int8_t)(two & 0xFFu);
                            v[i + 1] = (int)(int8_t)(two >> 8);
                        }
                        uint4 q;
                        q.x = pack_h2(v[0], v[1]);
                        q.y = pack_h2(v[2], v[3]);
                        q.z = pack_h2(v[4], v[5]);
                        q.w = pack_h2(v[6], v[7]);
                        *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = q;
                    }
                } else if (FMT == kQ5K) {
                    // stage p4 = sub-blocks 2*p4 (low nibbles) and 2*p4+1 (high nibbles) of quant
                    // bytes 32*p4 .. +31 at +48, each with its fifth bit from qh at +16 (bit 2*p4 or
                    // 2*p4 + 1 of qh[l])
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(raw + 48 + 32 * p4);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(raw + 48 + 32 * p4 + 16);
                    const uint4 h0 = *reinterpret_cast<const uint4 *>(raw + 16);
                    const uint4 h1 = *reinterpret_cast<const uint4 *>(raw + 32);
                    const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                    const uint32_t hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int j = 2 * p4 + (c >> 2);            // sub-block
                        const uint32_t qa = wv[2 * (c & 3)], qb = wv[2 * (c & 3) + 1];
                        const uint32_t ba = ((hv[2 * (c & 3)] >> j) & 0x01010101u) << 4;
                        const uint32_t bb = ((hv[2 * (c & 3) + 1] >> j) & 0x01010101u) << 4;
                        const uint32_t va = ((c < 4 ? qa : (qa >> 4)) & 0x0F0F0F0Fu) | ba;
                        const uint32_t vb = ((c < 4 ? qb : (qb >> 4)) & 0x0F0F0F0Fu) | bb;
                        uint4 v;
                        v.x = u5_2(va, 0x4140u);
                        v.y = u5_2(va, 0x4342u);
                        v.z = u5_2(vb, 0x4140u);
                        v.w = u5_2(vb, 0x4342u);
                        *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = v;
                    }
                } else if (FMT == kQ4K) {
                    // stage p4 = sub-blocks 2*p4 (low nibbles, k 0..31) and 2*p4+1
                    // (high nibbles, k 32..63) of quant bytes 32*p4 .. 32*p4+31
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * p4);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * p4 + 16);
                    const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t wa = wv[2 * (c & 3)], wb = wv[2 * (c & 3) + 1];
                        uint4 v;
                        if (c < 4) {
                            v.x = nib_lo2(wa, 0x4140u);
                            v.y = nib_lo2(wa, 0x4342u);
                            v.z = nib_lo2(wb, 0x4140u);
                            v.w = nib_lo2(wb, 0x4342u);
                        } else {
                            v.x = nib_hi2(wa, 0x4140u);
                            v.y = nib_hi2(wa, 0x4342u);
                            v.z = nib_hi2(wb, 0x4140u);
                            v.w = nib_hi2(wb, 0x4342u);
                        }
                        *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = v;
                    }
                } else {
                    // stage p4: half h = p4/2, quarters g0 = 2*(p4&1), g0+1; values q-32
                    const int lead = (int)((((long long)o * nsb + sb) * F::kBlockBytes) & 15);
                    const uint8_t *blk = raw + lead;
                    const uint8_t *Lq = blk + 64 * (p4 >> 1);
                    const uint8_t *Hq = blk + 128 + 32 * (p4 >> 1);
                    const int g0 = 2 * (p4 & 1);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int g = g0 + (c >> 2), l0 = 8 * (c & 3);
                        int v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int l = l0 + i;
                            const int lb = (g & 1) ? Lq[l + 32] : Lq[l];
                            const int lo = (g >= 2) ? (lb >> 4) : (lb & 15);
                            const int hi = (Hq[l] >> (2 * g)) & 3;
                            v[i] = row_ok ? ((lo | (hi << 4)) - 32) : 0;
                        }
                        uint4 q;
                        q.x = pack_h2(v[0], v[1]);
                        q.y = pack_h2(v[2], v[3]);
                        q.z = pack_h2(v[4], v[5]);
                        q.w = pack_h2(v[6], v[7]);
                        *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = q;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(b_full(s));
            }
            if (ok) mbar_arrive(r_empty(rs));
        }
    } else {
        // --------------------------------------------------------- epilogue --
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;            // TMEM lanes this warp may read
        const int c0 = (ew >> 2) * 64;           // column half of the tile
        const int tl = quarter * 32 + lane;      // token within the tile (TMEM lane)
        const int t = t0 + tl;
        const bool tok_ok = t < T;
        float yv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) yv[i] = 0.0f;
        bool ok = true;
        int acc = 0;
        const int nsub_total = nsb * L::kSubPerSb;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int ss = sb % SDS_STAGES;
            ok = mbar_wait_warp(s_full(ss), (sb / SDS_STAGES) & 1, abort_flag, kKid, SITE_E_SDS);
            if (!ok) break;
            // this token's q8_1 scale words for the super-block (L1-resident)
            const uint32_t *dsrow = (MODE == kFold && tok_ok) ? p.ds + (size_t)t * (K / 32) + sb * 8 : nullptr;
            const uint8_t *sds = smem + L::oSds + ss * L::kSdsBytes;
#pragma unroll 1
            for (int g = 0; g < L::kSubPerSb; ++g, ++acc) {
                const int slot = acc % ACC_SLOTS;
                ok = mbar_wait_warp(acc_full(slot), (acc / ACC_SLOTS) & 1, abort_flag, kKid, SITE_E_ACC);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dword = dsrow ? __ldg(dsrow + (F::kKSub == 32 ? g : (g >> 1))) : 0u;
                const float dx = __half2float(__ushort_as_half((unsigned short)(dword & 0xFFFFu)));
                const float dma = dx * (float)(int)(int16_t)(dword >> 16);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t rv[32];
                    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(slot * BN + c0 + hh * 32), rv);
                    tmem_ld_wait(rv);
                    if (hh == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty(slot));
                    }
                    const int cbase = c0 + hh * 32;
                    if (MODE == kFold) {
                        if (FMT == kQ4K || FMT == kQ5K) {
                            const float2 *sd2 = reinterpret_cast<const float2 *>(sds) + g * BN + cbase;
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float4 sv = *reinterpret_cast<const float4 *>(sd2 + i);
                                const float c0v = __uint_as_float(rv[i]), c1v = __uint_as_float(rv[i + 1]);
                                float a0 = yv[hh * 32 + i], a1 = yv[hh * 32 + i + 1];
                                a0 = fmaf(dx * sv.x, c0v, a0);
                                a0 = fmaf(dma, sv.y, a0);
                                a1 = fmaf(dx * sv.z, c1v, a1);
                                a1 = fmaf(dma, sv.w, a1);
                                yv[hh * 32 + i] = a0;
                                yv[hh * 32 + i + 1] = a1;
                            }
                        } else {
                            const float *sd1 = reinterpret_cast<const float *>(sds) + g * BN + cbase;
#pragma unroll
                            for (int i = 0; i < 32; i += 4) {
                                const float4 sv = *reinterpret_cast<const float4 *>(sd1 + i);
                                yv[hh * 32 + i + 0] = fmaf(dx * sv.x, __uint_as_float(rv[i + 0]), yv[hh * 32 + i + 0]);
                                yv[hh * 32 + i + 1] = fmaf(dx * sv.y, __uint_as_float(rv[i + 1]), yv[hh * 32 + i + 1]);
                                yv[hh * 32 + i + 2] = fmaf(dx * sv.z, __uint_as_float(rv[i + 2]), yv[hh * 32 + i + 2]);
                                yv[hh * 32 + i + 3] = fmaf(dx * sv.w, __uint_as_float(rv[i + 3]), yv[hh * 32 + i + 3]);
                            }
                        }
                    } else if (tok_ok) {
                        const int bidx = sb * L::kSubPerSb + g;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int oc = o0 + cbase + i;
                            if (oc < O)
                                p.sub[((size_t)t * O + oc) * nsub_total + bidx] =
                                    __float2int_rn(__uint_as_float(rv[i]));
                        }
                    }
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(s_empty(ss));
        }
        if (MODE == kFold && ok && tok_ok) {
            float *yrow = p.y + (size_t)t * O + o0 + c0;
            if ((O & 3) == 0 && o0 + c0 + 64 <= O) {
#pragma unroll
                for (int i = 0; i < 64; i += 4)
                    *reinterpret_cast<float4 *>(yrow + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (o0 + c0 + i < O) yrow[i] = yv[i];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// =========================================================================
// q4_K GEMM, production form.
//
// Same data flow as above, restructured so that the per-(token, row,
// sub-block) work left on the CUDA cores is one packed FMA and no role waits
// on another's bookkeeping:
//   * unpack warps multiply each 4-bit quant by its 6-bit sub-block scale
//     while converting it (sc*q <= 945 is exact in f16), so the tensor core
//     produces C'_b = sum (sc_b*q)*a = sc_b*C_b exactly;
//   * the epilogue accumulates acc = sum_b dx_b*C'_b over the 8 sub-blocks of
//     a super-block (dx_b is per token = per TMEM lane, a scalar of the
//     thread) and adds d*acc into the running output Y once per super-block;
//   * the min term sum_b (dx_b*ssum_b)*(-(dmin*m_b)) is a GEMM over the
//     sub-block index.  It runs on the tensor core in tf32 with each factor
//     split into a high and a low tf32 part (both factors are exact f32
//     products of an f16 value and a small integer, so the split loses only
//     the low*low term, ~2^-22 relative) and accumulates straight into Y's
//     TMEM columns: the first super-block's min term also initialises Y;
//   * two scale warps build the min-term operands and the per-row d and
//     per-token dx of super-block sb+1 while sb is being multiplied.
// TMEM columns: [0,384) three rotating sub-block accumulators, [384,512) Y.
// Warps: 0 TMA producer, 1 MMA issuer, 2-5 unpack, 6-13 epilogue, 14-15 scale.
// =========================================================================
namespace q4 {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int SCALE_WARP0 = 14;
constexpr int STG = 4;                           // operand ring (A and B tiles)
constexpr int RSTG = 3;                          // raw super-block ring
constexpr int SSTG = 2;                          // scale / min-operand ring
constexpr int NACC = 3;                          // rotating sub-block accumulators
constexpr uint32_t TM_ACC = 0, TM_Y = NACC * BN;
static_assert(TM_Y + BN <= 512, "TMEM budget");
constexpr uint32_t RAW_BYTES = BN * 144;
constexpr uint32_t MIN_OP_BYTES = 128 * 64;                       // 128 rows x 16 tf32 (8 hi, 8 lo)
constexpr uint32_t SDS_D = 2 * MIN_OP_BYTES;                      // d[BN] f32
constexpr uint32_t SDS_DX = SDS_D + BN * 4;                       // dx[8][BM] f32
constexpr uint32_t SDS_BYTES = SDS_DX + 8 * BM * 4;
constexpr uint32_t oA = 0;
constexpr uint32_t oB = oA + STG * A_BYTES;
constexpr uint32_t oRaw = oB + STG * B_BYTES;
constexpr uint32_t oSds = oRaw + RSTG * RAW_BYTES;
constexpr uint32_t oBar = oSds + SSTG * SDS_BYTES;
// a_full, b_full, st_empty [STG]; r_full, r_empty [RSTG]; s_full, s_empty
// [SSTG]; acc_full, acc_empty [NACC]; y_ready, y_free; mma_done
constexpr int kNumBars = 3 * STG + 2 * RSTG + 2 * SSTG + 2 * NACC + 3;
constexpr uint32_t oMisc = oBar + kNumBars * 8;
constexpr uint32_t kDynSmem = oMisc + 16 + 1024;
static_assert(kDynSmem <= 232448, "shared memory budget");
static_assert(oRaw % 1024 == 0 && RAW_BYTES % 1024 == 0, "raw ring alignment");
static_assert(oSds % 16 == 0 && SDS_BYTES % 16 == 0, "min operands must be 16-byte aligned");

// One row of a min-term operand in the no-swizzle K-major layout: 16 tf32
// (hi[0..7], lo[0..7]) as four 16-byte core-matrix rows; core matrices are
// 128 bytes apart along K and 8-row groups 512 bytes apart.
__device__ __forceinline__ void put_min_row(uint8_t *base, int r, const float (&h)[8], const float (&l)[8])
{
    uint8_t *q = base + (r >> 3) * 512 + (r & 7) * 16;
    *reinterpret_cast<float4 *>(q + 0) = make_float4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<float4 *>(q + 128) = make_float4(h[4], h[5], h[6], h[7]);
    *reinterpret_cast<float4 *>(q + 256) = make_float4(l[0], l[1], l[2], l[3]);
    *reinterpret_cast<float4 *>(q + 384) = make_float4(l[4], l[5], l[6], l[7]);
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

// (1024 + q) * m + a for the two nibbles selected into the 16-bit halves
__device__ __forceinline__ uint32_t nib2(uint32_t w, uint32_t sel, uint32_t mask, __half2 m, __half2 a)
{
    const uint32_t pr = __byte_perm(w, 0u, sel);
    const uint32_t h = (pr & mask) | 0x64006400u;
    return h2bits(__hfma2(*reinterpret_cast<const __half2 *>(&h), m, a));
}

// the 6-bit scale (sc) and min (mm) of sub-block j from the 12 packed bytes
// held in three words s0 (bytes 0-3), s1 (4-7), s2 (8-11)
__device__ __forceinline__ void q4K_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, int &sc, int &mm)
{
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        mm = (s1 >> (8 * j)) & 63;
    } else {
        const int i = j - 4;
        sc = ((s2 >> (8 * i)) & 15) | (((s0 >> (8 * i + 6)) & 3) << 4);
        mm = ((s2 >> (8 * i + 4)) & 15) | (((s1 >> (8 * i + 6)) & 3) << 4);
    }
}

}  // namespace q4

__global__ void __launch_bounds__(q4::NTHREADS, 1)
    mmq_q4K_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const Params p)
{
    using namespace q4;
    constexpr int kKid = 7;
    constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
    constexpr uint32_t kIdescTf32 = idesc_tf32_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int T = p.T, K = p.K, O = p.O;
    const int nks = K / BK, nsb = K / 256;

    const uint32_t bar0 = sbase + oBar;
    auto a_full = [&](int s) { return bar0 + 8u * s; };
    auto b_full = [&](int s) { return bar0 + 8u * (STG + s); };
    auto st_empty = [&](int s) { return bar0 + 8u * (2 * STG + s); };
    auto r_full = [&](int s) { return bar0 + 8u * (3 * STG + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (3 * STG + RSTG + s); };
    auto s_full = [&](int s) { return bar0 + 8u * (3 * STG + 2 * RSTG + s); };
    auto s_empty = [&](int s) { return bar0 + 8u * (3 * STG + 2 * RSTG + SSTG + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (3 * STG + 2 * RSTG + 2 * SSTG + s); };
    auto acc_empty = [&](int s) { return bar0 + 8u * (3 * STG + 2 * RSTG + 2 * SSTG + NACC + s); };
    const uint32_t y_ready = bar0 + 8u * (kNumBars - 3);
    const uint32_t y_free = bar0 + 8u * (kNumBars - 2);
    const uint32_t mma_done = bar0 + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + oMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STG; ++s) {
            mbar_init(a_full(s), 1);
            mbar_init(b_full(s), 128);
            mbar_init(st_empty(s), 1);
        }
        for (int s = 0; s < RSTG; ++s) {
            mbar_init(r_full(s), 1);
            mbar_init(r_empty(s), 128 + 64);                // unpack and scale threads
        }
        for (int s = 0; s < SSTG; ++s) {
            mbar_init(s_full(s), 64);                       // scale threads
            mbar_init(s_empty(s), NUM_EPI_WARPS + 1);       // epilogue warps + the MMA's commit
        }
        for (int s = 0; s < NACC; ++s) {
            mbar_init(acc_full(s), 1);
            mbar_init(acc_empty(s), NUM_EPI_WARPS);
        }
        mbar_init(y_ready, 1);
        mbar_init(y_free, NUM_EPI_WARPS);
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer --
        // raw super-block sb+1 is requested when stage 4*sb is, so its scales
        // can be prepared a super-block ahead of the multiplications
        if (lane == 0) {
            tma_prefetch(&tmA);
            tma_prefetch(&tmW);
        }
        int n_a = 0, n_r = 0;
        bool ok = true;
        auto issue_raw = [&](int sb) -> bool {
            const int rs = sb % RSTG;
            if (!mbar_wait_warp(r_empty(rs), ((sb / RSTG) & 1) ^ 1, abort_flag, kKid, SITE_P_RAW)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(r_full(rs), RAW_BYTES);
                tma_load_2d(sbase + oRaw + rs * RAW_BYTES, &tmW, r_full(rs), sb * 144, o0);
            }
            ++n_r;
            return true;
        };
        ok = issue_raw(0);
        for (int ks = 0; ks < nks && ok; ++ks) {
            if ((ks & 3) == 0 && (ks >> 2) + 1 < nsb) {
                ok = issue_raw((ks >> 2) + 1);
                if (!ok) break;
            }
            const int s = ks % STG;
            ok = mbar_wait_warp(st_empty(s), ((ks / STG) & 1) ^ 1, abort_flag, kKid, SITE_P_STAGE);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(a_full(s), A_BYTES);
                tma_load_2d(sbase + oA + s * A_BYTES, &tmA, a_full(s), ks * BK, t0);
            }
            ++n_a;
            __syncwarp();
        }
        if (!ok) {
            for (int i = max(0, n_a - STG); i < n_a; ++i) wait_drain(a_full(i % STG), (i / STG) & 1);
            for (int i = max(0, n_r - RSTG); i < n_r; ++i) wait_drain(r_full(i % RSTG), (i / RSTG) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer --
        if (lane == 0) {
            bool ok = true;
            int acc = 0;   // sub-block accumulator n lives in slot n % NACC
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % STG;
                const uint32_t par = (ks / STG) & 1;
                ok = mbar_wait(a_full(s), par, abort_flag, kKid, SITE_M_A) &&
                     mbar_wait(b_full(s), par, abort_flag, kKid, SITE_M_B);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_base = sbase + oA + s * A_BYTES;
                const uint32_t b_base = sbase + oB + s * B_BYTES;
#pragma unroll
                for (int g = 0; g < 2; ++g, ++acc) {
                    const int slot = acc % NACC;
                    ok = mbar_wait(acc_empty(slot), ((acc / NACC) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t koff = (uint32_t)(2 * g + kk) * 32u;
                        umma_f16(tmem_base + TM_ACC + slot * BN, sdesc_k_sw128(a_base + koff),
                                 sdesc_k_sw128(b_base + koff), kIdesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(acc_full(slot));
                }
                if (!ok) break;
                umma_commit(st_empty(s));
                if ((ks & 3) == 3) {
                    // min term of super-block sb straight into Y:
                    // Y (+)= A_min . B_min^T as hi.hi + hi.lo + lo.hi
                    const int sb = ks >> 2, ss = sb % SSTG;
                    ok = mbar_wait(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS) &&
                         (sb == 0 || mbar_wait(y_free, (sb - 1) & 1, abort_flag, kKid, SITE_M_ACC));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t am = sbase + oSds + ss * SDS_BYTES, bm = am + MIN_OP_BYTES;
                    const uint32_t ya = tmem_base + TM_Y;
                    umma_tf32(ya, sdesc_k_none(am, 128, 512), sdesc_k_none(bm, 128, 512), kIdescTf32,
                              sb > 0 ? 1u : 0u);
                    umma_tf32(ya, sdesc_k_none(am, 128, 512), sdesc_k_none(bm + 256, 128, 512), kIdescTf32, 1u);
                    umma_tf32(ya, sdesc_k_none(am + 256, 128, 512), sdesc_k_none(bm, 128, 512), kIdescTf32, 1u);
                    umma_commit(y_ready);
                    umma_commit(s_empty(ss));
                }
            }
            umma_commit(mma_done);
            if (!wait_drain(mma_done, 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        const int r = threadIdx.x - UNPACK_WARP0 * 32;   // weight row of the B tile
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RSTG;
            ok = mbar_wait(r_full(rs), (sb / RSTG) & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            const uint8_t *raw = smem + oRaw + rs * RAW_BYTES + r * 144;
            const uint4 hd = *reinterpret_cast<const uint4 *>(raw);
#pragma unroll
            for (int p4 = 0; p4 < 4; ++p4) {
                const int ks = sb * 4 + p4, s = ks % STG;
                int sc_lo, sc_hi, unused;
                q4K_scale_min(hd.y, hd.z, hd.w, 2 * p4, sc_lo, unused);
                q4K_scale_min(hd.y, hd.z, hd.w, 2 * p4 + 1, sc_hi, unused);
                // sub-block 2*p4 (low nibbles, k 0..31): (1024+q)*sc - 1024*sc
                // sub-block 2*p4+1 (high nibbles, k 32..63): (1024+16q)*(sc/16) - 64*sc
                const float slo = (float)sc_lo, shi = (float)sc_hi;
                const __half2 mlo = __float2half2_rn(slo), alo = __float2half2_rn(-1024.0f * slo);
                const __half2 mhi = __float2half2_rn(shi * 0.0625f), ahi = __float2half2_rn(-64.0f * shi);
                const uint4 w0 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * p4);
                const uint4 w1 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * p4 + 16);
                ok = mbar_wait(st_empty(s), ((ks / STG) & 1) ^ 1, abort_flag, kKid, SITE_U_STAGE);
                if (!ok) break;
                const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint8_t *brow = smem + oB + s * B_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t wa = wv[2 * (c & 3)], wb = wv[2 * (c & 3) + 1];
                    const uint32_t mask = c < 4 ? 0x000F000Fu : 0x00F000F0u;
                    const __half2 m2 = c < 4 ? mlo : mhi, a2 = c < 4 ? alo : ahi;
                    uint4 v;
                    v.x = nib2(wa, 0x4140u, mask, m2, a2);
                    v.y = nib2(wa, 0x4342u, mask, m2, a2);
                    v.z = nib2(wb, 0x4140u, mask, m2, a2);
                    v.w = nib2(wb, 0x4342u, mask, m2, a2);
                    *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(b_full(s));
            }
            if (ok) mbar_arrive(r_empty(rs));
        }
    } else if (warp < SCALE_WARP0) {
        // --------------------------------------------------------- epilogue --
        // Thread = one token (TMEM lane) x 64 weight rows (columns).
        //   per sub-block b:  acc += dx_b * C'_b             (packed FMA)
        //   per super-block:  Y = Y + d*acc  with Y in TMEM already holding
        //                     the min terms; the last super-block writes Y
        //                     to global memory instead
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;
        const int c0 = (ew >> 2) * 64;
        const int tl = quarter * 32 + lane;
        const int t = t0 + tl;
        const bool tok_ok = t < T;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float acc[64];
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int ss = sb % SSTG;
            ok = mbar_wait_warp(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS);
            if (!ok) break;
            const float *dxs = reinterpret_cast<const float *>(smem + oSds + ss * SDS_BYTES + SDS_DX);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int n = sb * 8 + g;
                const int slot = n % NACC;
                ok = mbar_wait_warp(acc_full(slot), (n / NACC) & 1, abort_flag, kKid, SITE_E_ACC);
                if (!ok) break;
                tc_fence_after();
                const float dx = dxs[g * BM + tl];
                const float2 dx2 = make_float2(dx, dx);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t rv[32];
                    tmem_ld32(tmem_base + lane_off + TM_ACC + (uint32_t)(slot * BN + c0 + hh * 32), rv);
                    tmem_ld_wait(rv);
                    if (hh == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty(slot));
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 cv = make_float2(__uint_as_float(rv[i]), __uint_as_float(rv[i + 1]));
                        float2 a = make_float2(acc[hh * 32 + i], acc[hh * 32 + i + 1]);
                        a = (g == 0) ? __fmul2_rn(cv, dx2) : __ffma2_rn(cv, dx2, a);
                        acc[hh * 32 + i] = a.x;
                        acc[hh * 32 + i + 1] = a.y;
                    }
                }
            }
            if (!ok) break;
            ok = mbar_wait_warp(y_ready, sb & 1, abort_flag, kKid, SITE_E_ACC);
            if (!ok) break;
            tc_fence_after();
            const float *dv = reinterpret_cast<const float *>(smem + oSds + ss * SDS_BYTES + SDS_D) + c0;
            const bool last = sb == nsb - 1;
            float *yrow = p.y + (size_t)(tok_ok ? t : 0) * O + o0 + c0;
            const bool vec = (O & 3) == 0 && o0 + c0 + 64 <= O;
#pragma unroll
            for (int q = 0; q < 4; ++q) {          // 16-column chunks: Y = Y + d*acc
                uint32_t yv[16];
                const uint32_t ya = tmem_base + lane_off + TM_Y + c0 + q * 16;
                tmem_ld16(ya, yv);
                tmem_ld_wait16(yv);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dv + q * 16 + i);
                    const float2 y0 = __ffma2_rn(make_float2(acc[q * 16 + i], acc[q * 16 + i + 1]),
                                                 make_float2(d4.x, d4.y),
                                                 make_float2(__uint_as_float(yv[i]), __uint_as_float(yv[i + 1])));
                    const float2 y1 = __ffma2_rn(make_float2(acc[q * 16 + i + 2], acc[q * 16 + i + 3]),
                                                 make_float2(d4.z, d4.w),
                                                 make_float2(__uint_as_float(yv[i + 2]), __uint_as_float(yv[i + 3])));
                    yv[i] = __float_as_uint(y0.x);
                    yv[i + 1] = __float_as_uint(y0.y);
                    yv[i + 2] = __float_as_uint(y1.x);
                    yv[i + 3] = __float_as_uint(y1.y);
                }
                if (!last) {
                    tmem_st16(ya, yv);
                } else if (tok_ok) {
                    if (vec) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(yrow + q * 16 + i) =
                                make_float4(__uint_as_float(yv[i]), __uint_as_float(yv[i + 1]),
                                            __uint_as_float(yv[i + 2]), __uint_as_float(yv[i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (o0 + c0 + q * 16 + i < O) yrow[q * 16 + i] = __uint_as_float(yv[i]);
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(y_free);
                mbar_arrive(s_empty(ss));
            }
        }
    } else {
        // ------------------------------------------------------- scale warps --
        // Per super-block, for weight rows r and r+64 of the tile: d (f32) and
        // the min-term operand row (-(dmin*m_j) split hi/lo); for tokens r and
        // r+64: dx_j (f32) and the min-term operand row (dx_j*ssum_j split
        // hi/lo).  The q8_1 words are fetched a super-block ahead.
        const int sr = threadIdx.x - SCALE_WARP0 * 32;   // 0..63
        uint4 dsn[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = t0 + sr + 64 * h;
            dsn[h][0] = dsn[h][1] = make_uint4(0u, 0u, 0u, 0u);
            if (t < T) {
                const uint4 *dp = reinterpret_cast<const uint4 *>(p.ds + (size_t)t * (K / 32));
                dsn[h][0] = __ldg(dp);
                dsn[h][1] = __ldg(dp + 1);
            }
        }
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RSTG, ss = sb % SSTG;
            ok = mbar_wait(r_full(rs), (sb / RSTG) & 1, abort_flag, kKid, SITE_U_RAW) &&
                 mbar_wait(s_empty(ss), ((sb / SSTG) & 1) ^ 1, abort_flag, kKid, SITE_U_SDS);
            if (!ok) break;
            uint8_t *slot = smem + oSds + ss * SDS_BYTES;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = sr + 64 * h;
                const uint4 hd = *reinterpret_cast<const uint4 *>(smem + oRaw + rs * RAW_BYTES + r * 144);
                const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                reinterpret_cast<float *>(slot + SDS_D)[r] = d;
                float bh[8], bl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    int sc, mm;
                    q4K_scale_min(hd.y, hd.z, hd.w, j, sc, mm);
                    const float v = -(dmin * (float)mm);            // exact: 11-bit x 6-bit
                    bh[j] = to_tf32(v);
                    bl[j] = to_tf32(v - bh[j]);
                }
                put_min_row(slot + MIN_OP_BYTES, r, bh, bl);
                const uint32_t w[8] = {dsn[h][0].x, dsn[h][0].y, dsn[h][0].z, dsn[h][0].w,
                                       dsn[h][1].x, dsn[h][1].y, dsn[h][1].z, dsn[h][1].w};
                float ah[8], al[8];
                float *dxs = reinterpret_cast<float *>(slot + SDS_DX);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float dx = __half2float(__ushort_as_half((unsigned short)(w[j] & 0xFFFFu)));
                    const float v = dx * (float)(int)(int16_t)(w[j] >> 16);   // exact: 11-bit x 12-bit
                    ah[j] = to_tf32(v);
                    al[j] = to_tf32(v - ah[j]);
                    dxs[j * BM + r] = dx;
                }
                put_min_row(slot, r, ah, al);
                const int t = t0 + r;
                if (t < T && sb + 1 < nsb) {
                    const uint4 *dp = reinterpret_cast<const uint4 *>(p.ds + (size_t)t * (K / 32) + (sb + 1) * 8);
                    dsn[h][0] = __ldg(dp);
                    dsn[h][1] = __ldg(dp + 1);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(s_full(ss));
            mbar_arrive(r_empty(rs));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// =========================================================================
// q4_K GEMM with super-block accumulation (production).
//
// The sum over a super-block's 8 sub-blocks of dx_b*sc_b*C_b is computed by
// the tensor core itself: the activation operand is the dequantised q8_1
// value v = f32(d16)*q split into two exact f16 planes (v = hi + lo, see the
// quantiser), the weight operand is sc*q (exact), so each product is exact in
// f32 and one TMEM accumulator per super-block receives
//     D_sb[t][o] = sum_{k in sb} v[t][k] * sc_b(o)*q[o][k]
// through two MMAs per 16-k step (hi plane, lo plane).  The epilogue then
// needs one packed FMA per output per super-block, Y += d*D_sb (Y held in
// registers).  The min term rides in the same accumulator: the tensor core
// also adds sum_j (dx_j*ssum_j) * (-(dmin*m_j)/d) (split-tf32 MMAs over the
// sub-block index), so that d*D_sb carries both terms of the super-block.
// For rows with d == 0 the weight operand is zero and the min operand is
// divided by 1 instead.  The per-sub-block integer dots are not formed here
// (see mmq_q4K_kernel / the sub-block diagnostics for those); the result
// differs from them only in f32 rounding.
//
// Two issuing threads.  On sm_103a issuing a 128x128x16 MMA occupies the
// issuing thread for most of the 64 cycles the MMA executes, and any
// dependent shared-memory access of that thread (an mbarrier wait included)
// waits behind its queued MMAs, so a single issuer that synchronises once
// per stage leaves the tensor pipe idle for a good part of every stage.  Two
// threads in warps on different SM sub-partitions therefore issue the 64-k
// stages alternately (even stages / odd stages), each into accumulators of
// its own, and the epilogue adds the two: while one synchronises, the other's
// MMAs keep the pipe busy, and every accumulator still sees its MMAs in one
// fixed order, so results are reproducible bit for bit.
// Each stage has a single "full" barrier (TMA bytes of both activation
// planes + the 128 unpack threads' arrivals) and a single "empty" barrier.
// The MMA issuers request the activation tiles: when an issuer has seen its
// previous stage ks - 2 complete, the slot of stage ks + 1 is free, and it
// issues that stage's TMA before its own stage ks, the earliest moment the
// slot allows (an unpack warp, busy converting, would reach it later and put
// the copy's latency on the critical path).  Stage ks uses
// operand slot ks % STG but barriers ks % (2 STG): a parity wait can only
// tell apart phases one apart, so every waiter must see each phase of the
// barriers it waits on.  With one barrier per slot and an odd ring, stages
// ks and ks + STG belong to different issuers, and an issuer waiting for
// stage ks + 2 STG while stage ks + STG was still filling would pass at once
// on the parity of the phase before it.  With 2 STG barriers all stages on
// one barrier belong to one issuer.  The raw weight
// super-blocks (128 rows x 144 bytes) arrive by TMA one super-block ahead;
// the unpack and scale threads copy what they need to registers at the
// start of a super-block and release the raw slot at once.
// TMEM: [0,256) even-stage accumulators, [256,512) odd-stage accumulators,
// two super-blocks each (rotating).
// Warps: 1 and 14 MMA issuers (even / odd stages; + activation TMA), 2-5
// unpack (+ raw weight TMA), 6-13 epilogue, 0 and 15 scale.
// =========================================================================
namespace q4s {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int MMA_WARP_ODD = 14;
constexpr int SCALE_WARP_B = 15;                  // scale warps: 0 and 15
constexpr int STG = 3;                            // operand ring: A hi, A lo, B per 64-k stage
constexpr int RSTG = 2;                           // raw weight super-block ring
constexpr int SSTG = 2;                           // scale / min-operand ring
constexpr int NACC = 2;                           // rotating super-block accumulators per issuer
constexpr uint32_t TM_EVEN = 0, TM_ODD = NACC * BN;
static_assert(TM_ODD + NACC * BN <= 512, "TMEM budget");
constexpr uint32_t A_STAGE = 2 * A_BYTES;         // hi and lo planes
constexpr uint32_t STAGE_BYTES = A_STAGE + B_BYTES;
constexpr uint32_t MIN_OP_BYTES = 128 * 64;
constexpr uint32_t SDS_D = 2 * MIN_OP_BYTES;
constexpr uint32_t SDS_BYTES = SDS_D + BN * 4;
constexpr int SBAR = 2 * STG;                     // full / empty barriers: stage ks uses ks % SBAR
constexpr uint32_t oStage = 0;
constexpr uint32_t oRaw = oStage + STG * STAGE_BYTES;   // then the raw ring, scale ring and barriers (SbLayout)
// full, empty [SBAR]; s_full [SSTG]; acc_full, acc_empty [NACC] (shared by the
// even and odd accumulators of a super-block); r_full, r_empty [RSTG];
// done [2] (each issuer's stage completions); mma_done
constexpr int kNumBars = 2 * SBAR + SSTG + 2 * NACC + 2 * RSTG + 2 + 1;
static_assert(STAGE_BYTES % 1024 == 0 && oRaw % 1024 == 0 && SDS_BYTES % 16 == 0, "ring alignment");
static_assert(NACC >= SSTG, "a scale slot is rewritten only after its accumulator was released");

// Per-format part of the layout: the raw ring holds the rows' whole blocks
// (q4_K 144 bytes, q5_K 176), everything after it moves with its size.
template <int FMT>
struct SbLayout {
    static constexpr int RAW_ROW = FMT == kQ5K ? 176 : 144;
    static constexpr uint32_t RAW_BYTES = BN * RAW_ROW;
    static constexpr uint32_t oSds = oRaw + RSTG * RAW_BYTES;
    static constexpr uint32_t oBar = oSds + SSTG * SDS_BYTES;
    static constexpr uint32_t oMisc = oBar + kNumBars * 8;
    static constexpr uint32_t kDynSmem = oMisc + 16 + 1024;
    static_assert(kDynSmem <= 232448, "shared memory budget");
    static_assert(RAW_BYTES % 1024 == 0 && oSds % 16 == 0, "ring alignment");
};

// Two f16 values sc*q from the two bytes of x selected by sel (x holds the
// quants already masked: q in the low nibble, or 16q in the high nibble):
// the bytes become the low halves of 1024 + b, then one packed FMA with
// (m, a) = (sc, -1024 sc) or (sc/16, -64 sc).  Every step is exact.
__device__ __forceinline__ uint32_t magic2(uint32_t x, uint32_t sel, __half2 m, __half2 a)
{
    const uint32_t h = __byte_perm(x, 0x64646464u, sel);
    return q4::h2bits(__hfma2(*reinterpret_cast<const __half2 *>(&h), m, a));
}

// SwiGLU pass: gate [128][GU_STRIDE] then up [128][GU_STRIDE] f32 in the operand
// ring (a row stride of 17 x 16 bytes puts eight consecutive tokens' 16-byte
// accesses in eight different bank groups)
constexpr int GU_STRIDE = 68;
static_assert(2 * BM * GU_STRIDE * 4 <= STG * STAGE_BYTES, "SwiGLU staging fits the operand ring");

// silu(g) * u in f32: g / (1 + e^-g) with each operation rounded once (no contraction)
__device__ __forceinline__ float swiglu_f32(float g, float u)
{
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// round_half_away(x / d) with the quotient rounded to f32 as IEEE division
// does, without the division where the result cannot depend on it: with
// r = fl(1/d), z = fl(x * r) is within |y| * 2^-22 of the correctly rounded
// quotient fl(y) (y = x / d), which for |y| <= 127.5 is below 2^-14; unless z
// lies within 2^-14 of a half-integer (or r is not a finite normal number)
// both round to the same integer, and otherwise the IEEE quotient is taken.
__device__ __forceinline__ int q8_round_quotient(float x, float d, float r)
{
    const float z = x * r;
    const float a = fabsf(z);
    if (r < 1e30f && a < 128.0f && fabsf(a - floorf(a) - 0.5f) > 0x1p-14f) return (int)roundf(z);
    return (int)roundf(__fdiv_rn(x, d));
}

}  // namespace q4s

// SWIGLU: the tile's output is not stored as y but finished as silu(gate)*up and
// quantised to q8_1 (Params::h_xa).
// FMT: kQ4K, or kQ5K (the same header and scale packing, a 5-bit quant whose
// fifth bits come from a 32-byte qh plane: sc*q <= 1953 is still exact in f16).
template <int FMT, bool SWIGLU>
__global__ void __launch_bounds__(q4s::NTHREADS, 1)
    mmq_q4K_sb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const Params p)
{
    using namespace q4s;
    using SL = SbLayout<FMT>;
    constexpr int RAW_ROW = SL::RAW_ROW;
    constexpr uint32_t RAW_BYTES = SL::RAW_BYTES, oSds = SL::oSds, oBar = SL::oBar, oMisc = SL::oMisc;
    constexpr int kKid = 9;
    constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
    constexpr uint32_t kIdescTf32 = idesc_tf32_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int T = p.T, K = p.K, O = p.O;
    // this CTA's super-blocks: [sb_base, sb_base + nsb) of the K/256 in a row
    const int nsb_row = K / 256;
    const int sb_base = blockIdx.z * p.sb_per_split;
    const int nsb = min(nsb_row - sb_base, p.sb_per_split);
    const int nks = nsb * 4;

    const uint32_t bar0 = sbase + oBar;
    auto full = [&](int b) { return bar0 + 8u * b; };
    auto empty = [&](int b) { return bar0 + 8u * (SBAR + b); };
    auto s_full = [&](int s) { return bar0 + 8u * (2 * SBAR + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (2 * SBAR + SSTG + s); };
    auto acc_empty = [&](int s) { return bar0 + 8u * (2 * SBAR + SSTG + NACC + s); };
    auto r_full = [&](int s) { return bar0 + 8u * (2 * SBAR + SSTG + 2 * NACC + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (2 * SBAR + SSTG + 2 * NACC + RSTG + s); };
    auto done = [&](int s) { return bar0 + 8u * (2 * SBAR + SSTG + 2 * NACC + 2 * RSTG + s); };
    const uint32_t mma_done = bar0 + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + oMisc + 4);
    auto stage_a = [&](int s) { return sbase + oStage + (uint32_t)s * STAGE_BYTES; };

    if (threadIdx.x == 0) {
        for (int b = 0; b < SBAR; ++b) {
            mbar_init(full(b), 1 + 128);                    // TMA issue (with its bytes) + unpack threads
            mbar_init(empty(b), 1);                         // the commit of the stage's issuer
        }
        for (int s = 0; s < SSTG; ++s) mbar_init(s_full(s), 64);   // scale threads
        for (int s = 0; s < NACC; ++s) {
            mbar_init(acc_full(s), 2);                      // both issuers' commits
            mbar_init(acc_empty(s), NUM_EPI_WARPS);         // after the epilogue has also read d
        }
        for (int s = 0; s < RSTG; ++s) {
            mbar_init(r_full(s), 1);
            mbar_init(r_empty(s), 128 + 64);                // unpack and scale threads
        }
        mbar_init(done(0), 1);
        mbar_init(done(1), 1);
        mbar_init(mma_done, 2);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 1 || warp == MMA_WARP_ODD) {
        // ----------------------------------------------------- MMA issuers --
        if (lane == 0) {
            const int me = warp == 1 ? 0 : 1;   // stages with ks % 2 == me
            bool ok = true;
            // activation tiles of stage k: [2T][K] tensor, hi plane rows 0..T-1, lo plane rows T..2T-1
            auto load_a = [&](int k) {
                mbar_arrive_expect_tx(full(k % SBAR), A_STAGE);
                tma_load_2d(stage_a(k % STG), &tmA, full(k % SBAR), (sb_base * 4 + k) * BK, t0);
                tma_load_2d(stage_a(k % STG) + A_BYTES, &tmA, full(k % SBAR), (sb_base * 4 + k) * BK, T + t0);
            };
            int last_a = -1;   // last stage whose activation tiles this thread requested
            if (me == 0) {
                tma_prefetch(&tmA);
                for (int k = 0; k < STG && k < nks; ++k) load_a(k);
                last_a = min(STG, nks) - 1;
            }
            for (int ks = me; ks < nks && ok; ks += 2) {
                const int s = ks % STG, fb = ks % SBAR;
                const int sb = ks >> 2, p4 = ks & 3, slot = sb % NACC;
                // Throttle: this issuer's previous stage has completed.  At most two stages
                // are then queued in the tensor pipe (the other issuer's, executing, and this
                // one), and the rest of the ring is free for loading.
                const int n_mine = ks >> 1;   // stages this issuer has issued so far
                ok = n_mine == 0 || mbar_wait(done(me), (n_mine - 1) & 1, abort_flag, kKid, SITE_M_A);
                if (!ok) break;
                // stage ks - 2 has completed, so the slot of stage ks + 1 is free
                if (ks >= 2 && ks + 1 < nks) {
                    load_a(ks + 1);
                    last_a = ks + 1;
                }
                ok = mbar_wait(full(fb), (ks / SBAR) & 1, abort_flag, kKid, SITE_M_A) &&
                     (p4 > 1 || mbar_wait(acc_empty(slot), ((sb / NACC) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC));
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_hi = stage_a(s);
                const uint64_t dh = sdesc_k_sw128(a_hi), dl = sdesc_k_sw128(a_hi + A_BYTES),
                               db = sdesc_k_sw128(a_hi + A_STAGE);
                const uint32_t d_acc = tmem_base + (me ? TM_ODD : TM_EVEN) + slot * BN;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // +32 bytes along K within the 128-byte swizzled rows = +2 in the address field
                    umma_f16(d_acc, dh + 2 * kk, db + 2 * kk, kIdesc, (p4 <= 1 && kk == 0) ? 0u : 1u);
                    umma_f16(d_acc, dl + 2 * kk, db + 2 * kk, kIdesc, 1u);
                }
                if (p4 == 3) {
                    // min term of this super-block, into the odd accumulator
                    const int ss = sb % SSTG;
                    ok = mbar_wait(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t am = sbase + oSds + ss * SDS_BYTES, bm = am + MIN_OP_BYTES;
                    umma_tf32(d_acc, sdesc_k_none(am, 128, 512), sdesc_k_none(bm, 128, 512), kIdescTf32, 1u);
                    umma_tf32(d_acc, sdesc_k_none(am, 128, 512), sdesc_k_none(bm + 256, 128, 512), kIdescTf32, 1u);
                    umma_tf32(d_acc, sdesc_k_none(am + 256, 128, 512), sdesc_k_none(bm, 128, 512), kIdescTf32, 1u);
                }
                if (p4 >= 2) umma_commit(acc_full(slot));   // this issuer's last stage of the super-block
                umma_commit(empty(fb));
                umma_commit(done(me));
            }
            umma_commit(mma_done);
            if (!wait_drain(mma_done, 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
            if (!ok)   // let this thread's activation copies in flight land before the CTA exits
                for (int i = max(0, last_a - 2 * STG + 1); i <= last_a; ++i)
                    if (i < STG ? me == 0 : ((i - 1) & 1) == me) wait_drain(full(i % SBAR), (i / SBAR) & 1);
        }
        __syncwarp();
    } else if (warp >= UNPACK_WARP0 && warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        // Thread = one weight row (rows past O arrive zero-filled).  At the
        // start of a super-block it copies the row's 144 raw bytes to
        // registers; per 64-k stage it writes the row's 64 values sc*q as f16
        // into the swizzled B tile (zeros when the row's d is zero).  Thread 0
        // also issues the raw tile one super-block ahead.
        const int r = threadIdx.x - UNPACK_WARP0 * 32;
        bool ok = true;
        int n_raw = 0;     // raw super-blocks requested (thread 0), for the drain on abort
        if (r == 0) {
            tma_prefetch(&tmW);
            mbar_arrive_expect_tx(r_full(0), RAW_BYTES);
            tma_load_2d(sbase + oRaw, &tmW, r_full(0), sb_base * RAW_ROW, o0);
            n_raw = 1;
        }
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RSTG;
            ok = mbar_wait(r_full(rs), (sb / RSTG) & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            constexpr int NCUR = RAW_ROW / 16;   // q4_K: header + 8 quant words; q5_K: + 2 qh words
            uint4 cur[NCUR];
            const uint4 *raw = reinterpret_cast<const uint4 *>(smem + oRaw + rs * RAW_BYTES + r * RAW_ROW);
#pragma unroll
            for (int i = 0; i < NCUR; ++i) cur[i] = raw[i];
            fence_proxy_async_smem();   // these reads before the next TMA write into the slot
            mbar_arrive(r_empty(rs));
            if (r == 0 && sb + 1 < nsb) {
                const int rn = (sb + 1) % RSTG;
                ok = mbar_wait(r_empty(rn), (((sb + 1) / RSTG) & 1) ^ 1, abort_flag, kKid, SITE_P_RAW);
                if (ok && !(g_inject == 1 && sb == 0)) {   // (test-only: mode 1 withholds this copy)
                    mbar_arrive_expect_tx(r_full(rn), RAW_BYTES);
                    tma_load_2d(sbase + oRaw + rn * RAW_BYTES, &tmW, r_full(rn), (sb_base + sb + 1) * RAW_ROW, o0);
                    n_raw = sb + 2;
                }
            }
            // the row's 64 values sc*q of stage p4 of this super-block as f16
            auto convert = [&](int p4, uint4 (&vv)[8]) {
                int sc_lo, sc_hi, unused;
                q4::q4K_scale_min(cur[0].y, cur[0].z, cur[0].w, 2 * p4, sc_lo, unused);
                q4::q4K_scale_min(cur[0].y, cur[0].z, cur[0].w, 2 * p4 + 1, sc_hi, unused);
                const bool d_zero = (cur[0].x & 0x7FFFu) == 0u;
                const float slo = d_zero ? 0.0f : (float)sc_lo, shi = d_zero ? 0.0f : (float)sc_hi;
                const __half2 mlo = __float2half2_rn(slo), alo = __float2half2_rn(-1024.0f * slo);
                const __half2 mhi = __float2half2_rn(shi * 0.0625f), ahi = __float2half2_rn(-64.0f * shi);
                if constexpr (FMT == kQ5K) {
                    // 5-bit values: nibble | fifth bit (bit 2*p4 or 2*p4 + 1 of qh[l]) << 4, with
                    // (m, a) = (sc, -1024 sc) for both sub-blocks
                    const __half2 mh5 = __float2half2_rn(shi), ah5 = __float2half2_rn(-1024.0f * shi);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 q = cur[3 + 2 * p4 + (c >> 1)];
                        const uint4 hq = cur[1 + (c >> 1)];
                        const uint32_t w_a = (c & 1) ? q.z : q.x, w_b = (c & 1) ? q.w : q.y;
                        const uint32_t b_a = (c & 1) ? hq.z : hq.x, b_b = (c & 1) ? hq.w : hq.y;
                        const uint32_t la = (w_a & 0x0F0F0F0Fu) | (((b_a >> (2 * p4)) & 0x01010101u) << 4);
                        const uint32_t lb = (w_b & 0x0F0F0F0Fu) | (((b_b >> (2 * p4)) & 0x01010101u) << 4);
                        const uint32_t ha = ((w_a >> 4) & 0x0F0F0F0Fu) | (((b_a >> (2 * p4 + 1)) & 0x01010101u) << 4);
                        const uint32_t hb = ((w_b >> 4) & 0x0F0F0F0Fu) | (((b_b >> (2 * p4 + 1)) & 0x01010101u) << 4);
                        vv[c] = make_uint4(q4s::magic2(la, 0x4140u, mlo, alo), q4s::magic2(la, 0x4342u, mlo, alo),
                                           q4s::magic2(lb, 0x4140u, mlo, alo), q4s::magic2(lb, 0x4342u, mlo, alo));
                        vv[c + 4] = make_uint4(q4s::magic2(ha, 0x4140u, mh5, ah5), q4s::magic2(ha, 0x4342u, mh5, ah5),
                                               q4s::magic2(hb, 0x4140u, mh5, ah5), q4s::magic2(hb, 0x4342u, mh5, ah5));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 q = cur[1 + 2 * p4 + (c >> 1)];
                        const uint32_t w_a = (c & 1) ? q.z : q.x, w_b = (c & 1) ? q.w : q.y;
                        const uint32_t la = w_a & 0x0F0F0F0Fu, lb = w_b & 0x0F0F0F0Fu;
                        const uint32_t ha = w_a & 0xF0F0F0F0u, hb = w_b & 0xF0F0F0F0u;
                        vv[c] = make_uint4(q4s::magic2(la, 0x4140u, mlo, alo), q4s::magic2(la, 0x4342u, mlo, alo),
                                           q4s::magic2(lb, 0x4140u, mlo, alo), q4s::magic2(lb, 0x4342u, mlo, alo));
                        vv[c + 4] = make_uint4(q4s::magic2(ha, 0x4140u, mhi, ahi), q4s::magic2(ha, 0x4342u, mhi, ahi),
                                               q4s::magic2(hb, 0x4140u, mhi, ahi), q4s::magic2(hb, 0x4342u, mhi, ahi));
                    }
                }
            };
            // stage p4's values are converted before waiting for its slot, and
            // stage p4 + 1's while stage p4's stores drain (before the proxy fence)
            uint4 va[8], vb[8];
            convert(0, va);
#pragma unroll
            for (int p4 = 0; p4 < 4; ++p4) {
                const int ks = sb * 4 + p4, s = ks % STG, fb = ks % SBAR;
                uint4 (&vc)[8] = (p4 & 1) ? vb : va;
                uint4 (&vn)[8] = (p4 & 1) ? va : vb;
                // slot s is free once stage ks - STG's MMAs have completed
                ok = ks < STG ||
                     mbar_wait(empty((ks - STG) % SBAR), ((ks - STG) / SBAR) & 1, abort_flag, kKid, SITE_U_STAGE);
                if (!ok) break;
                uint8_t *brow = smem + oStage + s * STAGE_BYTES + A_STAGE + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = vc[c];
                if (p4 < 3) convert(p4 + 1, vn);
                fence_proxy_async_smem();
                mbar_arrive(full(fb));
            }
        }
        if (!ok && r == 0)
            for (int i = max(0, n_raw - RSTG); i < n_raw; ++i) wait_drain(r_full(i % RSTG), (i / RSTG) & 1);
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NUM_EPI_WARPS) {
        // --------------------------------------------------------- epilogue --
        // Thread = one token (TMEM lane) x 64 weight rows; Y += d*(D_even +
        // D_odd) per super-block in registers.
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;
        const int c0 = (ew >> 2) * 64;
        const int tl = quarter * 32 + lane;
        const int t = t0 + tl;
        const bool tok_ok = t < T;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float yv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) yv[i] = 0.0f;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int slot = sb % NACC, ss = sb % SSTG;
            ok = mbar_wait_warp(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS) &&
                 mbar_wait_warp(acc_full(slot), (sb / NACC) & 1, abort_flag, kKid, SITE_E_ACC);
            if (!ok) break;
            tc_fence_after();
            const float *dv = reinterpret_cast<const float *>(smem + oSds + ss * SDS_BYTES + SDS_D) + c0;
            const uint32_t col = tmem_base + lane_off + slot * BN + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t ra[16], rb[16];
                tmem_ld16(col + TM_EVEN + q * 16, ra);
                tmem_ld16(col + TM_ODD + q * 16, rb);
                tmem_ld_wait2(ra, rb);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dv + q * 16 + i);
                    const float2 s0 = __fadd2_rn(make_float2(__uint_as_float(ra[i]), __uint_as_float(ra[i + 1])),
                                                 make_float2(__uint_as_float(rb[i]), __uint_as_float(rb[i + 1])));
                    const float2 s1 = __fadd2_rn(make_float2(__uint_as_float(ra[i + 2]), __uint_as_float(ra[i + 3])),
                                                 make_float2(__uint_as_float(rb[i + 2]), __uint_as_float(rb[i + 3])));
                    const int e = q * 16 + i;
                    const float2 y0 = __ffma2_rn(s0, make_float2(d4.x, d4.y), make_float2(yv[e], yv[e + 1]));
                    const float2 y1 = __ffma2_rn(s1, make_float2(d4.z, d4.w), make_float2(yv[e + 2], yv[e + 3]));
                    yv[e] = y0.x;
                    yv[e + 1] = y0.y;
                    yv[e + 2] = y1.x;
                    yv[e + 3] = y1.y;
                }
            }
            // both accumulators and this super-block's d have been read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(slot));
        }
        if constexpr (SWIGLU) {
            // Park the tile in shared memory for the CTA-wide SwiGLU pass at the
            // end (the operand ring is idle now that every MMA has completed):
            // columns 0..63 are the gate rows of features 64*bx .., columns
            // 64..127 the up rows of the same features.
            float *gu = reinterpret_cast<float *>(smem + oStage) + (c0 ? BM * q4s::GU_STRIDE : 0) + tl * q4s::GU_STRIDE;
#pragma unroll
            for (int i = 0; i < 64; i += 4)
                *reinterpret_cast<float4 *>(gu + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
        }
        const bool vec = (O & 3) == 0 && o0 + c0 + 64 <= O;
        auto store_row = [&](float *row) {
            if (vec) {
#pragma unroll
                for (int i = 0; i < 64; i += 4)
                    *reinterpret_cast<float4 *>(row + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (o0 + c0 + i < O) row[i] = yv[i];
            }
        };
        if (SWIGLU) {
            // written above
        } else if (p.part == nullptr || gridDim.z == 1) {
            if (ok && tok_ok) store_row(p.y + (size_t)t * O + o0 + c0);
        } else {
            // split-K: publish this split's partial sums; the last CTA of the
            // tile to arrive adds all splits in z order (deterministic)
            if (ok && tok_ok) store_row(p.part + ((size_t)blockIdx.z * T + t) * O + o0 + c0);
            __threadfence();
            named_bar_sync(1, NUM_EPI_WARPS * 32);
            uint32_t *last_flag = reinterpret_cast<uint32_t *>(smem + oMisc + 8);
            if (warp == EPI_WARP0 && lane == 0) {
                int *c = p.cnt + blockIdx.y * gridDim.x + blockIdx.x;
                const int prev = atomicAdd(c, 1);
                const bool last = prev == (int)gridDim.z - 1;
                if (last) *c = 0;   // ready for the next launch on this stream
                *last_flag = last ? 1u : 0u;
            }
            named_bar_sync(1, NUM_EPI_WARPS * 32);
            if (*last_flag && ok && tok_ok) {
                __threadfence();
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    float4 a4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    for (int z = 0; z < (int)gridDim.z; ++z) {
                        float4 v;
                        if (z == (int)blockIdx.z) {
                            v = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
                        } else {
                            const float *prow = p.part + ((size_t)z * T + t) * O + o0 + c0 + i;
                            if (vec) {
                                v = __ldcg(reinterpret_cast<const float4 *>(prow));
                            } else {
                                v.x = o0 + c0 + i < O ? __ldcg(prow) : 0.0f;
                                v.y = o0 + c0 + i + 1 < O ? __ldcg(prow + 1) : 0.0f;
                                v.z = o0 + c0 + i + 2 < O ? __ldcg(prow + 2) : 0.0f;
                                v.w = o0 + c0 + i + 3 < O ? __ldcg(prow + 3) : 0.0f;
                            }
                        }
                        a4.x += v.x;
                        a4.y += v.y;
                        a4.z += v.z;
                        a4.w += v.w;
                    }
                    yv[i] = a4.x;
                    yv[i + 1] = a4.y;
                    yv[i + 2] = a4.z;
                    yv[i + 3] = a4.w;
                }
                store_row(p.y + (size_t)t * O + o0 + c0);
            }
        }
    } else if (warp == 0 || warp == SCALE_WARP_B) {
        // ------------------------------------------------------- scale warps --
        // Per super-block, for weight rows r and r + 64: the multiplier d (1
        // where d == 0) and the min-term operand row (-(dmin*m_j)/d, split
        // hi/lo); for tokens r and r + 64: the min-term operand row
        // (dx_j*ssum_j split hi/lo).  Slot sb % SSTG is rewritten once
        // super-block sb - SSTG's accumulators have been released: its
        // min-term MMAs completed before they were handed to the epilogue,
        // and the epilogue releases them after reading d.  The weight headers
        // come from the raw tile, the q8_1 scale words are fetched one
        // super-block ahead.
        const int sr = (warp == 0 ? 0 : 32) + lane;   // 0..63
        uint4 dsn[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = t0 + sr + 64 * h;
            dsn[h][0] = dsn[h][1] = make_uint4(0u, 0u, 0u, 0u);
            if (t < T) {
                const uint4 *dp = reinterpret_cast<const uint4 *>(p.ds + (size_t)t * (K / 32) + sb_base * 8);
                dsn[h][0] = __ldg(dp);
                dsn[h][1] = __ldg(dp + 1);
            }
        }
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int ss = sb % SSTG, rs = sb % RSTG;
            ok = mbar_wait(r_full(rs), (sb / RSTG) & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            uint4 hdn[2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
                hdn[h] = *reinterpret_cast<const uint4 *>(smem + oRaw + rs * RAW_BYTES + (sr + 64 * h) * RAW_ROW);
            fence_proxy_async_smem();   // these reads before the next TMA write into the slot
            mbar_arrive(r_empty(rs));
            if (sb >= SSTG) {
                const int prev = sb - SSTG;
                ok = mbar_wait(acc_empty(prev % NACC), (prev / NACC) & 1, abort_flag, kKid, SITE_U_SDS);
                if (!ok) break;
            }
            uint8_t *slot = smem + oSds + ss * SDS_BYTES;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = sr + 64 * h;
                const uint4 hd = hdn[h];
                const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                const float mult = d != 0.0f ? d : 1.0f;
                const float rmult = __frcp_rn(mult);
                reinterpret_cast<float *>(slot + SDS_D)[r] = mult;
                float bh[8], bl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    int sc, mm;
                    q4::q4K_scale_min(hd.y, hd.z, hd.w, j, sc, mm);
                    const float v = -(dmin * (float)mm) * rmult;   // dmin*m exact: 11 x 6 bits
                    bh[j] = to_tf32(v);
                    bl[j] = to_tf32(v - bh[j]);
                }
                q4::put_min_row(slot + MIN_OP_BYTES, r, bh, bl);
                const uint32_t w[8] = {dsn[h][0].x, dsn[h][0].y, dsn[h][0].z, dsn[h][0].w,
                                       dsn[h][1].x, dsn[h][1].y, dsn[h][1].z, dsn[h][1].w};
                float ah[8], al[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float dx = __half2float(__ushort_as_half((unsigned short)(w[j] & 0xFFFFu)));
                    const float v = dx * (float)(int)(int16_t)(w[j] >> 16);   // exact: 11-bit x 12-bit
                    ah[j] = to_tf32(v);
                    al[j] = to_tf32(v - ah[j]);
                }
                q4::put_min_row(slot, r, ah, al);
                const int t = t0 + r;
                if (sb + 1 < nsb && t < T) {
                    const uint4 *dp = reinterpret_cast<const uint4 *>(p.ds + (size_t)t * (K / 32) + (sb_base + sb + 1) * 8);
                    dsn[h][0] = __ldg(dp);
                    dsn[h][1] = __ldg(dp + 1);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(s_full(ss));
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (SWIGLU) {
        // ------------------------------------- SwiGLU + q8_1, all threads --
        // Thread i takes half hh = i % 2 (16 features) of q8_1 block
        // blk = (i / 2) % 2 of token tl = i / 4: h = silu(g)*u for its 16
        // features, then the block's amax and sum through the lane pair, and
        // the block quantised exactly as mmq_quantize_q8_1 quantises.
        const int i = threadIdx.x;
        const int hh = i & 1, blk = (i >> 1) & 1, tl = i >> 2;
        const int t = t0 + tl;
        const int j0 = 32 * blk + 16 * hh;   // first feature of this thread within the tile
        const float *gp = reinterpret_cast<const float *>(smem + oStage) + tl * q4s::GU_STRIDE + j0;
        const float *up = gp + BM * q4s::GU_STRIDE;
        float h[16];
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
            const float4 g4 = *reinterpret_cast<const float4 *>(gp + c);
            const float4 u4 = *reinterpret_cast<const float4 *>(up + c);
            h[c] = q4s::swiglu_f32(g4.x, u4.x);
            h[c + 1] = q4s::swiglu_f32(g4.y, u4.y);
            h[c + 2] = q4s::swiglu_f32(g4.z, u4.z);
            h[c + 3] = q4s::swiglu_f32(g4.w, u4.w);
        }
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fabsf(h[c]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const float d32 = amax != 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
        const float rd = amax != 0.0f ? __frcp_rn(d32) : 0.0f;
        const __half dh = __float2half_rn(d32);
        const float df = __half2float(dh);
        uint32_t hw[8], lw[8], qw[4];
        int ssum = 0;
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
            int qa = 0, qb = 0;
            if (amax != 0.0f) {
                qa = min(127, max(-127, q4s::q8_round_quotient(h[c], d32, rd)));
                qb = min(127, max(-127, q4s::q8_round_quotient(h[c + 1], d32, rd)));
            }
            ssum += qa + qb;
            const uint32_t pair = (uint32_t)(uint8_t)qa | ((uint32_t)(uint8_t)qb << 8);
            if ((c & 2) == 0)
                qw[c >> 2] = pair;
            else
                qw[c >> 2] |= pair << 16;
            // v = f32(d16)*q exact in f32; hi = f16(v), lo = f16(v - hi), both exact
            const float2 v = make_float2(df * (float)qa, df * (float)qb);
            const __half2 hv = __float22half2_rn(v);
            const float2 bv = __half22float2(hv);
            const __half2 lv = __float22half2_rn(make_float2(v.x - bv.x, v.y - bv.y));
            hw[c >> 1] = q4::h2bits(hv);
            lw[c >> 1] = q4::h2bits(lv);
        }
        ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
        if (t < T && *abort_flag == 0u) {
            const int F = O >> 1;
            const int f0 = blockIdx.x * 64 + j0;
            uint4 *ph = reinterpret_cast<uint4 *>(p.h_xa + (size_t)t * F + f0);
            uint4 *pl = reinterpret_cast<uint4 *>(p.h_xa + (size_t)T * F + (size_t)t * F + f0);
            ph[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            ph[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            pl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            pl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
            if (hh == 0)
                p.h_ds[(size_t)t * (F / 32) + f0 / 32] =
                    (uint32_t)__half_as_ushort(dh) | ((uint32_t)(uint16_t)(int16_t)ssum << 16);
            if (p.h_qs != nullptr)
                *reinterpret_cast<uint4 *>(p.h_qs + (size_t)t * F + f0) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Production q4_K launch: activations as the [2T][K] f16 hi/lo planes.
// ksplit <= 1 or part == nullptr: one CTA per output tile covers all of K.
// With swiglu outputs (h_xa != nullptr): y unused, O = 2F gate/up rows interleaved by 64, no split.
// fmt: kQ4K or kQ5K (plain y output only for kQ5K).
int launch_q4K_sb(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K, int ksplit,
                  float *part, int *cnt, mmq_stream_t stream, uint16_t *h_xa = nullptr, uint32_t *h_ds = nullptr,
                  int8_t *h_qs = nullptr, int fmt = kQ4K)
{
    if (fmt == kQ5K && (h_xa || ksplit > 1)) return MMQ_ERR_SHAPE;
    const int row_bytes = fmt == kQ5K ? 176 : 144;
    if (T < 0 || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    if (h_xa && (O % 128 != 0 || ksplit > 1)) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !xa || !ds || (!y && !h_xa) || (h_xa && !h_ds)) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xa) || !aligned16(ds) || (y && !aligned16(y)) || (h_xa && !aligned16(h_xa)) ||
        (h_ds && ((uintptr_t)h_ds & 3u)) || (h_qs && !aligned16(h_qs)))
        return MMQ_ERR_ALIGN;
    const int nsb = K / 256;
    int sbps = nsb, splits = 1;
    if (part != nullptr && ksplit > 1) {
        if (!cnt) return MMQ_ERR_NULL;
        if (!aligned16(part) || ((uintptr_t)cnt & 3u)) return MMQ_ERR_ALIGN;
        sbps = (nsb + min(ksplit, nsb) - 1) / min(ksplit, nsb);
        splits = (nsb + sbps - 1) / sbps;
    }
    int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    CUtensorMap tmA, tmW;
    rc = make_tmap_2d(&tmA, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, 2ull * (uint64_t)T, (uint64_t)K * 2, BK,
                      BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MMQ_OK) return rc;
    rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)nsb * row_bytes, (uint64_t)O,
                      (uint64_t)nsb * row_bytes, row_bytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    static bool attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q4K_sb_kernel<kQ4K, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)q4s::SbLayout<kQ4K>::kDynSmem) != cudaSuccess ||
            cudaFuncSetAttribute(mmq_q4K_sb_kernel<kQ4K, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)q4s::SbLayout<kQ4K>::kDynSmem) != cudaSuccess ||
            cudaFuncSetAttribute(mmq_q4K_sb_kernel<kQ5K, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)q4s::SbLayout<kQ5K>::kDynSmem) != cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    Params prm{};
    prm.w = static_cast<const uint8_t *>(w);
    prm.ds = ds;
    prm.y = y;
    prm.sub = nullptr;
    prm.T = T;
    prm.O = O;
    prm.K = K;
    prm.sb_per_split = sbps;
    prm.part = splits > 1 ? part : nullptr;
    prm.cnt = splits > 1 ? cnt : nullptr;
    prm.h_xa = h_xa;
    prm.h_ds = h_ds;
    prm.h_qs = h_qs;
    const dim3 grid((unsigned)((O + BN - 1) / BN), (unsigned)((T + BM - 1) / BM), (unsigned)splits);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (fmt == kQ5K)
        mmq_q4K_sb_kernel<kQ5K, false><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ5K>::kDynSmem, cs>>>(tmA, tmW, prm);
    else if (h_xa)
        mmq_q4K_sb_kernel<kQ4K, true><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ4K>::kDynSmem, cs>>>(tmA, tmW, prm);
    else
        mmq_q4K_sb_kernel<kQ4K, false><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ4K>::kDynSmem, cs>>>(tmA, tmW, prm);
    return launch_status();
}

// =========================================================================
// q6_K GEMM with super-block accumulation (production).
//
// As the production q4_K kernel, the tensor core accumulates a whole 256-k
// super-block: D_sb[t][o] = sum_k v[t][k] * sc_u(o)*(q-32)[o][k] with v the
// exact hi/lo f16 planes of the dequantised activations, and the epilogue
// adds d*D_sb once per super-block.  The weight values sc*(q-32) reach
// +-4096 and above 2048 f16 holds only even integers, so the weight operand
// is split into two exact f16 planes too: hi = f16(sc*(q-32)) and
// lo = sc*(q-32) - hi in {-1, 0, 1}.  Per 16-k step the tensor core runs
// A_hi*B_hi + A_lo*B_hi + A_hi*B_lo; the dropped A_lo*B_lo is below 2^-22
// of the product.  q6_K has no min term.
// Stages are 32-k wide (one 16-weight sub-block pair; 64-byte swizzled
// rows) with four tiles each: A hi, A lo, B hi, B lo.
// Raw blocks (210 bytes, 2-byte aligned in memory) arrive by one bulk copy
// per row of the 16-byte-aligned 224-byte window around them; the unpack
// threads realign them in registers.
// TMEM: [0,256) even-stage accumulators, [256,512) odd-stage accumulators.
// Warps: 0 raw-weight producer, 15 activation TMA producer, 1 and 14 MMA
// issuers (even / odd stages), 2-5 unpack (thread = weight row), 6-13
// epilogue.
// =========================================================================
namespace q6s {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int MMA_WARP_ODD = 14;
constexpr int ATMA_WARP = 15;
constexpr int KS = 32;                            // k per stage
constexpr int SPS = 256 / KS;                     // stages per super-block
constexpr int STG = 4;                            // operand ring
constexpr int RSTG = 2;                           // raw super-block ring
constexpr int NACC = 2;                           // rotating accumulators per issuer
constexpr int RAW_ROW = 224;                      // 16-byte-aligned window holding one 210-byte block
constexpr uint32_t TM_EVEN = 0, TM_ODD = NACC * BN;
static_assert(TM_ODD + NACC * BN <= 512, "TMEM budget");
constexpr uint32_t TILE = 128 * KS * 2;           // one 128 x 32 f16 operand tile
constexpr uint32_t A_STAGE = 2 * TILE;            // activation hi and lo planes
constexpr uint32_t STAGE_BYTES = 4 * TILE;        // A hi, A lo, B hi, B lo
constexpr uint32_t RAW_BYTES = BN * RAW_ROW;
constexpr uint32_t oStage = 0;
constexpr uint32_t oRaw = oStage + STG * STAGE_BYTES;
constexpr uint32_t oMult = oRaw + RSTG * RAW_BYTES;   // d per weight row, [NACC][BN] f32
constexpr uint32_t oBar = oMult + NACC * BN * 4;
// full, empty [STG]; acc_full, acc_empty, m_full [NACC]; r_full, r_empty [RSTG];
// done [2]; mma_done
constexpr int kNumBars = 2 * STG + 3 * NACC + 2 * RSTG + 2 + 1;
constexpr uint32_t oMisc = oBar + kNumBars * 8;
constexpr uint32_t kDynSmem = oMisc + 16 + 1024;
static_assert(kDynSmem <= 232448, "shared memory budget");
static_assert(TILE % 512 == 0 && STAGE_BYTES % 1024 == 0 && oRaw % 1024 == 0 && RAW_BYTES % 16 == 0,
              "64-byte swizzle atoms are 512 bytes; bulk copies need 16-byte alignment");

// NW consecutive 32-bit words of a raw row starting at the (2-byte aligned)
// byte offset `off`; `row` is 16-byte aligned.  Reads the 16-byte chunks from
// off & ~15 up to the one holding byte (off & ~3) + 4*NW (the funnel shift's
// extra word), which must lie in shared memory.
template <int NW>
__device__ __forceinline__ void row_words(const uint8_t *row, int off, uint32_t (&w)[NW])
{
    constexpr int NC = (NW + 7) / 4;
    uint32_t c[NC * 4];
    const uint4 *src = reinterpret_cast<const uint4 *>(row + (off & ~15));
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const uint4 v = src[i];
        c[4 * i] = v.x;
        c[4 * i + 1] = v.y;
        c[4 * i + 2] = v.z;
        c[4 * i + 3] = v.w;
    }
    const uint32_t sh = (uint32_t)(off & 3) * 8u;
    switch ((off >> 2) & 3) {
    case 0:
#pragma unroll
        for (int j = 0; j < NW; ++j) w[j] = __funnelshift_r(c[j], c[j + 1], sh);
        break;
    case 1:
#pragma unroll
        for (int j = 0; j < NW; ++j) w[j] = __funnelshift_r(c[j + 1], c[j + 2], sh);
        break;
    case 2:
#pragma unroll
        for (int j = 0; j < NW; ++j) w[j] = __funnelshift_r(c[j + 2], c[j + 3], sh);
        break;
    default:
#pragma unroll
        for (int j = 0; j < NW; ++j) w[j] = __funnelshift_r(c[j + 3], c[j + 4], sh);
        break;
    }
}

// Four q6_K values (bytes of q = 0..63, packed in a word) -> two f16 pairs of
// sc*(q-32) as exact hi and lo planes.
__device__ __forceinline__ void q6_pairs(uint32_t q4, __half2 sc2, uint32_t &h0, uint32_t &h1, uint32_t &l0,
                                         uint32_t &l1)
{
    const __half2 bias = __half2half2(__ushort_as_half(0x6420));   // 1056 = 1024 + 32
    const uint32_t a = __byte_perm(q4, 0x64646464u, 0x4140u), b = __byte_perm(q4, 0x64646464u, 0x4342u);
    const __half2 qa = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);   // q - 32, exact
    const __half2 qb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    const __half2 ha = __hmul2(qa, sc2), hb = __hmul2(qb, sc2);              // rounded product
    const __half2 la = __hfma2(qa, sc2, __hneg2(ha)), lb = __hfma2(qb, sc2, __hneg2(hb));   // exact remainder
    h0 = q4::h2bits(ha);
    h1 = q4::h2bits(hb);
    l0 = q4::h2bits(la);
    l1 = q4::h2bits(lb);
}

}  // namespace q6s

__global__ void __launch_bounds__(q6s::NTHREADS, 1)
    mmq_q6K_sb_kernel(const __grid_constant__ CUtensorMap tmA, const Params p)
{
    using namespace q6s;
    constexpr int kKid = 10;
    constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int T = p.T, K = p.K, O = p.O;
    const int nsb = K / 256, nks = nsb * SPS;

    const uint32_t bar0 = sbase + oBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STG + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (2 * STG + s); };
    auto acc_empty = [&](int s) { return bar0 + 8u * (2 * STG + NACC + s); };
    auto m_full = [&](int s) { return bar0 + 8u * (2 * STG + 2 * NACC + s); };
    auto r_full = [&](int s) { return bar0 + 8u * (2 * STG + 3 * NACC + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (2 * STG + 3 * NACC + RSTG + s); };
    auto done = [&](int s) { return bar0 + 8u * (2 * STG + 3 * NACC + 2 * RSTG + s); };
    const uint32_t mma_done = bar0 + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + oMisc + 4);
    auto stage_a = [&](int s) { return sbase + oStage + (uint32_t)s * STAGE_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STG; ++s) {
            mbar_init(full(s), 1 + 128);                    // activation producer (with its bytes) + unpack
            mbar_init(empty(s), 1);                         // the commit of the stage's issuer
        }
        for (int s = 0; s < NACC; ++s) {
            mbar_init(acc_full(s), 2);                      // both issuers' commits
            mbar_init(acc_empty(s), NUM_EPI_WARPS);         // after the epilogue has also read d
            mbar_init(m_full(s), 128);                      // unpack threads' d
        }
        for (int s = 0; s < RSTG; ++s) {
            mbar_init(r_full(s), 32);                       // raw producer lanes (with their bytes)
            mbar_init(r_empty(s), 128);                     // unpack threads
        }
        mbar_init(done(0), 1);
        mbar_init(done(1), 1);
        mbar_init(mma_done, 2);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // --------------------------------------------------- raw producer --
        // One bulk copy per row of the 224-byte window around its block;
        // past the buffer's last full 16-byte granule the bytes are copied
        // one by one.
        const int nrows = min(BN, O - o0);
        const long long nbytes = (long long)O * nsb * 210;
        bool ok = true;
        int n_r = 0;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RSTG;
            ok = mbar_wait(r_empty(rs), ((sb / RSTG) & 1) ^ 1, abort_flag, kKid, SITE_P_RAW);
            if (!ok) break;
            const uint32_t dst = sbase + oRaw + rs * RAW_BYTES;
            uint32_t mine = 0;
            for (int r = lane; r < nrows; r += 32) {
                const long long start = ((long long)(o0 + r) * nsb + sb) * 210;
                const long long a = start & ~15ll;
                uint32_t sz = RAW_ROW;
                if (a + RAW_ROW > nbytes) {
                    sz = (uint32_t)((nbytes - a) & ~15ll);
                    uint8_t *drow = smem + oRaw + rs * RAW_BYTES + r * RAW_ROW;
                    for (long long i = a + sz; i < start + 210; ++i) drow[i - a] = p.w[i];
                }
                mine += sz;
            }
            mbar_arrive_expect_tx(r_full(rs), mine);
            for (int r = lane; r < nrows; r += 32) {
                const long long start = ((long long)(o0 + r) * nsb + sb) * 210;
                const long long a = start & ~15ll;
                uint32_t sz = RAW_ROW;
                if (a + RAW_ROW > nbytes) sz = (uint32_t)((nbytes - a) & ~15ll);
                if (sz) bulk_load(dst + r * RAW_ROW, p.w + a, sz, r_full(rs));
            }
            ++n_r;
        }
        if (!ok)
            for (int i = max(0, n_r - RSTG); i < n_r; ++i) wait_drain(r_full(i % RSTG), (i / RSTG) & 1);
    } else if (warp == ATMA_WARP) {
        // ---------------------------------------------- activation producer --
        if (lane == 0) {
            tma_prefetch(&tmA);
            int n_a = 0;
            bool ok = true;
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % STG;
                ok = mbar_wait(empty(s), ((ks / STG) & 1) ^ 1, abort_flag, kKid, SITE_P_STAGE);
                if (!ok) break;
                // the activation tensor is [2T][K]: hi plane rows 0..T-1, lo plane rows T..2T-1
                mbar_arrive_expect_tx(full(s), A_STAGE);
                tma_load_2d(stage_a(s), &tmA, full(s), ks * KS, t0);
                tma_load_2d(stage_a(s) + TILE, &tmA, full(s), ks * KS, T + t0);
                ++n_a;
            }
            if (!ok)
                for (int i = max(0, n_a - STG); i < n_a; ++i) wait_drain(full(i % STG), (i / STG) & 1);
        }
        __syncwarp();
    } else if (warp == 1 || warp == MMA_WARP_ODD) {
        // ----------------------------------------------------- MMA issuers --
        if (lane == 0) {
            const int me = warp == 1 ? 0 : 1;   // stages with ks % 2 == me
            bool ok = true;
            for (int ks = me; ks < nks && ok; ks += 2) {
                const int s = ks % STG;
                const int sb = ks / SPS, jb = ks % SPS, slot = sb % NACC;
                const int n_mine = ks >> 1;
                ok = (n_mine == 0 || mbar_wait(done(me), (n_mine - 1) & 1, abort_flag, kKid, SITE_M_A)) &&
                     mbar_wait(full(s), (ks / STG) & 1, abort_flag, kKid, SITE_M_A) &&
                     (jb > 1 || mbar_wait(acc_empty(slot), ((sb / NACC) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC));
                if (!ok) break;
                tc_fence_after();
                const uint32_t a_hi = stage_a(s);
                const uint64_t dah = sdesc_k_sw64(a_hi), dal = sdesc_k_sw64(a_hi + TILE);
                const uint64_t dbh = sdesc_k_sw64(a_hi + A_STAGE), dbl = sdesc_k_sw64(a_hi + A_STAGE + TILE);
                const uint32_t d_acc = tmem_base + (me ? TM_ODD : TM_EVEN) + slot * BN;
#pragma unroll
                for (int kk = 0; kk < KS / 16; ++kk) {
                    // +32 bytes along K inside the swizzled rows = +2 in the address field
                    umma_f16(d_acc, dah + 2 * kk, dbh + 2 * kk, kIdesc, (jb <= 1 && kk == 0) ? 0u : 1u);
                    umma_f16(d_acc, dal + 2 * kk, dbh + 2 * kk, kIdesc, 1u);
                    umma_f16(d_acc, dah + 2 * kk, dbl + 2 * kk, kIdesc, 1u);
                }
                if (jb >= SPS - 2) umma_commit(acc_full(slot));   // this issuer's last stage of the super-block
                umma_commit(empty(s));
                umma_commit(done(me));
            }
            umma_commit(mma_done);
            if (!wait_drain(mma_done, 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp >= UNPACK_WARP0 && warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        // Thread = one weight row.  Per half super-block it realigns the
        // row's 64 ql and 32 qh bytes into registers; per 32-k stage it writes
        // the row's 32 values sc*(q-32) as exact hi and lo f16 planes.
        const int r = threadIdx.x - UNPACK_WARP0 * 32;
        const int o = o0 + r;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int rs = sb % RSTG, slot = sb % NACC;
            ok = mbar_wait(r_full(rs), (sb / RSTG) & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            const uint8_t *row = smem + oRaw + rs * RAW_BYTES + r * RAW_ROW;
            // rows past O were not copied: their (stale) bytes feed weight rows that are never stored
            const int lead = (int)((((long long)min(o, O - 1) * nsb + sb) * 210) & 15);
            uint32_t scw[4];
            row_words<4>(row, lead + 192, scw);
            const uint16_t d16 = *reinterpret_cast<const uint16_t *>(row + lead + 208);
            // d of this super-block for the epilogue
            if (sb >= NACC) {
                const int prev = sb - NACC;
                ok = mbar_wait(acc_empty(prev % NACC), (prev / NACC) & 1, abort_flag, kKid, SITE_U_SDS);
                if (!ok) break;
            }
            reinterpret_cast<float *>(smem + oMult + slot * BN * 4)[r] =
                o < O ? __half2float(__ushort_as_half(d16)) : 0.0f;
            mbar_arrive(m_full(slot));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t ql[16], qh[8];
                row_words<16>(row, lead + 64 * h, ql);
                row_words<8>(row, lead + 128 + 32 * h, qh);
                if (h == 1) {
                    fence_proxy_async_smem();   // these reads before the next bulk copy into the slot
                    mbar_arrive(r_empty(rs));
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int jb = 4 * h + g, ks = sb * SPS + jb, s = ks % STG;
                    // sub-blocks 2jb and 2jb+1: scale bytes 2jb, 2jb+1
                    const uint32_t sw = scw[jb >> 1];
                    const int sc0 = (int)(int8_t)((sw >> (16 * (jb & 1))) & 0xFFu);
                    const int sc1 = (int)(int8_t)((sw >> (16 * (jb & 1) + 8)) & 0xFFu);
                    const __half2 s0 = __float2half2_rn((float)sc0), s1 = __float2half2_rn((float)sc1);
                    // values i = 0..31 of group g: ql byte 32*(g&1)+i (low or high nibble),
                    // qh byte i bits 2g..2g+1
                    uint4 vh[4], vl[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t hh[4], ll[4];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t lw = ql[8 * (g & 1) + 2 * c + e], hw = qh[2 * c + e];
                            const uint32_t lo4 = (g < 2 ? lw : (lw >> 4)) & 0x0F0F0F0Fu;
                            const uint32_t hi2 = ((hw >> (2 * g)) & 0x03030303u) << 4;
                            q6_pairs(lo4 | hi2, c < 2 ? s0 : s1, hh[2 * e], hh[2 * e + 1], ll[2 * e], ll[2 * e + 1]);
                        }
                        vh[c] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        vl[c] = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
                    ok = mbar_wait(empty(s), ((ks / STG) & 1) ^ 1, abort_flag, kKid, SITE_U_STAGE);
                    if (!ok) break;
                    // 64-byte swizzle: 16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3)
                    uint8_t *bh = smem + oStage + s * STAGE_BYTES + A_STAGE + (r >> 3) * 512 + (r & 7) * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int cc = (c ^ ((r >> 1) & 3)) << 4;
                        *reinterpret_cast<uint4 *>(bh + cc) = vh[c];
                        *reinterpret_cast<uint4 *>(bh + TILE + cc) = vl[c];
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(full(s));
                }
                if (!ok) break;
            }
        }
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NUM_EPI_WARPS) {
        // --------------------------------------------------------- epilogue --
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;
        const int c0 = (ew >> 2) * 64;
        const int tl = quarter * 32 + lane;
        const int t = t0 + tl;
        const bool tok_ok = t < T;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float yv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) yv[i] = 0.0f;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int slot = sb % NACC;
            ok = mbar_wait_warp(m_full(slot), (sb / NACC) & 1, abort_flag, kKid, SITE_E_SDS) &&
                 mbar_wait_warp(acc_full(slot), (sb / NACC) & 1, abort_flag, kKid, SITE_E_ACC);
            if (!ok) break;
            tc_fence_after();
            const float *dv = reinterpret_cast<const float *>(smem + oMult + slot * BN * 4) + c0;
            const uint32_t col = tmem_base + lane_off + slot * BN + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t ra[16], rb[16];
                tmem_ld16(col + TM_EVEN + q * 16, ra);
                tmem_ld16(col + TM_ODD + q * 16, rb);
                tmem_ld_wait2(ra, rb);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dv + q * 16 + i);
                    const float2 s0 = __fadd2_rn(make_float2(__uint_as_float(ra[i]), __uint_as_float(ra[i + 1])),
                                                 make_float2(__uint_as_float(rb[i]), __uint_as_float(rb[i + 1])));
                    const float2 s1 = __fadd2_rn(make_float2(__uint_as_float(ra[i + 2]), __uint_as_float(ra[i + 3])),
                                                 make_float2(__uint_as_float(rb[i + 2]), __uint_as_float(rb[i + 3])));
                    const int e = q * 16 + i;
                    const float2 y0 = __ffma2_rn(s0, make_float2(d4.x, d4.y), make_float2(yv[e], yv[e + 1]));
                    const float2 y1 = __ffma2_rn(s1, make_float2(d4.z, d4.w), make_float2(yv[e + 2], yv[e + 3]));
                    yv[e] = y0.x;
                    yv[e + 1] = y0.y;
                    yv[e + 2] = y1.x;
                    yv[e + 3] = y1.y;
                }
            }
            // both accumulators and this super-block's d have been read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(slot));
        }
        if (ok && tok_ok) {
            float *yrow = p.y + (size_t)t * O + o0 + c0;
            if ((O & 3) == 0 && o0 + c0 + 64 <= O) {
#pragma unroll
                for (int i = 0; i < 64; i += 4)
                    *reinterpret_cast<float4 *>(yrow + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (o0 + c0 + i < O) yrow[i] = yv[i];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Production q6_K launch: activations as the [2T][K] f16 hi/lo planes.
int launch_q6K_sb(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                  mmq_stream_t stream)
{
    (void)ds;
    if (T < 0 || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !xa || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xa) || !aligned16(y)) return MMQ_ERR_ALIGN;
    int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    CUtensorMap tmA;
    rc = make_tmap_2d(&tmA, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, 2ull * (uint64_t)T, (uint64_t)K * 2,
                      q6s::KS, BM, CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc != MMQ_OK) return rc;
    static bool attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q6K_sb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)q6s::kDynSmem) != cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    Params prm{};
    prm.w = static_cast<const uint8_t *>(w);
    prm.ds = ds;
    prm.y = y;
    prm.sub = nullptr;
    prm.T = T;
    prm.O = O;
    prm.K = K;
    prm.sb_per_split = K / 256;
    prm.part = nullptr;
    prm.cnt = nullptr;
    const dim3 grid((unsigned)((O + BN - 1) / BN), (unsigned)((T + BM - 1) / BM));
    mmq_q6K_sb_kernel<<<grid, q6s::NTHREADS, q6s::kDynSmem, reinterpret_cast<cudaStream_t>(stream)>>>(tmA, prm);
    return launch_status();
}

// =========================================================================
// Small-T q4_K GEMM (T <= 16): the pages' per-sub-block form on the int8
// warp MMA.
//
// With few tokens the GEMM is bound by streaming the weights from HBM, and
// the cost that matters is how many instructions turn a weight byte into a
// tensor-core operand.  mma.sync m16n8k32 (s8 x s8 -> s32) takes exactly one
// q4_K sub-block (32 k) per instruction, the unsigned nibbles are int8
// operands after one AND per four weights, and the int8 activations qs are
// used as they are.  Every MMA gives the exact integer dots C_b of one
// sub-block for 16 tokens x 8 weight rows; the f32 fold
//     y += dx_b*(d*sc_b)*C_b + (dx_b*ssum_b)*(-(dmin*m_b))
// follows per sub-block ("31 . r28", 2.3).
// CTA = 8 warps on the same 16 weight rows (two MMAs per activation
// fragment); warp w takes the w-th eighth of the super-blocks, and the eight
// partial sums are added in warp order through shared memory
// (deterministic).  Each warp stages the next super-block's activation rows
// and scale words in shared memory with cp.async and loads the weights from
// global memory one super-block ahead.
// =========================================================================
namespace smt {

constexpr int NWARPS = 8;
constexpr int NTHREADS = NWARPS * 32;
constexpr int ROWS = 16;         // weight rows per CTA: two MMA N tiles
constexpr int MAXT = 16;         // tokens: one MMA M tile
constexpr int A_ROW = 256 + 16;  // staged activation row (bytes): 256 k + pad (conflict-free fragment reads)
constexpr int D_ROW = 48;        // staged scale-word row: 8 words + pad
constexpr int BUF = MAXT * A_ROW + MAXT * D_ROW;   // one super-block of one warp
static_assert(BUF % 16 == 0, "cp.async destinations are 16-byte aligned");

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy; with src_bytes = 0 nothing is read and the
// destination is zero-filled
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

}  // namespace smt

__global__ void __launch_bounds__(smt::NTHREADS, 2)
    mmq_q4K_small_kernel(const uint8_t *__restrict__ w, const int8_t *__restrict__ qs, const uint32_t *__restrict__ ds,
                         float *__restrict__ y, int T, int O, int K)
{
    using namespace smt;
    extern __shared__ __align__(16) uint8_t sm[];
    float *part = reinterpret_cast<float *>(sm + NWARPS * 2 * BUF);   // [NWARPS][MAXT][ROWS]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;   // MMA group and thread in group
    const int o0 = blockIdx.x * ROWS;
    const int nsb = K / 256;
    const int per = (nsb + NWARPS - 1) / NWARPS;
    const int sb0 = min(nsb, warp * per), sb1 = min(nsb, sb0 + per);
    uint8_t *wbuf = sm + warp * 2 * BUF;
    const uint32_t wbuf_s = smem_u32(wbuf);

    // B rows of this thread: o0 + g (tile 0) and o0 + 8 + g (tile 1); C columns:
    // rows o0 + 8 n + 2 tig + {0, 1} of tile n
    const uint8_t *wb[2], *wc[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        wb[n] = w + (size_t)min(o0 + 8 * n + g, O - 1) * nsb * 144;
        wc[n][0] = w + (size_t)min(o0 + 8 * n + 2 * tig, O - 1) * nsb * 144;
        wc[n][1] = w + (size_t)min(o0 + 8 * n + 2 * tig + 1, O - 1) * nsb * 144;
    }
    // stage super-block sb's activations (16 rows x 256 B) and scale words (16 x 32 B) into buffer b
    auto stage = [&](int sb, int b) {
        const uint32_t base = wbuf_s + b * BUF;
// token rows >= T are zero-filled (their outputs are never stored)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i, row = c >> 4, ch = c & 15;
            const int t = min(row, T - 1);
            cp_async16(base + row * A_ROW + ch * 16, qs + (size_t)t * K + sb * 256 + ch * 16, row < T ? 16u : 0u);
        }
        {
            const int row = lane >> 1, ch = lane & 1;
            const int t = min(row, T - 1);
            cp_async16(base + MAXT * A_ROW + row * D_ROW + ch * 16, ds + (size_t)t * (K / 32) + sb * 8 + ch * 4,
                       row < T ? 16u : 0u);
        }
        cp_async_commit();
    };
    uint4 nq[2][2], nh[2][2];
    auto load_w = [&](int sb) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const uint8_t *b = wb[n] + (size_t)sb * 144 + 16;
            nq[n][0] = make_uint4(__ldg(reinterpret_cast<const uint32_t *>(b + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 16 + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 32 + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 48 + 4 * tig)));
            nq[n][1] = make_uint4(__ldg(reinterpret_cast<const uint32_t *>(b + 64 + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 80 + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 96 + 4 * tig)),
                                  __ldg(reinterpret_cast<const uint32_t *>(b + 112 + 4 * tig)));
            nh[n][0] = __ldg(reinterpret_cast<const uint4 *>(wc[n][0] + (size_t)sb * 144));
            nh[n][1] = __ldg(reinterpret_cast<const uint4 *>(wc[n][1] + (size_t)sb * 144));
        }
    };
    float acc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.0f;
    if (sb0 < sb1) {
        stage(sb0, 0);
        load_w(sb0);
    }
    for (int sb = sb0; sb < sb1; ++sb) {
        const int b = (sb - sb0) & 1;
        uint4 q[2][2], h[2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                q[n][e] = nq[n][e];
                h[n][e] = nh[n][e];
            }
        if (sb + 1 < sb1) {
            stage(sb + 1, b ^ 1);
            load_w(sb + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        const uint8_t *abuf = wbuf + b * BUF;
        const uint32_t *dbuf = reinterpret_cast<const uint32_t *>(abuf + MAXT * A_ROW);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t a[4];
            a[0] = *reinterpret_cast<const uint32_t *>(abuf + g * A_ROW + 32 * j + 4 * tig);
            a[1] = *reinterpret_cast<const uint32_t *>(abuf + (g + 8) * A_ROW + 32 * j + 4 * tig);
            a[2] = *reinterpret_cast<const uint32_t *>(abuf + g * A_ROW + 32 * j + 16 + 4 * tig);
            a[3] = *reinterpret_cast<const uint32_t *>(abuf + (g + 8) * A_ROW + 32 * j + 16 + 4 * tig);
            const uint32_t da = dbuf[g * (D_ROW / 4) + j], db = dbuf[(g + 8) * (D_ROW / 4) + j];
            const float dxa = __half2float(__ushort_as_half((unsigned short)(da & 0xFFFFu)));
            const float dxb = __half2float(__ushort_as_half((unsigned short)(db & 0xFFFFu)));
            const float sma = dxa * (float)(int)(int16_t)(da >> 16), smb = dxb * (float)(int)(int16_t)(db >> 16);
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                // sub-block j: low (j even) or high (j odd) nibbles of bytes 32 (j/2) ..
                const uint32_t wl = (j & 2) ? (j & 4 ? q[n][1].z : q[n][0].z) : (j & 4 ? q[n][1].x : q[n][0].x);
                const uint32_t wh = (j & 2) ? (j & 4 ? q[n][1].w : q[n][0].w) : (j & 4 ? q[n][1].y : q[n][0].y);
                const uint32_t b0 = ((j & 1) ? (wl >> 4) : wl) & 0x0F0F0F0Fu;
                const uint32_t b1 = ((j & 1) ? (wh >> 4) : wh) & 0x0F0F0F0Fu;
                int c[4] = {0, 0, 0, 0};
                mma_s8(c, a, b0, b1);
                int sc0, m0, sc1, m1;
                q4::q4K_scale_min(h[n][0].y, h[n][0].z, h[n][0].w, j, sc0, m0);
                q4::q4K_scale_min(h[n][1].y, h[n][1].z, h[n][1].w, j, sc1, m1);
                const float d0 = __half2float(__ushort_as_half((unsigned short)(h[n][0].x & 0xFFFFu)));
                const float d1 = __half2float(__ushort_as_half((unsigned short)(h[n][1].x & 0xFFFFu)));
                const float dm0 = __half2float(__ushort_as_half((unsigned short)(h[n][0].x >> 16)));
                const float dm1 = __half2float(__ushort_as_half((unsigned short)(h[n][1].x >> 16)));
                const float dsv0 = d0 * (float)sc0, dsv1 = d1 * (float)sc1;
                const float dmv0 = -(dm0 * (float)m0), dmv1 = -(dm1 * (float)m1);
                // c0, c1: token g, rows 2 tig, 2 tig + 1 of tile n; c2, c3: token g + 8
                acc[n][0] += (dxa * dsv0) * (float)c[0] + sma * dmv0;
                acc[n][1] += (dxa * dsv1) * (float)c[1] + sma * dmv1;
                acc[n][2] += (dxb * dsv0) * (float)c[2] + smb * dmv0;
                acc[n][3] += (dxb * dsv1) * (float)c[3] + smb * dmv1;
            }
        }
        __syncwarp();   // the buffer is restaged two super-blocks later
    }
    // partial sums of this warp's super-blocks -> shared memory; warp order fixed
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        part[(warp * MAXT + g) * ROWS + 8 * n + 2 * tig] = acc[n][0];
        part[(warp * MAXT + g) * ROWS + 8 * n + 2 * tig + 1] = acc[n][1];
        part[(warp * MAXT + g + 8) * ROWS + 8 * n + 2 * tig] = acc[n][2];
        part[(warp * MAXT + g + 8) * ROWS + 8 * n + 2 * tig + 1] = acc[n][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < MAXT * ROWS; i += NTHREADS) {
        const int t = i / ROWS, n = i % ROWS;
        if (t < T && o0 + n < O) {
            float s = 0.0f;
#pragma unroll
            for (int v = 0; v < NWARPS; ++v) s += part[(v * MAXT + t) * ROWS + n];
            y[(size_t)t * O + o0 + n] = s;
        }
    }
}

int launch_q4K_small(const void *w, const int8_t *qs, const uint32_t *ds, float *y, int T, int O, int K,
                     mmq_stream_t stream)
{
    if (T < 0 || T > smt::MAXT || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !qs || !ds || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(qs) || !aligned16(ds) || !aligned16(y)) return MMQ_ERR_ALIGN;
    int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    constexpr int kSmem = smt::NWARPS * 2 * smt::BUF + smt::NWARPS * smt::MAXT * smt::ROWS * 4;
    static bool attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q4K_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
            cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    const dim3 grid((unsigned)((O + smt::ROWS - 1) / smt::ROWS));
    mmq_q4K_small_kernel<<<grid, smt::NTHREADS, kSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(w), qs, ds, y, T, O, K);
    return launch_status();
}

// =========================================================================
// q4_K GEMM for few tokens (T <= 64): weight-stationary tcgen05 form.
//
// With few tokens the GEMM streams the weights once and does little else, so
// the weight rows take the 128-lane M side of the MMA and reach it from
// tensor memory rather than shared memory: each unpack thread owns one weight
// row, turns a super-block's 256 quants into the exact f16 products sc*q
// (sc*q <= 945; zeros where d == 0) and writes them with tcgen05.st into the
// A operand's TMEM columns (row = lane, column c = k pair 2c, 2c+1).  The
// tokens are the B operand: the exact hi and lo f16 planes of the dequantised
// activations, staged by TMA in the 128-byte swizzle as one tile of 2N rows
// (N hi rows, then N lo rows; N = 16, 32 or 64 >= T, rows past T read as zero
// or as finite values whose outputs are never stored), so that one MMA per
// 16-k step yields D_hi and D_lo side by side.  Per super-block
//     D[o][t] = sum_k sc*q[o][k] * (hi + lo)[t][k]
//             + sum_j (-(dmin*m_j)/mult)[o] * (dx_j*ssum_j)[t]
// (16 f16 MMAs and 3 split-tf32 MMAs for the min term into the hi columns;
// mult = d, or 1 where d == 0), and the epilogue adds mult*(D_hi + D_lo) to
// the running f32 output: the two-term fold of "31 . r28" (2.3) taken per
// super-block, as in the production kernel.
// Work: one cluster of up to 8 CTAs per 128-row tile, the CTAs taking
// consecutive super-block ranges; their partial sums meet in shared memory
// and the cluster's first CTA adds them in rank order through distributed
// shared memory (no global scratch, the same result on every call).
// Warps: 0 TMA producer; 1 and 2 MMA issuers (even / odd units, each into
// accumulators of its own); 3 builds the tokens' min-term operand from the
// q8_1 scale words; 4-7 and 8-11 unpack (even / odd units, thread = weight
// row); 12-15 epilogue (thread = weight row).
// The rings that alternating agents wait on (raw weights, activation
// chunks, TMEM A buffers) have twice as many full / empty barriers as slots:
// unit i uses slot i % S and barriers i % 2S, so every barrier is waited on
// by one agent through consecutive phases (a parity wait cannot tell apart
// phases two apart); the other rings are even-sized and waited on in order.
// =========================================================================
struct WtParams {
    const uint8_t *w;   // [O][nsb] q4_K blocks
    float *y;           // [T][O]
    int T, O, K;
    int sb_per_split;   // super-blocks per CTA of a cluster
};

namespace wts {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int WT_HELPER = 3;
constexpr int WT_UNPACK0 = 4;
constexpr int WT_EPI0 = 12;
constexpr int MAX_CLUSTER = 8;
constexpr uint32_t RAW_BYTES = 128 * 144;     // one super-block of 128 weight rows
constexpr uint32_t AMIN_BYTES = 128 * 64;     // 128 rows x (8 hi + 8 lo) tf32, no swizzle

template <int N>
struct Cfg {
    static constexpr int NM = 2 * N;                                // MMA N: hi rows then lo rows
    static constexpr int ABUF = N == 64 ? 2 : 3;                    // TMEM A buffers (128 columns each)
    static constexpr int NACC = N == 16 ? 4 : 2;                    // accumulators (NM columns each)
    static constexpr int CSTG = N == 16 ? 16 : (N == 32 ? 10 : 8);  // activation chunk ring (64 k each)
    static constexpr int DSTG = 4;                                  // scale-word / min-operand ring
    static constexpr int RSTG = N == 64 ? 3 : 4;                    // raw weight ring
    static constexpr int RB = 2 * RSTG, CB = 2 * CSTG, AB = 2 * ABUF;   // barriers of the rings above
    static constexpr uint32_t PLANE = N * 128;                      // 64 k x N rows of one plane
    static constexpr uint32_t CH_BYTES = 2 * PLANE;                 // hi rows then lo rows
    static constexpr uint32_t DS_BYTES = N * 32;                    // [N][8] q8_1 scale words
    static constexpr uint32_t oBMIN = DS_BYTES;                     // [N] rows x (8 hi + 8 lo) tf32
    static constexpr uint32_t D_SLOT = ((DS_BYTES + N * 64 + 127) / 128) * 128;
    static constexpr uint32_t TM_A = 0;
    static constexpr uint32_t TM_ACC = ABUF * 128;
    static constexpr uint32_t oX = 0;
    static constexpr uint32_t oDsr = oX + CSTG * CH_BYTES;
    static constexpr uint32_t oRaw = oDsr + DSTG * D_SLOT;
    static constexpr uint32_t oAmin = oRaw + RSTG * RAW_BYTES;
    static constexpr uint32_t oBar = oAmin + ABUF * AMIN_BYTES;
    // raw_full, raw_empty [RB]; c_full, c_empty [CB]; d_full, d_empty, bmin_full [DSTG];
    // a_full, a_empty [AB]; acc_full, acc_empty [NACC]; done [2]
    static constexpr int kNumBars = 2 * RB + 2 * CB + 3 * DSTG + 2 * AB + 2 * NACC + 2;
    static_assert(DSTG % 2 == 0 && NACC % 2 == 0, "rings with one barrier per slot must be even-sized");
    static constexpr uint32_t oMisc = oBar + kNumBars * 8;
    static constexpr uint32_t kDynSmem = oMisc + 16 + 1024;
    static_assert(TM_ACC + NACC * NM <= 512, "TMEM budget");
    static_assert(kDynSmem <= 232448, "shared memory budget");
    static_assert(CH_BYTES % 1024 == 0, "128-byte swizzled tiles need 1024-byte alignment");
    static_assert(oDsr % 128 == 0 && D_SLOT % 128 == 0 && oRaw % 128 == 0 && oAmin % 16 == 0, "copy alignment");
    static_assert(128u * N * 4u <= CSTG * CH_BYTES, "partial sums fit in the activation ring");
};

}  // namespace wts

template <int N>
__global__ void __launch_bounds__(wts::NTHREADS, 1)
    mmq_q4K_wt_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmD, const WtParams p)
{
    using namespace wts;
    using C = Cfg<N>;
    constexpr int kKid = 11;
    constexpr uint32_t kIdesc = idesc_f16_f32(128, C::NM);
    constexpr uint32_t kIdescTf32 = idesc_tf32_f32(128, N);
    constexpr int RSTG = C::RSTG, CSTG = C::CSTG, DSTG = C::DSTG, ABUF = C::ABUF, NACC = C::NACC;
    constexpr int RB = C::RB, CB = C::CB, AB = C::AB;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, O = p.O, nsb = p.K / 256;
    const int tile = (int)blockIdx.y, ks = (int)gridDim.x;
    const int sb0 = (int)blockIdx.x * p.sb_per_split;
    const int n = max(0, min(nsb, sb0 + p.sb_per_split) - sb0);

    const uint32_t bar0 = sbase + C::oBar;
    auto raw_full = [&](int b) { return bar0 + 8u * b; };
    auto raw_empty = [&](int b) { return bar0 + 8u * (RB + b); };
    auto c_full = [&](int b) { return bar0 + 8u * (2 * RB + b); };
    auto c_empty = [&](int b) { return bar0 + 8u * (2 * RB + CB + b); };
    constexpr int kD = 2 * RB + 2 * CB;
    auto d_full = [&](int s) { return bar0 + 8u * (kD + s); };
    auto d_empty = [&](int s) { return bar0 + 8u * (kD + DSTG + s); };
    auto bmin_full = [&](int s) { return bar0 + 8u * (kD + 2 * DSTG + s); };
    constexpr int kA = kD + 3 * DSTG;
    auto a_full = [&](int b) { return bar0 + 8u * (kA + b); };
    auto a_empty = [&](int b) { return bar0 + 8u * (kA + AB + b); };
    auto acc_full = [&](int a) { return bar0 + 8u * (kA + 2 * AB + a); };
    auto acc_empty = [&](int a) { return bar0 + 8u * (kA + 2 * AB + NACC + a); };
    auto done = [&](int e) { return bar0 + 8u * (C::kNumBars - 2 + e); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + C::oMisc + 4);

    // the producer's copies: raw weights and q8_1 scale words of unit i;
    // activation chunk j (64 k of unit j/4, hi and lo planes)
    auto issue_raw = [&](int i) {
        const int rs = i % RSTG, rb = i % RB;
        mbar_arrive_expect_tx(raw_full(rb), RAW_BYTES);
        tma_load_2d(sbase + C::oRaw + rs * RAW_BYTES, &tmW, raw_full(rb), (sb0 + i) * 144, tile * 128);
    };
    auto issue_ds = [&](int i) {
        const int dsl = i % DSTG;
        mbar_arrive_expect_tx(d_full(dsl), C::DS_BYTES);
        tma_load_2d(sbase + C::oDsr + dsl * C::D_SLOT, &tmD, d_full(dsl), (sb0 + i) * 8, 0);
    };
    auto issue_chunk = [&](int j) {
        // a box of the activation planes viewed as [K/64 chunks][2 planes][T rows][64 k]:
        // lands as [hi rows 0..N-1, lo rows 0..N-1] (rows past T zero)
        const int cs = j % CSTG, cb = j % CB;
        mbar_arrive_expect_tx(c_full(cb), C::CH_BYTES);
        tma_load_4d(sbase + C::oX + cs * C::CH_BYTES, &tmX, c_full(cb), 0, 0, 0, sb0 * 4 + j);
    };

    if (threadIdx.x == 0) {
        tma_prefetch(&tmX);
        tma_prefetch(&tmW);
        tma_prefetch(&tmD);
        for (int b = 0; b < RB; ++b) {
            mbar_init(raw_full(b), 1);
            mbar_init(raw_empty(b), 4);       // the four unpack warps of one group
        }
        for (int b = 0; b < CB; ++b) {
            mbar_init(c_full(b), 1);
            mbar_init(c_empty(b), 1);         // the issuer's commit
        }
        for (int s = 0; s < DSTG; ++s) {
            mbar_init(d_full(s), 1);
            mbar_init(d_empty(s), 1);         // the issuer's commit (after the helper is done)
            mbar_init(bmin_full(s), 1);       // the helper warp
        }
        for (int b = 0; b < AB; ++b) {
            mbar_init(a_full(b), 4);
            mbar_init(a_empty(b), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 4);       // the four epilogue warps
        }
        mbar_init(done(0), 1);
        mbar_init(done(1), 1);
        *abort_flag = 0u;
        fence_mbar_init();
        // the first unit's copies overlap the setup; the producer issues the rest
        if (n > 0) {
            issue_raw(0);
            issue_ds(0);
            for (int j = 0; j < 4; ++j) issue_chunk(j);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer --
        int n_r = min(n, 1), n_d = min(n, 1), n_c = min(4 * n, 4);
        bool ok = true;
        for (int i = 1; i < n && ok; ++i) {
            // a slot is free once the unit RSTG before (the chunk CSTG before) has released it
            ok = i < RSTG ||
                 mbar_wait_warp(raw_empty((i - RSTG) % RB), ((i - RSTG) / RB) & 1, abort_flag, kKid, SITE_P_RAW);
            if (!ok) break;
            if (lane == 0) issue_raw(i);
            ++n_r;
            ok = mbar_wait_warp(d_empty(i % DSTG), ((i / DSTG) & 1) ^ 1, abort_flag, kKid, SITE_P_STAGE);
            if (!ok) break;
            if (lane == 0) issue_ds(i);
            ++n_d;
            for (int j = 4 * i; j < 4 * i + 4 && ok; ++j) {
                ok = j < CSTG ||
                     mbar_wait_warp(c_empty((j - CSTG) % CB), ((j - CSTG) / CB) & 1, abort_flag, kKid, SITE_P_STAGE);
                if (!ok) break;
                if (lane == 0) issue_chunk(j);
                ++n_c;
            }
        }
        if (!ok && lane == 0) {
            // let copies already in flight land before the CTA exits
            for (int i = max(0, n_r - RSTG); i < n_r; ++i) wait_drain(raw_full(i % RB), (i / RB) & 1);
            for (int i = max(0, n_d - DSTG); i < n_d; ++i) wait_drain(d_full(i % DSTG), (i / DSTG) & 1);
            for (int j = max(0, n_c - CSTG); j < n_c; ++j) wait_drain(c_full(j % CB), (j / CB) & 1);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ----------------------------------------------------- MMA issuers --
        if (lane == 0) {
            const int e = warp - 1;
            bool ok = true;
            for (int i = e; i < n && ok; i += 2) {
                const int buf = i % ABUF, ab = i % AB, dsl = i % DSTG, acc = i % NACC;
                // every wait of the unit before its first MMA: a wait of the issuing
                // thread queues behind that thread's MMAs still in flight
                ok = mbar_wait(a_full(ab), (i / AB) & 1, abort_flag, kKid, SITE_M_A) &&
                     mbar_wait(acc_empty(acc), ((i / NACC) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC);
                for (int c = 0; c < 4 && ok; ++c)
                    ok = mbar_wait(c_full((4 * i + c) % CB), ((4 * i + c) / CB) & 1, abort_flag, kKid, SITE_M_B);
                ok = ok && mbar_wait(bmin_full(dsl), (i / DSTG) & 1, abort_flag, kKid, SITE_E_SDS);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_acc = tmem_base + C::TM_ACC + acc * C::NM;
                const uint32_t a_col = tmem_base + C::TM_A + buf * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint64_t bd = sdesc_k_sw128(sbase + C::oX + ((4 * i + c) % CSTG) * C::CH_BYTES);
#pragma unroll
                    for (int s = 0; s < 4; ++s)   // +32 bytes per 16-k step inside the swizzled rows
                        umma_f16_ts(d_acc, a_col + 8 * (4 * c + s), bd + (uint64_t)(2 * s), kIdesc,
                                    (c | s) != 0 ? 1u : 0u);
                }
                // min term into the hi columns: A_min . B_min^T as hi.hi + hi.lo + lo.hi
                const uint64_t am = sdesc_k_none(sbase + C::oAmin + buf * AMIN_BYTES, 128, 512);
                const uint64_t bm = sdesc_k_none(sbase + C::oDsr + dsl * C::D_SLOT + C::oBMIN, 128, 512);
                umma_tf32(d_acc, am, bm, kIdescTf32, 1u);
                umma_tf32(d_acc, am, bm + (256 >> 4), kIdescTf32, 1u);
                umma_tf32(d_acc, am + (256 >> 4), bm, kIdescTf32, 1u);
#pragma unroll
                for (int c = 0; c < 4; ++c) umma_commit(c_empty((4 * i + c) % CB));
                umma_commit(acc_full(acc));
                umma_commit(a_empty(ab));
                umma_commit(d_empty(dsl));
            }
            umma_commit(done(e));
            if (!wait_drain(done(e), 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == WT_HELPER) {
        // ------------------------------------- token min-term operand (B_min) --
        // Row t: (dx_j*ssum_j) for the 8 sub-blocks, split into tf32 hi + lo
        // (an exact f32 product of an 11-bit and a 12-bit integer value).
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
            const int dsl = i % DSTG;
            ok = mbar_wait_warp(d_full(dsl), (i / DSTG) & 1, abort_flag, kKid, SITE_U_SDS);
            if (!ok) break;
            uint8_t *db = smem + C::oDsr + dsl * C::D_SLOT;
#pragma unroll
            for (int t = lane; t < N; t += 32) {
                const uint4 a = *reinterpret_cast<const uint4 *>(db + t * 32);
                const uint4 b = *reinterpret_cast<const uint4 *>(db + t * 32 + 16);
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                float ah[8], al[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float dx = __half2float(__ushort_as_half((unsigned short)(wv[j] & 0xFFFFu)));
                    const float v = dx * (float)(int)(int16_t)(wv[j] >> 16);
                    ah[j] = to_tf32(v);
                    al[j] = to_tf32(v - ah[j]);
                }
                q4::put_min_row(db + C::oBMIN, t, ah, al);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bmin_full(dsl));
        }
    } else if (warp >= WT_UNPACK0 && warp < WT_EPI0) {
        // ------------------------------------------------------ unpack warps --
        const int g = (warp - WT_UNPACK0) >> 2;     // units with i % 2 == g
        const int r = (warp & 3) * 32 + lane;       // weight row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        for (int i = g; i < n && ok; i += 2) {
            const int rs = i % RSTG, buf = i % ABUF;
            ok = mbar_wait_warp(raw_full(i % RB), (i / RB) & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            uint4 cur[9];
            const uint4 *raw = reinterpret_cast<const uint4 *>(smem + C::oRaw + rs * RAW_BYTES + r * 144);
#pragma unroll
            for (int k = 0; k < 9; ++k) cur[k] = raw[k];
            fence_proxy_async_smem();   // these reads before the next TMA write into the slot
            __syncwarp();
            if (lane == 0) mbar_arrive(raw_empty(i % RB));
            const bool d_zero = (cur[0].x & 0x7FFFu) == 0u;
            const float d = __half2float(__ushort_as_half((unsigned short)(cur[0].x & 0xFFFFu)));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(cur[0].x >> 16)));
            const float rmult = __frcp_rn(d_zero ? 1.0f : d);
            float bh[8], bl[8];
            int scs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int sc, mm;
                q4::q4K_scale_min(cur[0].y, cur[0].z, cur[0].w, j, sc, mm);
                scs[j] = d_zero ? 0 : sc;
                const float v = -(dmin * (float)mm) * rmult;   // dmin*m exact: 11 x 6 bits
                bh[j] = to_tf32(v);
                bl[j] = to_tf32(v - bh[j]);
            }
            // TMEM buffer buf is free once unit i - ABUF's MMAs have completed
            ok = i < ABUF ||
                 mbar_wait_warp(a_empty((i - ABUF) % AB), ((i - ABUF) / AB) & 1, abort_flag, kKid, SITE_U_STAGE);
            if (!ok) break;
            tc_fence_after();
            const uint32_t acol = tmem_base + lane_off + C::TM_A + buf * 128;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                // sub-blocks 2pp (low nibbles) and 2pp+1 (high nibbles) of bytes 32pp..32pp+31
                const float slo = (float)scs[2 * pp], shi = (float)scs[2 * pp + 1];
                const __half2 mlo = __float2half2_rn(slo), alo = __float2half2_rn(-1024.0f * slo);
                const __half2 mhi = __float2half2_rn(shi * 0.0625f), ahi = __float2half2_rn(-64.0f * shi);
                uint32_t v[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 qv = cur[1 + 2 * pp + h];
                    const uint32_t wd[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const int c = 2 * (4 * h + wi);   // word 4h+wi holds the k pairs of columns c, c+1
                        const uint32_t lo = wd[wi] & 0x0F0F0F0Fu, hi = wd[wi] & 0xF0F0F0F0u;
                        v[c] = q4s::magic2(lo, 0x4140u, mlo, alo);
                        v[c + 1] = q4s::magic2(lo, 0x4342u, mlo, alo);
                        v[16 + c] = q4s::magic2(hi, 0x4140u, mhi, ahi);
                        v[16 + c + 1] = q4s::magic2(hi, 0x4342u, mhi, ahi);
                    }
                }
                tmem_st32(acol + 32 * pp, v);
            }
            q4::put_min_row(smem + C::oAmin + buf * AMIN_BYTES, r, bh, bl);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(i % AB));
        }
    } else if (warp >= WT_EPI0) {
        // --------------------------------------------------------- epilogue --
        const int r = (warp & 3) * 32 + lane;
        const int o = tile * 128 + r;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        float yv[N];
#pragma unroll
        for (int t = 0; t < N; ++t) yv[t] = 0.0f;
        // this row's d for unit i (rows past O: unused)
        auto load_d = [&](int i) -> uint32_t {
            if (o >= O) return 0u;
            return __ldg(reinterpret_cast<const unsigned short *>(p.w + ((size_t)o * nsb + (size_t)(sb0 + i)) * 144));
        };
        uint32_t d_next = n > 0 ? load_d(0) : 0u;
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
            const uint32_t dcur = d_next;
            if (i + 1 < n) d_next = load_d(i + 1);
            const int acc = i % NACC;
            ok = mbar_wait_warp(acc_full(acc), (i / NACC) & 1, abort_flag, kKid, SITE_E_ACC);
            if (!ok) break;
            tc_fence_after();
            const float mult =
                (dcur & 0x7FFFu) == 0u ? 1.0f : __half2float(__ushort_as_half((unsigned short)dcur));
            const uint32_t col = tmem_base + lane_off + C::TM_ACC + acc * C::NM;
#pragma unroll
            for (int q = 0; q < N; q += 16) {
                uint32_t a[16], b[16];
                tmem_ld16(col + q, a);         // D_hi of tokens q..q+15
                tmem_ld16(col + N + q, b);     // D_lo
                tmem_ld_wait2(a, b);
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    yv[q + t] = fmaf(mult, __uint_as_float(a[t]) + __uint_as_float(b[t]), yv[q + t]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(acc));
        }
        if (ks == 1) {
            if (ok && o < O) {
#pragma unroll
                for (int t = 0; t < N; ++t)
                    if (t < T) p.y[(size_t)t * O + o] = yv[t];
            }
        } else if (ok) {
            // this CTA's partial sums -> the (now idle) activation ring as
            // [t/4][row][4]: consecutive rows are consecutive 16-byte words
            float4 *red = reinterpret_cast<float4 *>(smem + C::oX) + r;
#pragma unroll
            for (int t = 0; t < N; t += 4) red[(t / 4) * 128] = make_float4(yv[t], yv[t + 1], yv[t + 2], yv[t + 3]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (ks > 1) {
        // the cluster's CTAs have left their partial sums in shared memory
        cluster_sync_all();
        if (cluster_ctarank() == 0 && warp >= WT_EPI0) {
            const int r = (warp & 3) * 32 + lane, o = tile * 128 + r;
            const uint32_t red = sbase + C::oX + (uint32_t)(r * 16);
            if (o < O) {
#pragma unroll
                for (int q = 0; q < N; q += 16) {
                    float s[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) s[t] = 0.0f;
                    for (int c0 = 0; c0 < ks; c0 += 4) {
                        // the loads of up to four ranks in flight, then added in rank order
                        // (the same sum on every call)
                        float4 v[4][4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (c0 + c < ks) {
                                const uint32_t src = dsmem_addr(red + (uint32_t)(q / 4) * 2048u, (uint32_t)(c0 + c));
#pragma unroll
                                for (int k = 0; k < 4; ++k) v[c][k] = ld_dsmem_f4(src + 2048u * k);
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (c0 + c < ks) {
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    s[4 * k] += v[c][k].x;
                                    s[4 * k + 1] += v[c][k].y;
                                    s[4 * k + 2] += v[c][k].z;
                                    s[4 * k + 3] += v[c][k].w;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (q + t < T) p.y[(size_t)(q + t) * O + o] = s[t];
                }
            }
        }
        // keep every CTA's shared memory until the first CTA has read it
        cluster_sync_all();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// SMs of the current device (cached per device)
static int device_sms()
{
    static int sms[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        sms[dev] = v;
    }
    return sms[dev];
}

// token tile of the weight-stationary kernel for T tokens (0: T too large)
static int wt_ntile(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : (T <= 64 ? 64 : 0)); }

template <int N>
int launch_wt_n(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                mmq_stream_t stream)
{
    using C = wts::Cfg<N>;
    const int nsb = K / 256, tiles = (O + 127) / 128;
    // CTAs per tile (cluster size): as many as keep the grid within one wave, at most 8
    const int sms = device_sms();
    int ks = std::max(1, std::min({wts::MAX_CLUSTER, nsb, (sms > 0 ? sms : 1) / tiles}));
    const int per = (nsb + ks - 1) / ks;
    ks = (nsb + per - 1) / per;
    CUtensorMap tmX, tmW, tmD;
    // xa [2][T][K] f16 as dims (64 k, T rows, 2 planes, K/64 chunks)
    const uint64_t xdims[4] = {64, (uint64_t)T, 2, (uint64_t)(K / 64)};
    const uint64_t xstr[3] = {(uint64_t)K * 2, (uint64_t)T * K * 2, 128};
    const uint32_t xbox[4] = {64, (uint32_t)N, 2, 1};
    int rc = make_tmap_4d(&tmX, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xdims, xstr, xbox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MMQ_OK) return rc;
    rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)nsb * 144, (uint64_t)O, (uint64_t)nsb * 144,
                      144, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    rc = make_tmap_2d(&tmD, ds, CU_TENSOR_MAP_DATA_TYPE_UINT32, (uint64_t)(K / 32), (uint64_t)T, (uint64_t)(K / 32) * 4,
                      8, N, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    static bool attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(mmq_q4K_wt_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::kDynSmem) != cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    WtParams prm;
    prm.w = static_cast<const uint8_t *>(w);
    prm.y = y;
    prm.T = T;
    prm.O = O;
    prm.K = K;
    prm.sb_per_split = per;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks, (unsigned)tiles, 1);
    cfg.blockDim = dim3(wts::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::kDynSmem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mmq_q4K_wt_kernel<N>, tmX, tmW, tmD, prm) != cudaSuccess) return launch_status();
    return launch_status();
}

int launch_q4K_wt(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                  mmq_stream_t stream)
{
    if (T < 0 || O < 1 || K < 256 || K > (1 << 20) || (K & 255) || wt_ntile(T) == 0) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !xa || !ds || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xa) || !aligned16(ds) || !aligned16(y)) return MMQ_ERR_ALIGN;
    int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    switch (wt_ntile(T)) {
    case 16: return launch_wt_n<16>(w, xa, ds, y, T, O, K, stream);
    case 32: return launch_wt_n<32>(w, xa, ds, y, T, O, K, stream);
    default: return launch_wt_n<64>(w, xa, ds, y, T, O, K, stream);
    }
}

template <int FMT, int MODE>
int launch(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int32_t *sub, int T, int O, int K,
           mmq_stream_t stream)
{
    using L = Layout<FMT>;
    if (T < 0 || O < 1 || K < 256 || K > (1 << 20) || (K & 255)) return MMQ_ERR_SHAPE;
    const long long nsb = K / 256;
    if (T == 0) return MMQ_OK;
    if (!w || !xh || (MODE == kFold && (!ds || !y)) || (MODE == kSubdots && !sub)) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(xh) || (ds && !aligned16(ds)) || (y && !aligned16(y)) ||
        (sub && !aligned16(sub)))
        return MMQ_ERR_ALIGN;
    int rc = check_arch();
    if (rc != MMQ_OK) return rc;

    CUtensorMap tmA, tmW;
    rc = make_tmap_2d(&tmA, xh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, BK, BM,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MMQ_OK) return rc;
    if (FMT == kQ4K || FMT == kQ5K) {
        const uint64_t rb = (uint64_t)(nsb * Fmt<FMT>::kBlockBytes);
        rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, rb, (uint64_t)O, rb, Fmt<FMT>::kBlockBytes, BN,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != MMQ_OK) return rc;
    } else if (FMT == kQ8_0) {
        // a row of K/32 34-byte blocks viewed as 16-bit elements (K % 256 == 0 makes it 16-byte aligned)
        const uint64_t rb = (uint64_t)(nsb * 272);
        rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT16, rb / 2, (uint64_t)O, rb, 136, BN,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != MMQ_OK) return rc;
    } else {
        std::memset(&tmW, 0, sizeof(tmW));   // q6_K stages its rows with plain bulk copies
    }

    const bool prod_q4K = (FMT == kQ4K && MODE == kFold);
    auto kern = prod_q4K ? mmq_q4K_kernel : mmq_gemm_kernel<FMT, MODE>;
    const uint32_t dyn_smem = prod_q4K ? q4::kDynSmem : L::kDynSmem;
    // the shared-memory attribute is set once per device (keeps the launch
    // path free of attribute calls, e.g. while a stream is being captured)
    static bool attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) != cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    Params prm{};
    prm.w = static_cast<const uint8_t *>(w);
    prm.ds = ds;
    prm.y = y;
    prm.sub = sub;
    prm.T = T;
    prm.O = O;
    prm.K = K;
    const dim3 grid((unsigned)((O + BN - 1) / BN), (unsigned)((T + BM - 1) / BM));
    kern<<<grid, prod_q4K ? q4::NTHREADS : NUM_THREADS, dyn_smem, reinterpret_cast<cudaStream_t>(stream)>>>(tmA, tmW,
                                                                                                    prm);
    return launch_status();
}

}  // namespace
}  // namespace mmq

extern "C" int mmq_gemm_q4K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
}

extern "C" int mmq_gemm_q5K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream, nullptr, nullptr, nullptr,
                              mmq::kQ5K);
}

extern "C" int mmq_gemm_q4K_small_imma(const void *w, const int8_t *qs, const uint32_t *ds, float *y, int T, int O,
                                       int K, mmq_stream_t stream)
{
    return mmq::launch_q4K_small(w, qs, ds, y, T, O, K, stream);
}

extern "C" int mmq_gemm_q4K_small(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O,
                                  int K, mmq_stream_t stream)
{
    return mmq::launch_q4K_wt(w, xa, ds, y, T, O, K, stream);
}

extern "C" int mmq_splitk_sizes(int T, int O, int K, int ksplit, int64_t *part_floats, int64_t *counters)
{
    if (T < 1 || O < 1 || K < 256 || K > (1 << 20) || (K & 255) || ksplit < 1) return MMQ_ERR_SHAPE;
    const int nsb = K / 256;
    const int sbps = (nsb + std::min(ksplit, nsb) - 1) / std::min(ksplit, nsb);
    const int splits = (nsb + sbps - 1) / sbps;
    if (part_floats) *part_floats = splits > 1 ? (int64_t)splits * T * O : 0;
    if (counters) *counters = (int64_t)((O + mmq::BN - 1) / mmq::BN) * ((T + mmq::BM - 1) / mmq::BM);
    return MMQ_OK;
}

extern "C" int mmq_gemm_q4K_splitk(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O,
                                   int K, int ksplit, float *part, int *counters, mmq_stream_t stream)
{
    if (ksplit < 1) return MMQ_ERR_SHAPE;
    if (ksplit > 1 && (!part || !counters)) return MMQ_ERR_NULL;
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, ksplit, part, counters, stream);
}

extern "C" int mmq_gemm_q4K_swiglu(const void *w_gu, const uint16_t *xa, const uint32_t *ds, uint16_t *h_xa,
                                   uint32_t *h_ds, int8_t *h_qs, int T, int F, int K, mmq_stream_t stream)
{
    if (F < 64 || F % 64 != 0 || F > (1 << 20)) return MMQ_ERR_SHAPE;
    if (!h_xa || !h_ds) return MMQ_ERR_NULL;
    return mmq::launch_q4K_sb(w_gu, xa, ds, nullptr, T, 2 * F, K, 1, nullptr, nullptr, stream, h_xa, h_ds, h_qs);
}

// Scratch of mmq_gemm_q4K_splitk_static: partial sums and tile counters in
// the library's own device memory (zero-initialised at module load; every
// completed launch leaves the counters at zero).
constexpr int64_t kStaticPartFloats = (int64_t)1 << 22;   // 16 MiB of f32 partial sums
constexpr int64_t kStaticCounters = 8192;                 // output tiles
static __device__ __align__(256) float g_splitk_part[kStaticPartFloats];
static __device__ __align__(256) int g_splitk_cnt[kStaticCounters];

extern "C" int mmq_gemm_q4K_splitk_static(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T,
                                          int O, int K, int ksplit, mmq_stream_t stream)
{
    if (T == 0) return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
    int64_t part_floats = 0, tiles = 0;
    const int rc = mmq_splitk_sizes(T, O, K, ksplit, &part_floats, &tiles);
    if (rc != MMQ_OK) return rc;
    // one split (ksplit == 1, or a single super-block per row) uses no scratch at all
    if (part_floats == 0) return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
    if (part_floats > kStaticPartFloats || tiles > kStaticCounters) return MMQ_ERR_SCRATCH;
    // device addresses of the two arrays, looked up once per device (with that
    // device current) under a lock, so that concurrent first calls from several
    // host threads do not race on the table
    static float *part[64];
    static int *cnt[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    float *pp = nullptr;
    int *cc = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!part[dev] || !cnt[dev]) {
            void *a = nullptr, *b = nullptr;
            if (cudaGetSymbolAddress(&a, g_splitk_part) != cudaSuccess ||
                cudaGetSymbolAddress(&b, g_splitk_cnt) != cudaSuccess)
                return mmq::launch_status();
            part[dev] = static_cast<float *>(a);
            cnt[dev] = static_cast<int *>(b);
        }
        pp = part[dev];
        cc = cnt[dev];
    }
    return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, ksplit, pp, cc, stream);
}

extern "C" int mmq_gemm_q4K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ4K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_gemm_q6K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q6K_sb(w, xa, ds, y, T, O, K, stream);
}

extern "C" int mmq_gemm_q6K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ6K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q4K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ4K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_gemm_q5K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ5K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_gemm_q8_0(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                             mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ8_0, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q5K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ5K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q8_0(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                      mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ8_0, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q6K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ6K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_fault_inject(int mode, int wait_limit_us)
{
    if (mode < 0 || mode > 1) return MMQ_ERR_SHAPE;
    const unsigned long long lim =
        wait_limit_us > 0 ? (unsigned long long)wait_limit_us * 1000ull : mmq::kWaitLimitNs;
    if (cudaMemcpyToSymbol(mmq::g_inject, &mode, sizeof(mode)) != cudaSuccess ||
        cudaMemcpyToSymbol(mmq::g_wait_limit_ns, &lim, sizeof(lim)) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return MMQ_OK;
}

// extra detail of the last failure reported by mmq_check_status (host side)
static int g_last_failure[4];

extern "C" int mmq_check_status(mmq_stream_t stream, int *detail)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        if (detail) detail[0] = detail[1] = detail[2] = detail[3] = 0;
        return MMQ_ERR_CUDA;
    }
    int h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(h, mmq::g_status, sizeof(h)) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    if (h[0] != 0) {
        const int zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        cudaMemcpyToSymbol(mmq::g_status, zero, sizeof(zero));
        for (int i = 0; i < 4; ++i) g_last_failure[i] = h[4 + i];
    }
    if (detail)
        for (int i = 0; i < 4; ++i) detail[i] = h[i];
    return h[0];
}

extern "C" int mmq_last_failure_info(int *info)
{
    if (!info) return MMQ_ERR_NULL;
    for (int i = 0; i < 4; ++i) info[i] = g_last_failure[i];
    return MMQ_OK;
}

// decode-shaped q4_K and q6_K products (mmq_gemv_q4K, mmq_gemv_q6K): in this unit for their bounded waits
// and the status word
#include "mmq_gemv.cuh"
#include "mmq_gemv_q6.cuh"
