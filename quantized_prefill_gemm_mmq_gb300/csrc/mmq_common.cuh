// mmq_common.cuh -- tile shapes, weight-format descriptions, kernel parameters,
// wait sites and small unpack helpers shared by the GEMM kernels of libmmq.
// Included only by mmq_gemm.cu (one translation unit owns every kernel, so
// that all of them report into the one device status word that
// mmq_check_status reads).
#pragma once

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
    // production q4_K / q6_K, one split: nonzero when y is written by tensor
    // stores of the tile (y's row stride O*4 bytes a multiple of 16)
    int y_tma;
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

}  // namespace
}  // namespace mmq
