// mmq_prod_q6K.cuh -- the production q6_K GEMM (super-block accumulation,
// exact hi/lo weight planes; mmq_gemm_q6K) and its launcher.
#pragma once

namespace mmq {
namespace {

// =========================================================================
// q6_K GEMM with super-block accumulation (production).
//
// The layout of the production q4_K kernel: the weight rows are the MMA's A
// operand (M = 128 weight rows = TMEM lanes) and the two exact f16 planes of
// the dequantised activations of 128 tokens, stacked (hi rows, then lo rows),
// its B operand (N = 256), so one accumulator per super-block receives
//     D_sb[o][t]       = sum_{k in sb} sc(o,k)*(q-32)[o][k] * hi[t][k]
//     D_sb[o][128 + t] = sum_{k in sb} sc(o,k)*(q-32)[o][k] * lo[t][k]
// and the epilogue adds Y += d*(D_hi + D_lo) once per super-block.  The
// weight values sc*(q-32) reach +-4096 and above 2048 f16 holds only even
// integers, so the weight operand is two exact f16 planes too:
// w_hi = f16(sc*(q-32)) and w_lo = sc*(q-32) - w_hi in {-1, 0, 1}.  Per 16-k
// step the tensor core runs w_hi x (hi | lo) and w_lo x (hi | lo) into the
// same accumulator: all four products, each exact in f32.  (Dropping
// w_lo x lo, N = 128 for the second MMA, measured no faster.)  q6_K has no
// min term.
// 64-k stages (128-byte swizzled rows) of four tiles: activation hi and lo
// (one B operand of 256 rows), weight hi, weight lo.  Raw blocks are 210
// bytes, so rows are 2-byte aligned in memory, but eight consecutive rows
// span 8*nsb*210 bytes, a multiple of 16: viewed as [O/8][8*nsb*210] bytes,
// the blocks of super-block sb in rows 8g + i (i fixed, g = 0..15) are one
// 2-D TMA box of 16 x 224 bytes (the 16-byte-aligned window around them),
// so a super-block of the tile arrives as eight boxes, one super-block
// ahead.  (One bulk copy per row was measured ~9400 cycles from issue to
// arrival against ~1600 for the boxes; it remains for the one tile that
// holds an incomplete group of eight rows.)  At the start of a super-block
// each unpack thread realigns its row's 208 bytes of quants and scales into
// registers and releases the slot at once.
// One MMA-issuing thread waiting once per stage on a merged "full" barrier;
// TMEM: two rotating super-block accumulators of 256 columns; the output
// tile leaves through TMA tensor stores when O is a multiple of 4.
// Warps: 0 raw-weight producer, 1 MMA issuer, 14 activation TMA producer,
// 2-5 unpack (thread = weight row), 6-13 epilogue (weight row x 64 tokens).
// =========================================================================
namespace q6s {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int RAW_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int ACT_WARP = 14;
constexpr int STG = 3;                            // operand ring: act hi + lo, weight hi, weight lo per 64-k stage
constexpr int NACC = 2;                           // rotating super-block accumulators
constexpr int RAW_COPY = 224;                     // 16-byte-aligned window holding one 210-byte block
constexpr uint32_t RAW_PHASE = 16 * RAW_COPY;     // rows 8g + i of the tile, g = 0..15: one box
constexpr uint32_t ACC_COLS = 2 * BM;             // hi tokens, then lo tokens
static_assert(NACC * ACC_COLS <= 512, "TMEM budget");
constexpr uint32_t ACT_STAGE = 2 * A_BYTES;       // hi and lo planes of BM tokens
constexpr uint32_t W_TILE = B_BYTES;              // 128 weight rows x 64 k f16
constexpr uint32_t STAGE_BYTES = ACT_STAGE + 2 * W_TILE;
constexpr uint32_t RAW_BYTES = 8 * RAW_PHASE;
constexpr uint32_t oStage = 0;
constexpr uint32_t oRaw = oStage + STG * STAGE_BYTES;
constexpr uint32_t oMult = oRaw + RAW_BYTES;      // d per weight row, [NACC][BN] f32
constexpr uint32_t oBar = oMult + NACC * BN * 4;
// full, empty [STG]; acc_full, acc_empty, m_full [NACC]; r_full, r_empty; mma_done
constexpr int kNumBars = 2 * STG + 3 * NACC + 2 + 1;
constexpr uint32_t oMisc = oBar + kNumBars * 8;
constexpr uint32_t kDynSmem = oMisc + 16 + 1024;
static_assert(kDynSmem <= 232448, "shared memory budget");
static_assert(STAGE_BYTES % 1024 == 0 && oRaw % 1024 == 0 && RAW_PHASE % 128 == 0 && RAW_COPY % 16 == 0 &&
                  oMult % 16 == 0,
              "swizzle atoms are 1024-byte aligned; box destinations 128-byte, bulk copies 16-byte aligned");

// Raw slot position of tile row rho: box rho % 8, row rho / 8 of the box.
__device__ __forceinline__ uint32_t raw_row_off(int rho) { return (uint32_t)(rho & 7) * RAW_PHASE + (uint32_t)(rho >> 3) * RAW_COPY; }

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
    mmq_q6K_sb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmY, const Params p)
{
    using namespace q6s;
    constexpr int kKid = 10;
    constexpr uint32_t kIdesc = idesc_f16_f32(BN, ACC_COLS);      // M = weight rows, N = hi + lo tokens

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int T = p.T, K = p.K, O = p.O;
    const int nsb = K / 256, nks = nsb * 4;

    const uint32_t bar0 = sbase + oBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STG + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (2 * STG + s); };
    auto acc_empty = [&](int s) { return bar0 + 8u * (2 * STG + NACC + s); };
    auto m_full = [&](int s) { return bar0 + 8u * (2 * STG + 2 * NACC + s); };
    const uint32_t r_full = bar0 + 8u * (2 * STG + 3 * NACC);
    const uint32_t r_empty = r_full + 8u;
    const uint32_t mma_done = bar0 + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + oMisc + 4);
    auto stage_a = [&](int s) { return sbase + oStage + (uint32_t)s * STAGE_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STG; ++s) {
            mbar_init(full(s), 1 + 128);                    // the TMA request (with its bytes) + unpack threads
            mbar_init(empty(s), 1);                         // the issuer's commit
        }
        for (int s = 0; s < NACC; ++s) {
            mbar_init(acc_full(s), 1);                      // the issuer's commit
            mbar_init(acc_empty(s), NUM_EPI_WARPS);         // after the epilogue has also read d
            mbar_init(m_full(s), 128);                      // unpack threads' d
        }
        mbar_init(r_full, 32);                              // raw producer lanes (with their bytes)
        mbar_init(r_empty, 128);                            // unpack threads
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == MMA_WARP) {
        // ------------------------------------------------------ MMA issuer --
        if (lane == 0) {
            bool ok = true;
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % STG;
                const int sb = ks >> 2, p4 = ks & 3, slot = sb % NACC;
                ok = (p4 != 0 || mbar_wait(acc_empty(slot), ((sb / NACC) & 1) ^ 1, abort_flag, kKid, SITE_M_ACC)) &&
                     mbar_wait(full(s), (ks / STG) & 1, abort_flag, kKid, SITE_M_A);
                if (!ok) break;
                tc_fence_after();
                const uint32_t st = stage_a(s);
                const uint64_t dx = sdesc_k_sw128(st);                        // hi rows then lo rows: B
                const uint64_t dwh = sdesc_k_sw128(st + ACT_STAGE);           // weight hi plane: A
                const uint64_t dwl = sdesc_k_sw128(st + ACT_STAGE + W_TILE);  // weight lo plane: A
                const uint32_t d_acc = tmem_base + slot * ACC_COLS;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // +32 bytes along K within the 128-byte swizzled rows = +2 in the address field
                    umma_f16(d_acc, dwh + 2 * kk, dx + 2 * kk, kIdesc, (p4 == 0 && kk == 0) ? 0u : 1u);
                    umma_f16(d_acc, dwl + 2 * kk, dx + 2 * kk, kIdesc, 1u);
                }
                if (p4 == 3) umma_commit(acc_full(slot));
                umma_commit(empty(s));
            }
            umma_commit(mma_done);
            if (!wait_drain(mma_done, 0)) record_error(kStatusTimeout, kKid, SITE_DRAIN);
        }
        __syncwarp();
    } else if (warp == ACT_WARP) {
        // ------------------------------------------- activation TMA producer --
        // activation tiles of stage k: [2T][K] tensor, hi plane rows 0..T-1, lo plane rows T..2T-1
        if (lane == 0) {
            tma_prefetch(&tmA);
            bool ok = true;
            int n_a = 0;   // stages requested, for the drain on abort
            for (int ks = 0; ks < nks && ok; ++ks) {
                const int s = ks % STG;
                // slot s is free once stage ks - STG's MMAs have completed
                ok = ks < STG || mbar_wait(empty(s), ((ks / STG) - 1) & 1, abort_flag, kKid, SITE_P_STAGE);
                if (!ok) break;
                mbar_arrive_expect_tx(full(s), ACT_STAGE);
                tma_load_2d(stage_a(s), &tmA, full(s), ks * BK, t0);
                tma_load_2d(stage_a(s) + A_BYTES, &tmA, full(s), ks * BK, T + t0);
                n_a = ks + 1;
            }
            // On abort: let the copies in flight land before the CTA exits (a
            // stage's barrier also counts the unpack threads' arrivals, so
            // where those stopped first this wait ends at its time limit).
            if (!ok)
                for (int i = max(0, n_a - STG); i < n_a; ++i) wait_drain(full(i % STG), (i / STG) & 1);
        }
        __syncwarp();
    } else if (warp == RAW_WARP) {
        // --------------------------------------------------- raw producer --
        // Tiles made of whole groups of eight rows: eight TMA boxes per
        // super-block (rows past O arrive zero-filled).  The tile holding an
        // incomplete group: one bulk copy per row of the 224-byte window
        // around its block (past the buffer's last full 16-byte granule the
        // bytes are copied one by one; rows past O are not copied).
        const int nrows = min(BN, O - o0);
        const long long nbytes = (long long)O * nsb * 210;
        const bool boxes = (O % 8) == 0 || o0 + BN <= 8 * (O / 8);
        if (boxes && lane == 0) tma_prefetch(&tmW);
        bool ok = true;
        int n_r = 0;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            ok = mbar_wait(r_empty, (sb & 1) ^ 1, abort_flag, kKid, SITE_P_RAW);
            if (!ok) break;
            if (boxes) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(r_full, RAW_BYTES);
#pragma unroll 1
                    for (int i = 0; i < 8; ++i)
                        tma_load_2d(sbase + oRaw + i * RAW_PHASE, &tmW, r_full,
                                    (int)((((long long)i * nsb + sb) * 210) & ~15ll), o0 / 8);
                } else {
                    mbar_arrive(r_full);
                }
                n_r = sb + 1;
                continue;
            }
            uint32_t mine = 0;
            for (int r = lane; r < nrows; r += 32) {
                const long long start = ((long long)(o0 + r) * nsb + sb) * 210;
                const long long a = start & ~15ll;
                uint32_t sz = RAW_COPY;
                if (a + RAW_COPY > nbytes) {
                    sz = (uint32_t)((nbytes - a) & ~15ll);
                    uint8_t *drow = smem + oRaw + raw_row_off(r);
                    for (long long i = a + sz; i < start + 210; ++i) drow[i - a] = p.w[i];
                }
                mine += sz;
            }
            mbar_arrive_expect_tx(r_full, mine);
            for (int r = lane; r < nrows; r += 32) {
                const long long start = ((long long)(o0 + r) * nsb + sb) * 210;
                const long long a = start & ~15ll;
                uint32_t sz = RAW_COPY;
                if (a + RAW_COPY > nbytes) sz = (uint32_t)((nbytes - a) & ~15ll);
                if (sz) bulk_load(sbase + oRaw + raw_row_off(r), p.w + a, sz, r_full);
            }
            n_r = sb + 1;
        }
        if (!ok && n_r > 0) wait_drain(r_full, (n_r - 1) & 1);
    } else if (warp >= UNPACK_WARP0 && warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        // Thread = one weight row rho.  At the start of a super-block it
        // realigns the row's 128 ql, 64 qh and 16 scale bytes into registers
        // and publishes d; per 64-k stage it writes the row's 64 values
        // sc*(q-32) as exact hi and lo f16 planes into the swizzled tiles.
        // Threads 8p + i take rows 8*((p + i/2) % 16) + i: the eight threads of
        // a 16-byte access phase then store to eight different swizzle rows
        // and read their raw rows from four different bank groups.
        const int ut = threadIdx.x - UNPACK_WARP0 * 32;
        const int r = 8 * (((ut >> 3) + ((ut & 7) >> 1)) & 15) + (ut & 7);
        const int o = o0 + r;
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            const int slot = sb % NACC;
            ok = mbar_wait(r_full, sb & 1, abort_flag, kKid, SITE_U_RAW);
            if (!ok) break;
            const uint8_t *row = smem + oRaw + raw_row_off(r);
            // rows past O were not copied: their (stale) bytes feed weight rows that are never stored
            const int lead = (int)((((long long)min(o, O - 1) * nsb + sb) * 210) & 15);
            uint32_t w[52];   // block words: ql 0..31, qh 32..47, scales 48..51
            row_words<52>(row, lead, w);
            const uint16_t d16 = *reinterpret_cast<const uint16_t *>(row + lead + 208);
            fence_proxy_async_smem();   // these reads before the next bulk copy into the slot
            mbar_arrive(r_empty);
            // d of this super-block for the epilogue, once super-block sb - NACC's was read
            if (sb >= NACC) {
                const int prev = sb - NACC;
                ok = mbar_wait(acc_empty(prev % NACC), (prev / NACC) & 1, abort_flag, kKid, SITE_U_SDS);
                if (!ok) break;
            }
            reinterpret_cast<float *>(smem + oMult + slot * BN * 4)[r] = o < O ? __half2float(__ushort_as_half(d16)) : 0.0f;
            mbar_arrive(m_full(slot));
#pragma unroll
            for (int p4 = 0; p4 < 4; ++p4) {
                // stage p4 = values 64*p4 .. 64*p4 + 63 of the super-block: half h of 128,
                // groups g = 2*(p4 & 1) and g + 1 of 32 values.  Value i of group g: ql byte
                // 64h + 32*(g & 1) + i (low nibble for g < 2, high for g >= 2), qh byte
                // 32h + i bits 2g..2g+1, scale byte 8h + 2g + i/16.
                const int ks = sb * 4 + p4, s = ks % STG;
                const int h = p4 >> 1, odd = p4 & 1;
                // slot s is free once stage ks - STG's MMAs have completed
                ok = ks < STG || mbar_wait(empty(s), ((ks / STG) - 1) & 1, abort_flag, kKid, SITE_U_STAGE);
                if (!ok) break;
                uint8_t *bh = smem + oStage + s * STAGE_BYTES + ACT_STAGE + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    // 16-byte chunk c: values 8c .. 8c + 7 of the stage
                    const int gi = c >> 2, g = 2 * odd + gi, q = c & 3;
                    const int sub = 8 * h + 2 * g + (q >> 1);
                    const int sc = (int)(int8_t)((w[48 + (sub >> 2)] >> (8 * (sub & 3))) & 0xFFu);
                    const __half2 sc2 = __float2half2_rn((float)sc);
                    uint32_t hv[4], lv[4];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t lw = w[16 * h + 8 * gi + 2 * q + e], hw = w[32 + 8 * h + 2 * q + e];
                        const uint32_t lo4 = (odd ? (lw >> 4) : lw) & 0x0F0F0F0Fu;
                        const uint32_t hi2 = ((hw >> (2 * g)) & 0x03030303u) << 4;
                        q6_pairs(lo4 | hi2, sc2, hv[2 * e], hv[2 * e + 1], lv[2 * e], lv[2 * e + 1]);
                    }
                    const int cc = (c ^ (r & 7)) << 4;
                    *reinterpret_cast<uint4 *>(bh + cc) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<uint4 *>(bh + W_TILE + cc) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(full(s));
            }
        }
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + NUM_EPI_WARPS) {
        // --------------------------------------------------------- epilogue --
        // Thread = one weight row (TMEM lane) x 64 tokens; Y += d*(D_hi + D_lo)
        // per super-block in registers.
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;         // TMEM lanes 32*quarter.. are this warp's
        const int c0 = (ew >> 2) * 64;        // first token of this thread within the tile
        const int row = quarter * 32 + lane;  // weight row within the tile
        const int o = o0 + row;
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
            const float d = reinterpret_cast<const float *>(smem + oMult + slot * BN * 4)[row];
            const float2 d2 = make_float2(d, d);
            const uint32_t col = tmem_base + lane_off + slot * ACC_COLS + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t ra[16], rb[16];
                tmem_ld16(col + q * 16, ra);        // hi-plane products of tokens c0 + 16q ..
                tmem_ld16(col + BM + q * 16, rb);   // lo-plane products of the same tokens
                tmem_ld_wait2(ra, rb);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 s = __fadd2_rn(make_float2(__uint_as_float(ra[i]), __uint_as_float(ra[i + 1])),
                                                make_float2(__uint_as_float(rb[i]), __uint_as_float(rb[i + 1])));
                    const int e = q * 16 + i;
                    const float2 y = __ffma2_rn(s, d2, make_float2(yv[e], yv[e + 1]));
                    yv[e] = y.x;
                    yv[e + 1] = y.y;
                }
            }
            // the accumulator and this super-block's d have been read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(slot));
        }
        if (p.y_tma) {
            // the tile staged in the idle operand ring as four [128 tokens][32 rows]
            // boxes (one per TMEM lane quarter), written by four tensor stores; rows
            // past O and tokens past T are clipped by the map
            float *ys = reinterpret_cast<float *>(smem + oStage) + quarter * (BM * 32) + c0 * 32 + lane;
            if (ok) {   // (after an abort, copies in flight may still land in the ring)
#pragma unroll
                for (int i = 0; i < 64; ++i) ys[i * 32] = yv[i];
            }
            fence_proxy_async_smem();
            named_bar_sync(1, NUM_EPI_WARPS * 32);
            if (warp == EPI_WARP0 && lane == 0 && *abort_flag == 0u) {
                for (int q = 0; q < 4 && o0 + 32 * q < O; ++q)
                    tma_store_2d(&tmY, sbase + oStage + (uint32_t)q * (BM * 32 * 4), o0 + 32 * q, t0);
                bulk_commit_group();
                bulk_wait_all();
            }
        } else {
            // this thread's outputs: column o of rows t0 + c0 .. t0 + c0 + 63 of the [T][O] array
            const int nt = min(64, T - t0 - c0);
            if (ok && o < O) {
                float *base = p.y + (size_t)(t0 + c0) * O + o;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < nt) base[(size_t)i * O] = yv[i];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
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
    CUtensorMap tmA, tmW, tmY;
    rc = make_tmap_2d(&tmA, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, 2ull * (uint64_t)T, (uint64_t)K * 2,
                      BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MMQ_OK) return rc;
    // raw weights as [O/8][8*nsb*210] bytes, boxes of 16 groups x 224 bytes (unused when O < 8)
    std::memset(&tmW, 0, sizeof(tmW));
    const uint64_t group_bytes = 8ull * (uint64_t)(K / 256) * 210ull;
    if (O >= 8) {
        rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, group_bytes, (uint64_t)(O / 8), group_bytes,
                          q6s::RAW_COPY, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != MMQ_OK) return rc;
    }
    // y by tensor stores ([T][O] f32, boxes of 32 rows x 128 tokens) when its row stride allows
    const bool y_tma = (O % 4) == 0;
    std::memset(&tmY, 0, sizeof(tmY));
    if (y_tma) {
        rc = make_tmap_2d(&tmY, y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)O, (uint64_t)T, (uint64_t)O * 4, 32, BM,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != MMQ_OK) return rc;
    }
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
    prm.y_tma = y_tma ? 1 : 0;
    const dim3 grid((unsigned)((O + BN - 1) / BN), (unsigned)((T + BM - 1) / BM));
    mmq_q6K_sb_kernel<<<grid, q6s::NTHREADS, q6s::kDynSmem, reinterpret_cast<cudaStream_t>(stream)>>>(tmA, tmW, tmY, prm);
    return launch_status();
}

}  // namespace
}  // namespace mmq
