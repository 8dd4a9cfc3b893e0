// mmq_prod_q6K.cuh -- the production q6_K GEMM (super-block accumulation,
// exact hi/lo weight planes; mmq_gemm_q6K) and its launcher.
#pragma once

namespace mmq {
namespace {

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

}  // namespace
}  // namespace mmq
