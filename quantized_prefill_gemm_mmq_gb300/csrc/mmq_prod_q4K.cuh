// mmq_prod_q4K.cuh -- the production q4_K / q5_K GEMM (super-block
// accumulation on the tensor core; mmq_gemm_q4K, _q5K, the split-K forms and
// the chained FFN's SwiGLU epilogue, mmq_gemm_q4K_swiglu) and its launcher.
#pragma once

namespace mmq {
namespace {

// =========================================================================
// q4_K GEMM with super-block accumulation (production).
//
// The sum over a super-block's 8 sub-blocks of dx_b*sc_b*C_b is computed by
// the tensor core itself: the activation operand is the dequantised q8_1
// value v = f32(d16)*q split into two exact f16 planes (v = hi + lo, see the
// quantiser), the weight operand is sc*q (exact), so each product is exact in
// f32 and one TMEM accumulator per super-block receives
//     D_sb[o][t]     = sum_{k in sb} sc_b(o)*q[o][k] * hi[t][k]
//     D_sb[o][T + t] = sum_{k in sb} sc_b(o)*q[o][k] * lo[t][k]
// The weight tile is the MMA's A operand (M = 128 weight rows = TMEM lanes)
// and the two activation planes of the 128 tokens, stacked, its B operand
// (N = 256), so one 128x256x16 MMA per 16-k step covers both planes and the
// weight tile is read from shared memory once per step.  The epilogue needs
// one add and one FMA per output per super-block, Y += d*(D_hi + D_lo) (Y
// held in registers, d a per-thread scalar since a thread owns a weight row).
// The min term rides in the same accumulator: the tensor core also adds
// sum_j (-(dmin*m_j)/d) * (dx_j*ssum_j) (split-tf32 MMAs over the sub-block
// index, into the hi half), so that d*D_sb carries both terms of the
// super-block.  For rows with d == 0 the weight operand is zero and the min
// operand is divided by 1 instead.  The per-sub-block integer dots are not
// formed here (see mmq_q4K_kernel / the sub-block diagnostics for those);
// the result differs from them only in f32 rounding.
//
// One MMA-issuing thread; every accumulator sees its MMAs in one fixed order,
// so results are reproducible bit for bit.  Measured on sm_103a: 128x256x16
// MMAs issued back to back from distinct shared-memory tiles run at the full
// 128 cycles each and a commit that nobody waits for costs nothing, but an
// mbarrier wait by the issuing thread (even on a completed phase) returns
// only after that thread's queued MMAs have completed, so each wait between
// two stages leaves the tensor core idle for the wait's own latency.  The
// issuer therefore waits once per stage, on the stage's single "full"
// barrier (the activation tiles' TMA bytes and the 128 unpack threads'
// arrivals), and then issues the four MMAs and one commit.  (Splitting that
// barrier in two, handing the accumulator between two issuers after every
// stage, or two issuers on halves of the tokens were each measured slower.)
// Per 64-k stage the activation tiles (hi rows, then lo rows: one B operand
// of 256 K-major rows) are requested by a producer warp as soon as the slot
// is free.  The raw weight super-blocks (128 rows x 144 bytes) arrive by TMA
// one super-block ahead; the unpack and scale threads copy what they need to
// registers at the start of a super-block and release the raw slot at once.
// TMEM: two rotating super-block accumulators of 256 columns.  The finished
// output tile leaves through TMA tensor stores from the idle operand ring
// (one split, O a multiple of 4; otherwise every thread stores its column).
// Warps: 1 MMA issuer, 14 activation TMA, 2-5 unpack (+ raw weight TMA),
// 6-13 epilogue, 0 and 15 scale.
// =========================================================================
namespace q4s {

constexpr int NWARPS = 16;
constexpr int NTHREADS = NWARPS * 32;
constexpr int MMA_WARP = 1;
constexpr int ACT_WARP = 14;                      // activation TMA producer
constexpr int SCALE_WARP_B = 15;                  // scale warps: 0 and 15
constexpr int STG = 3;                            // operand ring: act hi, act lo, weights per 64-k stage
constexpr int RSTG = 2;                           // raw weight super-block ring
constexpr int SSTG = 2;                           // scale / min-operand ring
constexpr int NACC = 2;                           // rotating super-block accumulators
constexpr uint32_t ACC_COLS = 2 * BM;             // hi tokens, then lo tokens
static_assert(NACC * ACC_COLS <= 512, "TMEM budget");
constexpr uint32_t ACT_STAGE = 2 * A_BYTES;       // hi and lo planes of BM tokens
constexpr uint32_t STAGE_BYTES = ACT_STAGE + B_BYTES;
constexpr uint32_t MIN_OP_BYTES = 128 * 64;
constexpr uint32_t SDS_D = 2 * MIN_OP_BYTES;
constexpr uint32_t SDS_BYTES = SDS_D + BN * 4;
constexpr uint32_t oStage = 0;
constexpr uint32_t oRaw = oStage + STG * STAGE_BYTES;   // then the raw ring, scale ring and barriers (SbLayout)
// full, empty [STG]; s_full [SSTG]; acc_full, acc_empty [NACC]; r_full, r_empty [RSTG]; mma_done
constexpr int kNumBars = 2 * STG + SSTG + 2 * NACC + 2 * RSTG + 1;
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

}  // namespace q4s

// SWIGLU: the tile's output is not stored as y but finished as silu(gate)*up and
// quantised to q8_1 (Params::h_xa).
// FMT: kQ4K, or kQ5K (the same header and scale packing, a 5-bit quant whose
// fifth bits come from a 32-byte qh plane: sc*q <= 1953 is still exact in f16).
template <int FMT, bool SWIGLU>
__global__ void __launch_bounds__(q4s::NTHREADS, 1)
    mmq_q4K_sb_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmY, const Params p)
{
    using namespace q4s;
    using SL = SbLayout<FMT>;
    constexpr int RAW_ROW = SL::RAW_ROW;
    constexpr uint32_t RAW_BYTES = SL::RAW_BYTES, oSds = SL::oSds, oBar = SL::oBar, oMisc = SL::oMisc;
    constexpr int kKid = 9;
    constexpr uint32_t kIdesc = idesc_f16_f32(BN, ACC_COLS);      // M = weight rows, N = hi + lo tokens
    constexpr uint32_t kIdescTf32 = idesc_tf32_f32(BN, BM);       // min term: weight rows x tokens

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
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STG + s); };
    auto s_full = [&](int s) { return bar0 + 8u * (2 * STG + s); };
    auto acc_full = [&](int s) { return bar0 + 8u * (2 * STG + SSTG + s); };
    auto acc_empty = [&](int s) { return bar0 + 8u * (2 * STG + SSTG + NACC + s); };
    auto r_full = [&](int s) { return bar0 + 8u * (2 * STG + SSTG + 2 * NACC + s); };
    auto r_empty = [&](int s) { return bar0 + 8u * (2 * STG + SSTG + 2 * NACC + RSTG + s); };
    const uint32_t mma_done = bar0 + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + oMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + oMisc + 4);
    auto stage_a = [&](int s) { return sbase + oStage + (uint32_t)s * STAGE_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STG; ++s) {
            mbar_init(full(s), 1 + 128);                    // the TMA request (with its bytes) + unpack threads
            mbar_init(empty(s), 1);                         // the issuer's commit
        }
        for (int s = 0; s < SSTG; ++s) mbar_init(s_full(s), 64);   // scale threads
        for (int s = 0; s < NACC; ++s) {
            mbar_init(acc_full(s), 1);                      // the issuer's commit
            mbar_init(acc_empty(s), NUM_EPI_WARPS);         // after the epilogue has also read d
        }
        for (int s = 0; s < RSTG; ++s) {
            mbar_init(r_full(s), 1);
            mbar_init(r_empty(s), 128 + 64);                // unpack and scale threads
        }
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
                const uint64_t dw = sdesc_k_sw128(st + ACT_STAGE);   // weight tile: A, 128 rows
                const uint64_t dx = sdesc_k_sw128(st);               // hi rows then lo rows: B, 256 rows
                const uint32_t d_acc = tmem_base + slot * ACC_COLS;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    // +32 bytes along K within the 128-byte swizzled rows = +2 in the address field
                    umma_f16(d_acc, dw + 2 * kk, dx + 2 * kk, kIdesc, (p4 == 0 && kk == 0) ? 0u : 1u);
                if (p4 == 3) {
                    // min term of this super-block, into the hi half
                    const int ss = sb % SSTG;
                    ok = mbar_wait(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t am = sbase + oSds + ss * SDS_BYTES, bm = am + MIN_OP_BYTES;
                    umma_tf32(d_acc, sdesc_k_none(bm, 128, 512), sdesc_k_none(am, 128, 512), kIdescTf32, 1u);
                    umma_tf32(d_acc, sdesc_k_none(bm, 128, 512), sdesc_k_none(am + 256, 128, 512), kIdescTf32, 1u);
                    umma_tf32(d_acc, sdesc_k_none(bm + 256, 128, 512), sdesc_k_none(am, 128, 512), kIdescTf32, 1u);
                    umma_commit(acc_full(slot));
                }
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
                tma_load_2d(stage_a(s), &tmA, full(s), (sb_base * 4 + ks) * BK, t0);
                tma_load_2d(stage_a(s) + A_BYTES, &tmA, full(s), (sb_base * 4 + ks) * BK, T + t0);
                n_a = ks + 1;
            }
            // On abort: let the copies in flight land before the CTA exits.  A
            // stage's barrier also counts the unpack threads' arrivals, so
            // where those stopped first this wait ends at its time limit.
            if (!ok)
                for (int i = max(0, n_a - STG); i < n_a; ++i) wait_drain(full(i % STG), (i / STG) & 1);
        }
        __syncwarp();
    } else if (warp >= UNPACK_WARP0 && warp < EPI_WARP0) {
        // ------------------------------------------------------ unpack warps --
        // Thread = one weight row (rows past O arrive zero-filled).  At the
        // start of a super-block it copies the row's 144 raw bytes to
        // registers; per 64-k stage it writes the row's 64 values sc*q as f16
        // into the swizzled weight tile (zeros when the row's d is zero).
        // Thread 0 also issues the raw tile one super-block ahead.
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
                const int ks = sb * 4 + p4, s = ks % STG;
                uint4 (&vc)[8] = (p4 & 1) ? vb : va;
                uint4 (&vn)[8] = (p4 & 1) ? va : vb;
                // slot s is free once stage ks - STG's MMAs have completed
                ok = ks < STG || mbar_wait(empty(s), ((ks / STG) - 1) & 1, abort_flag, kKid, SITE_U_STAGE);
                if (!ok) break;
                uint8_t *brow = smem + oStage + s * STAGE_BYTES + ACT_STAGE + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(brow + ((c ^ (r & 7)) << 4)) = vc[c];
                if (p4 < 3) convert(p4 + 1, vn);
                fence_proxy_async_smem();
                mbar_arrive(full(s));
            }
        }
        if (!ok && r == 0)   // let the copies in flight land before the CTA exits
            for (int i = max(0, n_raw - RSTG); i < n_raw; ++i) wait_drain(r_full(i % RSTG), (i / RSTG) & 1);
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
            const int slot = sb % NACC, ss = sb % SSTG;
            ok = mbar_wait_warp(s_full(ss), (sb / SSTG) & 1, abort_flag, kKid, SITE_E_SDS) &&
                 mbar_wait_warp(acc_full(slot), (sb / NACC) & 1, abort_flag, kKid, SITE_E_ACC);
            if (!ok) break;
            tc_fence_after();
            const float d = reinterpret_cast<const float *>(smem + oSds + ss * SDS_BYTES + SDS_D)[row];
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
        if constexpr (SWIGLU) {
            // Park the tile in shared memory for the CTA-wide SwiGLU pass at the
            // end (the operand ring is idle now that every MMA has completed):
            // rows 0..63 are the gate rows of features 64*bx .., rows 64..127 the
            // up rows of the same features; stored [token][feature].
            float *gu = reinterpret_cast<float *>(smem + oStage) + (row >= 64 ? BM * q4s::GU_STRIDE : 0) + (row & 63) +
                        c0 * q4s::GU_STRIDE;
#pragma unroll
            for (int i = 0; i < 64; ++i) gu[i * q4s::GU_STRIDE] = yv[i];
        }
        // this thread's outputs: column o of rows t0 + c0 .. t0 + c0 + 63 of a [T][O] array
        const int nt = min(64, T - t0 - c0);
        const bool col_ok = o < O;
        auto store_col = [&](float *base) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (i < nt) base[(size_t)i * O] = yv[i];
        };
        if (SWIGLU) {
            // written above
        } else if ((p.part == nullptr || gridDim.z == 1) && p.y_tma) {
            // The tile staged in the idle operand ring as four [128 tokens][32 rows]
            // boxes (one per TMEM lane quarter; a warp's 32 rows are one 128-byte
            // row of its box), then written by four tensor stores; rows past O and
            // tokens past T are clipped by the map.
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
        } else if (p.part == nullptr || gridDim.z == 1) {
            if (ok && col_ok) store_col(p.y + (size_t)(t0 + c0) * O + o);
        } else {
            // split-K: publish this split's partial sums; the last CTA of the
            // tile to arrive adds all splits in z order (deterministic)
            if (ok && col_ok) store_col(p.part + ((size_t)blockIdx.z * T + t0 + c0) * O + o);
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
            if (*last_flag && ok && col_ok) {
                __threadfence();
                // eight outputs at a time, the other splits' eight loads issued together
#pragma unroll
                for (int c = 0; c < 64; c += 8) {
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
                    for (int z = 0; z < (int)gridDim.z; ++z) {
                        float v[8];
                        if (z == (int)blockIdx.z) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[i] = yv[c + i];
                        } else {
                            const float *pz = p.part + ((size_t)z * T + t0 + c0 + c) * O + o;
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[i] = c + i < nt ? __ldcg(pz + (size_t)i * O) : 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) a[i] += v[i];
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) yv[c + i] = a[i];
                }
                store_col(p.y + (size_t)(t0 + c0) * O + o);
            }
        }
    } else if (warp == 0 || warp == SCALE_WARP_B) {
        // ------------------------------------------------------- scale warps --
        // Per super-block, for weight rows r and r + 64: the multiplier d (1
        // where d == 0) and the min-term operand row (-(dmin*m_j)/d, split
        // hi/lo); for tokens r and r + 64: the min-term operand row
        // (dx_j*ssum_j split hi/lo).  Slot sb % SSTG is rewritten once
        // super-block sb - SSTG's accumulator has been released: its
        // min-term MMAs completed before it was handed to the epilogue,
        // and the epilogue releases it after reading d.  The weight headers
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
                qa = min(127, max(-127, q8::round_quotient(h[c], d32, rd)));
                qb = min(127, max(-127, q8::round_quotient(h[c + 1], d32, rd)));
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
    if (warp == MMA_WARP) {
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
    CUtensorMap tmA, tmW, tmY;
    rc = make_tmap_2d(&tmA, xa, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K, 2ull * (uint64_t)T, (uint64_t)K * 2, BK,
                      BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MMQ_OK) return rc;
    rc = make_tmap_2d(&tmW, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)nsb * row_bytes, (uint64_t)O,
                      (uint64_t)nsb * row_bytes, row_bytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != MMQ_OK) return rc;
    // y by tensor stores ([T][O] f32, boxes of 32 rows x 128 tokens) when its row stride allows
    const bool y_tma = !h_xa && splits == 1 && (O % 4) == 0;
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
    prm.y_tma = y_tma ? 1 : 0;
    const dim3 grid((unsigned)((O + BN - 1) / BN), (unsigned)((T + BM - 1) / BM), (unsigned)splits);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (fmt == kQ5K)
        mmq_q4K_sb_kernel<kQ5K, false><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ5K>::kDynSmem, cs>>>(tmA, tmW, tmY, prm);
    else if (h_xa)
        mmq_q4K_sb_kernel<kQ4K, true><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ4K>::kDynSmem, cs>>>(tmA, tmW, tmY, prm);
    else
        mmq_q4K_sb_kernel<kQ4K, false><<<grid, q4s::NTHREADS, q4s::SbLayout<kQ4K>::kDynSmem, cs>>>(tmA, tmW, tmY, prm);
    return launch_status();
}

}  // namespace
}  // namespace mmq
