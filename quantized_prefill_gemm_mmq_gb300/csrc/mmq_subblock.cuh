// mmq_subblock.cuh -- the per-sub-block GEMMs: the pages' method form, every
// 32-weight (q6_K: 16-weight) sub-block's exact integer dot formed by the
// tensor core in its own accumulator and folded in f32
// (mmq_gemm_q4K_subblock, mmq_gemm_q5K_subblock, mmq_gemm_q6K_subblock,
// mmq_gemm_q8_0, the mmq_debug_subdots_* diagnostics), and their launcher.
//
// Design of the first-generation pipeline (mmq_gemm_kernel):
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
#pragma once

namespace mmq {
namespace {

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

using kq::q4K_scale_min;   // the 6-bit scale and min of sub-block j (mmq_kquant.cuh)

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
