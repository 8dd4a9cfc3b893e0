// mmq_small.cuh -- the few-token q4_K GEMMs: the int8 warp-MMA form
// (mmq_gemm_q4K_small_imma) and the weight-stationary tcgen05 form with
// cluster split-K (mmq_gemm_q4K_small), and their launchers.
#pragma once

namespace mmq {
namespace {

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

}  // namespace
}  // namespace mmq
