// mmq_decode.cuh -- decode-shaped q4_K product for 1 <= T <= 4 tokens on the
// SIMT cores, with the q8_1 quantisation of the f32 tokens built in
// (mmq_gemv_q4K_f32).  Included by mmq_gemm.cu (its bounded waits report into
// the library's status word).
//
// The pages' per-sub-block form ("31 . r28 -- Direction-A raw-nibble NB
// kernel", 2.3 "The numerics contract"): for every 32-weight sub-block b the
// exact integer dot C_b of the unsigned 4-bit quants with the int8
// activations (__dp4a, int32), folded in f32 as
//     y += (dx*(d*sc_b))*C_b + (dx*ssum_b)*(-(dmin*m_b)).
// At T <= 4 the cost is reading W from HBM once, so the kernel is laid out
// for bytes in flight: every warp owns a ring of two chunks of up to 32 q4_K
// super-blocks of one row (4608 bytes), refilled by one bulk copy per chunk as
// soon as the warp has read it, and walks its rows (dealt round-robin over
// the CTAs, so every SM streams the same share of W) chunk after chunk.  In a
// chunk, lane l takes super-blocks l % 8, l % 8 + 8, ... and sub-block pair
// p = l / 8 (the 32 quant bytes whose low and high nibbles are sub-blocks 2p
// and 2p + 1), so both dots are whole in one lane: 16 __dp4a per token and
// super-block, no cross-lane sums.  Measured on this GB300 at T = 1 (us at
// 4096 x 4096 / 11008 x 4096 / 4096 x 22016, chunk super-blocks x chunks in
// flight): 8 x 4 7.4 / 18.1 / 17.2; 4 x 8 10.6 / 26.0 / 29.7; 16 x 4
// 5.5 / 14.2 / 15.1; 16 x 2 7.4 / 15.8 / 15.3; 32 x 2 5.4 / 12.9 / 14.1 --
// the cost per bulk copy, more than the bytes in flight, sets the pace.
// Eight times fewer copies through a CTA-shared ring of four 4-D TMA boxes
// (16 super-blocks of a CTA's eight consecutive rows per box, one row per
// warp, a slot refilled once all eight warps have read it) measured slower:
// 5.8 / 15.0 us, the 32-layer decode step 1.75 ms instead of 1.56.
//
// Built-in quantisation: every CTA first quantises the T tokens into shared
// memory with the same arithmetic as mmq_quantize_q8_1 (mmq_q8_1.cuh), so the
// codes, scales and sums are bit-identical to that kernel's and no separate
// quantise launch is needed.  The first chunks of W are requested before the
// previous kernel in the stream has completed (programmatic dependent
// launch); x is read and y written only after it has.
#pragma once

namespace mmq {
namespace {
namespace dec {

constexpr int KID = 14;                    // kernel id in the status word
constexpr int WARPS = 8;
constexpr int NTHREADS = WARPS * 32;
constexpr int CH = 32;                     // super-blocks per chunk (lane % 8 takes every eighth)
constexpr int NCH = 2;                     // chunks in flight per warp
constexpr uint32_t CHUNK_BYTES = CH * 144;
constexpr uint32_t WARP_RING = NCH * CHUNK_BYTES;
constexpr int MAXT = 4;
constexpr int MAXK = 32768;
// the quantised tokens: 272 bytes per 256-value super-block (16 bytes of
// padding), so that the eight super-blocks one load instruction touches fall
// in eight different bank groups
constexpr int XSB = 272;
// shared memory: rings [WARPS], barriers [WARPS][NCH], abort flag, then
// int8 codes [NT][K/256][XSB] and scale words [NT][K/32]
constexpr uint32_t oBar = WARPS * WARP_RING;
constexpr uint32_t oMisc = oBar + WARPS * NCH * 8;
constexpr uint32_t oX = oMisc + 16;
__host__ __device__ constexpr size_t smem_bytes(int nt, int K)
{
    return oX + (size_t)nt * (K / 256) * XSB + (size_t)nt * (K / 32) * 4;
}

// q6_K: 210-byte super-blocks are only 2-byte aligned, so a chunk is copied
// as the 16-byte-aligned window around it (up to 15 bytes before and after;
// the bytes past the end of W are loaded one by one instead) into a slot with
// 32 bytes of slack, and read back with funnel shifts.
constexpr int CH6 = 16;
constexpr int NCH6 = 2;
constexpr uint32_t SLOT6 = CH6 * 210 + 32;
constexpr uint32_t WARP_RING6 = NCH6 * SLOT6;
constexpr uint32_t oBar6 = WARPS * WARP_RING6;
constexpr uint32_t oMisc6 = oBar6 + WARPS * NCH6 * 8;
constexpr uint32_t oX6 = oMisc6 + 16;
static_assert(SLOT6 % 16 == 0 && oX6 % 16 == 0, "q6_K decode layout alignment");
__host__ __device__ constexpr size_t smem_bytes6(int nt, int K)
{
    return oX6 + (size_t)nt * (K / 256) * XSB + (size_t)nt * (K / 32) * 4;
}

}  // namespace dec

// q8_1 of the NT tokens x[t][0..K) (tokens >= T as zeros) into shared memory
// (codes [NT][K/256][XSB], scale words [NT][K/32]) by all NTHREADS threads,
// eight lanes per 32-block, with the arithmetic of mmq_quantize_q8_1; every
// lane of a warp runs the same trip count (block8 shuffles), and the loads of
// G blocks are issued before any of them is quantised.  Ends with a CTA barrier.
template <int NT>
__device__ __forceinline__ void quantize_tokens(const float *__restrict__ x, int64_t ldx, int T, int K,
                                                int8_t *xq, uint32_t *xd)
{
    using namespace dec;
    constexpr int G = 4, PER = NTHREADS / 8;
    const int nsb = K >> 8, nb = K >> 5;
    const int total = NT * nb, sub = threadIdx.x & 7;
    for (int base = 0; base < total; base += G * PER) {
        float4 v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int blk = base + g * PER + ((int)threadIdx.x >> 3);
            const int t = blk / nb, b = blk - t * nb;
            v[g] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (blk < total && t < T)
                // L2 loads, not the read-only path: under programmatic dependent launch this
                // kernel starts before x (the previous kernel's output) is written
                v[g] = __ldcg(reinterpret_cast<const float4 *>(x + (int64_t)t * ldx + 32 * b + 4 * sub));
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int blk = base + g * PER + ((int)threadIdx.x >> 3);
            const q8::Quad qd = q8::block8(v[g]);
            if (blk < total) {
                const int t = blk / nb, b = blk - t * nb;
                const int e = 32 * b + 4 * sub;   // value index within the token
                *reinterpret_cast<uint32_t *>(xq + ((size_t)t * nsb + (e >> 8)) * XSB + (e & 255)) =
                    (uint32_t)(uint8_t)qd.q0 | ((uint32_t)(uint8_t)qd.q1 << 8) | ((uint32_t)(uint8_t)qd.q2 << 16) |
                    ((uint32_t)(uint8_t)qd.q3 << 24);
                if (sub == 0) xd[t * nb + b] = q8::scale_word(qd.d16, qd.ssum);
            }
        }
    }
    __syncthreads();
}

template <int NT>
__global__ void __launch_bounds__(dec::NTHREADS) mmq_q4K_decode_kernel(const uint8_t *__restrict__ w,
                                                                       const float *__restrict__ x, int64_t ldx,
                                                                       float *__restrict__ y, int T, int O, int K)
{
    using namespace dec;
    extern __shared__ __align__(128) uint8_t dec_sm[];
    const uint32_t sbase = smem_u32(dec_sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K >> 8, nb = K >> 5;
    const int nch_row = (nsb + CH - 1) / CH;                 // chunks per row
    const int nwarps = (int)gridDim.x * WARPS;
    const int row0 = (int)blockIdx.x + (int)gridDim.x * warp;   // this warp's rows: row0, row0 + nwarps, ...
    const int nrows = row0 < O ? (O - 1 - row0) / nwarps + 1 : 0;
    const int nchunks = nrows * nch_row;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(dec_sm + oMisc);
    int8_t *xq = reinterpret_cast<int8_t *>(dec_sm + oX);                                // [NT][nsb][XSB]
    uint32_t *xd = reinterpret_cast<uint32_t *>(dec_sm + oX + (size_t)NT * nsb * XSB);    // [NT][nb]
    const uint32_t bar0 = sbase + oBar + warp * NCH * 8;

    if (threadIdx.x == 0) *abort_flag = 0u;
    if (lane == 0) {
        for (int s = 0; s < NCH; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    pdl_launch_dependents();

    // chunk c of this warp: row row0 + (c / nch_row) * nwarps, super-blocks
    // CH * (c % nch_row) .. (fewer in a row's last chunk); issued by lane 0
    auto issue = [&](int c) {
        const int r = row0 + (c / nch_row) * nwarps, k0 = (c % nch_row) * CH;
        const uint32_t n = (uint32_t)min(CH, nsb - k0) * 144u, slot = (uint32_t)(c % NCH);
        mbar_arrive_expect_tx(bar0 + 8 * slot, n);
        bulk_load(sbase + warp * WARP_RING + slot * CHUNK_BYTES, w + ((size_t)r * nsb + k0) * 144, n, bar0 + 8 * slot);
    };
    int issued = 0;   // chunks requested (lane 0)
    // W is never written by the kernel before this one (documented), so its
    // first chunks are requested before that kernel has completed
    if (lane == 0)
        for (; issued < NCH && issued < nchunks; ++issued) issue(issued);

    pdl_wait();   // x may be the previous kernel's output, y its input

    quantize_tokens<NT>(x, ldx, T, K, xq, xd);

    const int p = lane >> 3;   // sub-block pair
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        const int slot = c % NCH;
        ok = mbar_wait_warp(bar0 + 8 * slot, (uint32_t)((c / NCH) & 1), abort_flag, KID, SITE_U_STAGE);
        if (!ok) break;
        const int k0 = (c % nch_row) * CH;
#pragma unroll
        for (int sl = lane & 7; sl < CH; sl += 8) {
            if (sl >= nsb - k0) break;   // a row's last chunk may be short
            const uint8_t *blk = dec_sm + warp * WARP_RING + slot * CHUNK_BYTES + sl * 144;
            const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
            const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * p);   // quant bytes 32p .. 32p + 15
            const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * p);   // 32p + 16 .. 32p + 31
            const int sb = k0 + sl;
            int sc0, m0, sc1, m1;
            kq::q4K_scale_min(hd.y, hd.z, hd.w, 2 * p, sc0, m0);
            kq::q4K_scale_min(hd.y, hd.z, hd.w, 2 * p + 1, sc1, m1);
            const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
            const float dsc0 = d * (float)sc0, dmm0 = -(dmin * (float)m0);
            const float dsc1 = d * (float)sc1, dmm1 = -(dmin * (float)m1);
            const uint32_t M = 0x0F0F0F0Fu;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                // sub-block 2p: values 64p .. 64p + 31 of the super-block; 2p + 1: 64p + 32 ..
                const int8_t *xa = xq + ((size_t)t * nsb + sb) * XSB + 64 * p;
                const uint4 a0 = *reinterpret_cast<const uint4 *>(xa);
                const uint4 a1 = *reinterpret_cast<const uint4 *>(xa + 16);
                const uint4 a2 = *reinterpret_cast<const uint4 *>(xa + 32);
                const uint4 a3 = *reinterpret_cast<const uint4 *>(xa + 48);
                int c0 = __dp4a((int)(qa.x & M), (int)a0.x, 0);
                c0 = __dp4a((int)(qa.y & M), (int)a0.y, c0);
                c0 = __dp4a((int)(qa.z & M), (int)a0.z, c0);
                c0 = __dp4a((int)(qa.w & M), (int)a0.w, c0);
                c0 = __dp4a((int)(qb.x & M), (int)a1.x, c0);
                c0 = __dp4a((int)(qb.y & M), (int)a1.y, c0);
                c0 = __dp4a((int)(qb.z & M), (int)a1.z, c0);
                c0 = __dp4a((int)(qb.w & M), (int)a1.w, c0);
                int c1 = __dp4a((int)((qa.x >> 4) & M), (int)a2.x, 0);
                c1 = __dp4a((int)((qa.y >> 4) & M), (int)a2.y, c1);
                c1 = __dp4a((int)((qa.z >> 4) & M), (int)a2.z, c1);
                c1 = __dp4a((int)((qa.w >> 4) & M), (int)a2.w, c1);
                c1 = __dp4a((int)((qb.x >> 4) & M), (int)a3.x, c1);
                c1 = __dp4a((int)((qb.y >> 4) & M), (int)a3.y, c1);
                c1 = __dp4a((int)((qb.z >> 4) & M), (int)a3.z, c1);
                c1 = __dp4a((int)((qb.w >> 4) & M), (int)a3.w, c1);
                const uint32_t w0 = xd[t * nb + 8 * sb + 2 * p], w1 = xd[t * nb + 8 * sb + 2 * p + 1];
                const float dx0 = __half2float(__ushort_as_half((unsigned short)(w0 & 0xFFFFu)));
                const float dx1 = __half2float(__ushort_as_half((unsigned short)(w1 & 0xFFFFu)));
                const float s0 = (float)(int)(int16_t)(w0 >> 16), s1 = (float)(int)(int16_t)(w1 >> 16);
                acc[t] += (dx0 * dsc0) * (float)c0 + (dx0 * s0) * dmm0;
                acc[t] += (dx1 * dsc1) * (float)c1 + (dx1 * s1) * dmm1;
            }
        }
        // the slot's bytes have been read: order those reads before the copy that refills it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && issued < nchunks) issue(issued++);
        if ((c + 1) % nch_row == 0) {   // last chunk of a row: the warp's sum is the output
            const int r = row0 + (c / nch_row) * nwarps;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], m);
            }
            if (lane == 0) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    if (t < T) y[(size_t)t * O + r] = acc[t];
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
        }
    }
    if (!ok && lane == 0)   // let the copies in flight land before the CTA exits
        for (int i = max(0, issued - NCH); i < issued; ++i) wait_drain(bar0 + 8 * (i % NCH), (uint32_t)((i / NCH) & 1));
}

// 16 bytes at the (even) shared-memory offset o of buf, as four words
__device__ __forceinline__ uint4 ld16_even(const uint8_t *buf, uint32_t o)
{
    const uint32_t *w = reinterpret_cast<const uint32_t *>(buf + (o & ~3u));
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3];
    if ((o & 2u) == 0u) return make_uint4(w0, w1, w2, w3);
    const uint32_t w4 = w[4];
    return make_uint4(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16), __funnelshift_r(w2, w3, 16),
                      __funnelshift_r(w3, w4, 16));
}

// Decode-shaped q6_K product ("43 . r40 -- third resident block", 5: w =
// d*sc_u*(q-32) on 16-weight sub-blocks u; the pages' per-16 fold
// y += (dx*(d*sc_u))*C16_u with C16_u the exact integer dot of (q - 32) with
// the int8 activations), the q8_1 quantisation built in as for q4_K.  Per
// warp a ring of two chunks of up to 16 super-blocks of a row; in a chunk
// eight lanes share a super-block: lane j takes the 16 low-bit bytes
// L[32gq + 16hf ..] (gq = j / 2 % 2, hf = j % 2) of half h = j / 4 and the 16
// high-bit bytes H[16hf ..] of that half, i.e. the whole of sub-blocks
// u = 8h + 2gq + hf (low nibbles, bits 2gq..) and u + 4 (high nibbles,
// bits 2gq + 4..): 8 __dp4a per token and super-block, no cross-lane sums.
template <int NT>
__global__ void __launch_bounds__(dec::NTHREADS) mmq_q6K_decode_kernel(const uint8_t *__restrict__ w,
                                                                       const float *__restrict__ x, int64_t ldx,
                                                                       float *__restrict__ y, int T, int O, int K)
{
    using namespace dec;
    extern __shared__ __align__(128) uint8_t dec_sm[];
    const uint32_t sbase = smem_u32(dec_sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = K >> 8, nb = K >> 5;
    const int nch_row = (nsb + CH6 - 1) / CH6;
    const int nwarps = (int)gridDim.x * WARPS;
    const int row0 = (int)blockIdx.x + (int)gridDim.x * warp;
    const int nrows = row0 < O ? (O - 1 - row0) / nwarps + 1 : 0;
    const int nchunks = nrows * nch_row;
    const size_t total = (size_t)O * nsb * 210;   // bytes of W
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(dec_sm + oMisc6);
    int8_t *xq = reinterpret_cast<int8_t *>(dec_sm + oX6);
    uint32_t *xd = reinterpret_cast<uint32_t *>(dec_sm + oX6 + (size_t)NT * nsb * XSB);
    uint8_t *ring = dec_sm + warp * WARP_RING6;
    const uint32_t bar0 = sbase + oBar6 + warp * NCH6 * 8;

    if (threadIdx.x == 0) *abort_flag = 0u;
    if (lane == 0) {
        for (int s = 0; s < NCH6; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    pdl_launch_dependents();

    // chunk c: row row0 + (c / nch_row) * nwarps, super-blocks CH6 * (c % nch_row) ..;
    // bytes [B, E) of W land at slot offset B % 16 (issued by lane 0)
    auto issue = [&](int c) {
        const int r = row0 + (c / nch_row) * nwarps, k0 = (c % nch_row) * CH6;
        const size_t B = ((size_t)r * nsb + k0) * 210, E = B + (size_t)min(CH6, nsb - k0) * 210;
        const size_t Ba = B & ~(size_t)15, Ec = (E + 15) & ~(size_t)15;
        const uint32_t slot = (uint32_t)(c % NCH6), dst = sbase + warp * WARP_RING6 + slot * SLOT6;
        const size_t Eb = Ec <= total ? Ec : (E & ~(size_t)15);   // end of the bulk part
        mbar_arrive_expect_tx(bar0 + 8 * slot, (uint32_t)(Eb - Ba));
        bulk_load(dst, w + Ba, (uint32_t)(Eb - Ba), bar0 + 8 * slot);
        for (size_t b = Eb; b < E; ++b) ring[slot * SLOT6 + (b - Ba)] = w[b];   // last bytes of W
    };
    int issued = 0;
    if (lane == 0)
        for (; issued < NCH6 && issued < nchunks; ++issued) issue(issued);

    pdl_wait();

    quantize_tokens<NT>(x, ldx, T, K, xq, xd);

    const int j = lane & 7, h = j >> 2, gq = (j >> 1) & 1, hf = j & 1;
    const int u1 = 8 * h + 2 * gq + hf, u2 = u1 + 4;     // this lane's two sub-blocks
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        const int slot = c % NCH6;
        ok = mbar_wait_warp(bar0 + 8 * slot, (uint32_t)((c / NCH6) & 1), abort_flag, KID + 1, SITE_U_STAGE);
        if (!ok) break;
        __syncwarp();   // lane 0's byte stores of the buffer end, if any
        const int r = row0 + (c / nch_row) * nwarps, k0 = (c % nch_row) * CH6;
        const uint32_t off0 = (uint32_t)((((size_t)r * nsb + k0) * 210) & 15);
        const uint8_t *buf = ring + slot * SLOT6;
#pragma unroll
        for (int sl = lane >> 3; sl < CH6; sl += 4) {
            if (sl >= nsb - k0) break;
            const uint32_t ob = off0 + 210u * (uint32_t)sl;   // this super-block in the slot
            const uint4 L = ld16_even(buf, ob + 64 * h + 32 * gq + 16 * hf);
            const uint4 H = ld16_even(buf, ob + 128 + 32 * h + 16 * hf);
            const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(buf + ob + 208)));
            const float dsc1 = d * (float)(int)reinterpret_cast<const int8_t *>(buf + ob + 192)[u1];
            const float dsc2 = d * (float)(int)reinterpret_cast<const int8_t *>(buf + ob + 192)[u2];
            // q - 32 as signed bytes: low 4 bits from L, bits 4-5 from H
            auto vals = [&](uint32_t lw, uint32_t hw, int lsh, int hsh) {
                const uint32_t q = ((lw >> lsh) & 0x0F0F0F0Fu) | (((hw >> hsh) & 0x03030303u) << 4);
                return __vsub4(q, 0x20202020u);
            };
            const uint32_t v1[4] = {vals(L.x, H.x, 0, 2 * gq), vals(L.y, H.y, 0, 2 * gq), vals(L.z, H.z, 0, 2 * gq),
                                    vals(L.w, H.w, 0, 2 * gq)};
            const uint32_t v2[4] = {vals(L.x, H.x, 4, 2 * gq + 4), vals(L.y, H.y, 4, 2 * gq + 4),
                                    vals(L.z, H.z, 4, 2 * gq + 4), vals(L.w, H.w, 4, 2 * gq + 4)};
            const int sb = k0 + sl;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int8_t *xs = xq + ((size_t)t * nsb + sb) * XSB;
                const uint4 a1 = *reinterpret_cast<const uint4 *>(xs + 16 * u1);
                const uint4 a2 = *reinterpret_cast<const uint4 *>(xs + 16 * u2);
                int c1 = __dp4a((int)v1[0], (int)a1.x, 0);
                c1 = __dp4a((int)v1[1], (int)a1.y, c1);
                c1 = __dp4a((int)v1[2], (int)a1.z, c1);
                c1 = __dp4a((int)v1[3], (int)a1.w, c1);
                int c2 = __dp4a((int)v2[0], (int)a2.x, 0);
                c2 = __dp4a((int)v2[1], (int)a2.y, c2);
                c2 = __dp4a((int)v2[2], (int)a2.z, c2);
                c2 = __dp4a((int)v2[3], (int)a2.w, c2);
                const float dx1 = __half2float(__ushort_as_half((unsigned short)(xd[t * nb + 8 * sb + u1 / 2] & 0xFFFFu)));
                const float dx2 = __half2float(__ushort_as_half((unsigned short)(xd[t * nb + 8 * sb + u2 / 2] & 0xFFFFu)));
                acc[t] += (dx1 * dsc1) * (float)c1;
                acc[t] += (dx2 * dsc2) * (float)c2;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && issued < nchunks) issue(issued++);
        if ((c + 1) % nch_row == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], m);
            }
            if (lane == 0) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    if (t < T) y[(size_t)t * O + r] = acc[t];
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
        }
    }
    if (!ok && lane == 0)
        for (int i = max(0, issued - NCH6); i < issued; ++i) wait_drain(bar0 + 8 * (i % NCH6), (uint32_t)((i / NCH6) & 1));
}

template <int NT, bool Q6>
int launch_decode(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K, mmq_stream_t stream)
{
    const auto kernel = Q6 ? mmq_q6K_decode_kernel<NT> : mmq_q4K_decode_kernel<NT>;
    const size_t smem = Q6 ? dec::smem_bytes6(NT, K) : dec::smem_bytes(NT, K);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    static bool attr_done[64];
    if (!attr_done[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(Q6 ? dec::smem_bytes6(NT, dec::MAXK) : dec::smem_bytes(NT, dec::MAXK))) !=
            cudaSuccess)
            return launch_status();
        attr_done[dev] = true;
    }
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, dec::NTHREADS, smem) != cudaSuccess)
        return launch_status();
    if (per_sm < 1) per_sm = 1;
    // every CTA resident at once; rows dealt round-robin over them
    const long long want = ((long long)O + dec::WARPS - 1) / dec::WARPS;
    const long long cap = (long long)sms * per_sm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
    cfg.blockDim = dim3(dec::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may overlap the previous kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<const uint8_t *>(w), x, ldx, y, T, O, K) != cudaSuccess)
        return launch_status();
    return launch_status();
}

}  // namespace
}  // namespace mmq

namespace mmq {
namespace {

template <bool Q6>
int decode_entry(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K, mmq_stream_t stream)
{
    if (T < 0 || T > dec::MAXT || O < 1 || K < 256 || K > dec::MAXK || (K & 255) || ldx < K) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!w || !x || !y) return MMQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(x) || (ldx & 3) || !aligned16(y)) return MMQ_ERR_ALIGN;
    const int rc = check_arch();
    if (rc != MMQ_OK) return rc;
    if (T == 1) return launch_decode<1, Q6>(w, x, ldx, y, T, O, K, stream);
    if (T == 2) return launch_decode<2, Q6>(w, x, ldx, y, T, O, K, stream);
    return launch_decode<4, Q6>(w, x, ldx, y, T, O, K, stream);
}

}  // namespace
}  // namespace mmq

extern "C" int mmq_gemv_q4K_f32(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K,
                                mmq_stream_t stream)
{
    return mmq::decode_entry<false>(w, x, ldx, y, T, O, K, stream);
}

extern "C" int mmq_gemv_q6K_f32(const void *w, const float *x, int64_t ldx, float *y, int T, int O, int K,
                                mmq_stream_t stream)
{
    return mmq::decode_entry<true>(w, x, ldx, y, T, O, K, stream);
}
