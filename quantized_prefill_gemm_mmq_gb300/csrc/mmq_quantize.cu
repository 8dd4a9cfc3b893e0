// mmq_quantize.cu -- q8_1 quantisation of f32 activations.
//
// Per token t and 32-element block b ("31 . r28 -- Direction-A raw-nibble NB
// kernel", 3.2: q8_1 blocks of int8 values with an (f16 d | int16 ssum)
// pair; "19 . r14 -- B fragments via ldmatrix", 3.2(d) for the packing):
//   amax = max|x|, d32 = amax/127, q = clamp(round_half_away(x/d32), +-127),
//   ssum = sum q, stored d = f16_rne(d32); all-zero block -> 0, 0, 0.
// d32 is an IEEE round-to-nearest division (__fdiv_rn), and every quotient
// x/d32 is rounded exactly as its IEEE division would be (q8::round_quotient
// in mmq_q8_1.cuh, shared with every other q8_1 writer), so the result does
// not depend on fast-math flags.
//
// Optional outputs: qs (int8 values), xh (the same values as f16, the integer
// operand form) and xa (the dequantised activation f32(d16)*q as an exact
// pair of f16 planes hi + lo: every such value is a multiple of 2^-24 with at
// most 18 significant bits, so hi = f16(v) and lo = f16(v - hi) are both
// exact and hi + lo == v).
//
// Layout: four threads own one 32-block, eight consecutive floats each (two
// 16-byte loads issued together); the block's amax and ssum are reduced
// across the four lanes with shuffles (q8::block4).  The kernel is a
// grid-stride loop over all (t, b) blocks, a warp taking eight consecutive
// blocks per iteration (read 4 B, write up to 5.125 B per element).
#include <cuda_fp16.h>

#include "mmq_host.h"
#include "mmq_q8_1.cuh"

namespace mmq {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerWarp = 8;

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

__global__ void __launch_bounds__(kThreads) quantize_q8_1_kernel(
    const float *__restrict__ x, int64_t ldx, int T, int K, int8_t *__restrict__ qs,
    uint32_t *__restrict__ ds, uint16_t *__restrict__ xh, uint16_t *__restrict__ xa)
{
    const int nb = K >> 5;                                   // 32-blocks per token
    const int64_t nblocks = (int64_t)T * nb;
    const int lane = threadIdx.x & 31;
    const int sub = lane & 3;                                 // lane within the block's 4
    // warp-uniform loop: a warp covers kBlocksPerWarp consecutive blocks per
    // iteration, so every lane reaches every shuffle; lanes past the end only
    // skip loads and stores
    const int64_t warp_first = (((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5) * kBlocksPerWarp;
    const int64_t warp_step = ((int64_t)gridDim.x * kThreads >> 5) * kBlocksPerWarp;
    // this lane's block blk = (token t, block b), advanced by warp_step blocks per
    // iteration without a division
    int64_t blk = warp_first + (lane >> 2);
    int t = (int)(blk / nb), b = (int)(blk - (int64_t)t * nb);
    const int step_t = (int)(warp_step / nb), step_b = (int)(warp_step - (int64_t)step_t * nb);
    for (int64_t base = warp_first; base < nblocks; base += warp_step) {
        const bool live = blk < nblocks;
        const int k = b * 32 + sub * 8;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (live) {
            const float4 *src = reinterpret_cast<const float4 *>(x + (int64_t)t * ldx + k);
            v0 = __ldg(src);
            v1 = __ldg(src + 1);
        }
        const q8::Oct qd = q8::block4(v0, v1);
        const int64_t e = (int64_t)t * K + k, blk_here = blk;
        blk += warp_step;
        t += step_t;
        b += step_b;
        if (b >= nb) {
            b -= nb;
            ++t;
        }
        if (!live) continue;
        if (qs) {
            uint32_t w[2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
                w[h] = (uint32_t)(uint8_t)qd.q[4 * h] | ((uint32_t)(uint8_t)qd.q[4 * h + 1] << 8) |
                       ((uint32_t)(uint8_t)qd.q[4 * h + 2] << 16) | ((uint32_t)(uint8_t)qd.q[4 * h + 3] << 24);
            *reinterpret_cast<uint2 *>(qs + e) = make_uint2(w[0], w[1]);
        }
        if (xh) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = h2u(__halves2half2(__int2half_rn(qd.q[2 * i]), __int2half_rn(qd.q[2 * i + 1])));
            *reinterpret_cast<uint4 *>(xh + e) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const __half dh = qd.d16;
        if (xa) {
            // v = f32(d16) * q is exact in f32; hi = f16(v), lo = f16(v - hi), both exact
            const float df = __half2float(dh);
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 v = make_float2(df * (float)qd.q[2 * i], df * (float)qd.q[2 * i + 1]);
                const __half2 hv = __float22half2_rn(v);
                const float2 bv = __half22float2(hv);
                hw[i] = h2u(hv);
                lw[i] = h2u(__float22half2_rn(make_float2(v.x - bv.x, v.y - bv.y)));
            }
            *reinterpret_cast<uint4 *>(xa + e) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(xa + (int64_t)T * K + e) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        if (sub == 0) ds[blk_here] = q8::scale_word(dh, qd.ssum);
    }
}

}  // namespace
}  // namespace mmq

extern "C" int mmq_quantize_q8_1(const float *x, int64_t ldx, int T, int K, int8_t *qs, uint32_t *ds,
                                 uint16_t *xh, uint16_t *xa, mmq_stream_t stream)
{
    using namespace mmq;
    if (T < 0 || K < 32 || K > (1 << 20) || (K & 31) || ldx < K) return MMQ_ERR_SHAPE;
    if (T == 0) return MMQ_OK;
    if (!x || !ds || (!qs && !xh && !xa)) return MMQ_ERR_NULL;
    if (!aligned16(x) || (ldx & 3) || !aligned16(ds) || (qs && !aligned16(qs)) || (xh && !aligned16(xh)) ||
        (xa && !aligned16(xa)))
        return MMQ_ERR_ALIGN;
    const int a = check_arch();
    if (a != MMQ_OK) return a;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t threads = ((int64_t)T * (K / 32) + kBlocksPerWarp - 1) / kBlocksPerWarp * 32;
    int64_t grid = (threads + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;   // 8 resident blocks per SM
    if (grid > cap) grid = cap;
    quantize_q8_1_kernel<<<(unsigned)grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, ldx, T, K, qs, ds, xh, xa);
    return launch_status();
}
