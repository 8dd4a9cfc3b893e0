// mmq_q8_1.cuh -- the q8_1 quantisation of one 32-element block, shared by
// every kernel that writes q8_1 (mmq_quantize_q8_1, the chained FFN's SwiGLU
// epilogue, the decode GEMV's built-in quantisation), so that all of them
// produce the same bits.
//
// Per 32-element block ("31 . r28 -- Direction-A raw-nibble NB kernel", 3.2:
// q8_1 blocks of int8 values with an (f16 d | int16 ssum) pair):
//   amax = max|x|, d32 = amax/127 (IEEE division), q = clamp(round_half_away
//   (x/d32), +-127) with every quotient rounded as its IEEE division would
//   be, ssum = sum q, stored d = f16_rne(d32); an all-zero block -> 0, 0, 0.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace mmq {
namespace q8 {

// round_half_away(x / d), the quotient rounded to f32 as IEEE division does,
// without the division where the result cannot depend on it.  With
// r = fl(1/d), z = fl(x * r) differs from the exact quotient y by at most
// |y| * 2^-23 (two roundings), and the correctly rounded fl(y) from y by at
// most |y| * 2^-24, so |z - fl(y)| < |y| * 2^-22 <= 3.1e-5 for |y| <= 127.5.
// Unless z lies within 2^-14 (> that bound) of a half-integer, fl(y) is on
// the same side of it and both round to the same integer; near a half-integer
// (and when r is not a finite normal number) the quotient is taken exactly.
__device__ __forceinline__ int round_quotient(float x, float d, float r)
{
    const float z = x * r;
    const float a = fabsf(z);
    if (r < 1e30f && a < 128.0f && fabsf(a - floorf(a) - 0.5f) > 0x1p-14f) return (int)roundf(z);
    return (int)roundf(__fdiv_rn(x, d));
}

// One 32-block held by eight consecutive lanes (an aligned group of 8 within
// the warp), four values each.  Every lane of the warp must call it (the
// reductions shuffle across the group); q0..q3 are this lane's codes, d16
// and ssum the block's scale word fields (the same in all eight lanes).
struct Quad {
    int q0, q1, q2, q3;
    __half d16;
    int ssum;
};

__device__ __forceinline__ Quad block8(float4 v)
{
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m, 8));
    Quad o;
    o.q0 = o.q1 = o.q2 = o.q3 = 0;
    float d32 = 0.0f;
    if (amax != 0.0f) {
        d32 = __fdiv_rn(amax, 127.0f);
        const float r = __frcp_rn(d32);
        o.q0 = min(127, max(-127, round_quotient(v.x, d32, r)));
        o.q1 = min(127, max(-127, round_quotient(v.y, d32, r)));
        o.q2 = min(127, max(-127, round_quotient(v.z, d32, r)));
        o.q3 = min(127, max(-127, round_quotient(v.w, d32, r)));
    }
    int ssum = o.q0 + o.q1 + o.q2 + o.q3;
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, m, 8);
    o.ssum = ssum;
    o.d16 = __float2half_rn(d32);
    return o;
}

// The same block held by four consecutive lanes (an aligned group of 4),
// eight values each (a and b: values 0-3 and 4-7 of this lane's eight).
// Every lane of the warp must call it; q[] are this lane's codes.
struct Oct {
    int q[8];
    __half d16;
    int ssum;
};

__device__ __forceinline__ Oct block4(float4 a, float4 b)
{
    float amax = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                       fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1, 4));
    Oct o;
#pragma unroll
    for (int i = 0; i < 8; ++i) o.q[i] = 0;
    float d32 = 0.0f;
    if (amax != 0.0f) {
        d32 = __fdiv_rn(amax, 127.0f);
        const float r = __frcp_rn(d32);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) o.q[i] = min(127, max(-127, round_quotient(v[i], d32, r)));
    }
    int ssum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) ssum += o.q[i];
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 2, 4);
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1, 4);
    o.ssum = ssum;
    o.d16 = __float2half_rn(d32);
    return o;
}

// the scale word: low 16 bits f16 d, high 16 bits int16 ssum
__device__ __forceinline__ uint32_t scale_word(__half d16, int ssum)
{
    return (uint32_t)__half_as_ushort(d16) | ((uint32_t)(uint16_t)(int16_t)ssum << 16);
}

}  // namespace q8
}  // namespace mmq
