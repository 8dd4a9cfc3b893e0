// mmq_kquant.cuh -- k-quant field decoders shared by the kernels of libmmq.
#pragma once

#include <cstdint>

namespace mmq {
namespace kq {

// q4_K / q5_K: the 6-bit scale (sc) and min (mm) of sub-block j (0..7) from
// the 12 packed scale bytes held in three words s0 (bytes 0-3), s1 (4-7),
// s2 (8-11): sub-blocks 0-3 take the low 6 bits of bytes j and 4 + j;
// sub-blocks 4-7 take a nibble of byte 8 + (j - 4) for their low 4 bits and
// the top 2 bits of bytes j - 4 and j for their high 2 bits (the GGUF
// k-quant packing).
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

}  // namespace kq
}  // namespace mmq
