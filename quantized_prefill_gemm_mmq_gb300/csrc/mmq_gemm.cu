// mmq_gemm.cu -- the one translation unit of libmmq's GEMM kernels and their
// C entry points: q4_K / q5_K / q6_K / q8_0 x q8_1 prefill GEMMs on sm_103a
// tensor cores, Y[t][o] = sum_k W[o][k] X[t][k] in the block-wise integer form
// of the "minfer" pages ("31 . r28 -- Direction-A raw-nibble NB kernel", 2.3).
//
// Kernel families, one file each (all compiled here, so that every kernel
// reports into the one device status word that mmq_check_status reads):
//   mmq_common.cuh     tile shapes, format descriptions, parameters, helpers
//   mmq_subblock.cuh   the per-sub-block method form and its diagnostics
//   mmq_prod_q4K.cuh   production q4_K / q5_K GEMM, split-K, SwiGLU chain
//   mmq_prod_q6K.cuh   production q6_K GEMM
//   mmq_small.cuh      few-token q4_K GEMMs (int8 warp MMA, weight-stationary)
//   mmq_gemv.cuh,
//   mmq_gemv_q6.cuh    decode-shaped q4_K / q6_K products
// Every pipeline wait is bounded: after a time limit the kernel records
// MMQ_ERR_TIMEOUT in the device status word, all roles stop, in-flight work
// drains and tensor memory is freed.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "mmq_dev.cuh"
#include "mmq_host.h"

#include "mmq_common.cuh"
#include "mmq_kquant.cuh"
#include "mmq_q8_1.cuh"
#include "mmq_pdl.cuh"
#include "mmq_subblock.cuh"
#include "mmq_prod_q4K.cuh"
#include "mmq_prod_q6K.cuh"
#include "mmq_small.cuh"

extern "C" int mmq_gemm_q4K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
}

extern "C" int mmq_gemm_q5K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream, nullptr, nullptr, nullptr,
                              mmq::kQ5K);
}

extern "C" int mmq_gemm_q4K_small_imma(const void *w, const int8_t *qs, const uint32_t *ds, float *y, int T, int O,
                                       int K, mmq_stream_t stream)
{
    return mmq::launch_q4K_small(w, qs, ds, y, T, O, K, stream);
}

extern "C" int mmq_gemm_q4K_small(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O,
                                  int K, mmq_stream_t stream)
{
    return mmq::launch_q4K_wt(w, xa, ds, y, T, O, K, stream);
}

extern "C" int mmq_splitk_sizes(int T, int O, int K, int ksplit, int64_t *part_floats, int64_t *counters)
{
    if (T < 1 || O < 1 || K < 256 || K > (1 << 20) || (K & 255) || ksplit < 1) return MMQ_ERR_SHAPE;
    const int nsb = K / 256;
    const int sbps = (nsb + std::min(ksplit, nsb) - 1) / std::min(ksplit, nsb);
    const int splits = (nsb + sbps - 1) / sbps;
    if (part_floats) *part_floats = splits > 1 ? (int64_t)splits * T * O : 0;
    if (counters) *counters = (int64_t)((O + mmq::BN - 1) / mmq::BN) * ((T + mmq::BM - 1) / mmq::BM);
    return MMQ_OK;
}

extern "C" int mmq_gemm_q4K_splitk(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O,
                                   int K, int ksplit, float *part, int *counters, mmq_stream_t stream)
{
    if (ksplit < 1) return MMQ_ERR_SHAPE;
    if (ksplit > 1 && (!part || !counters)) return MMQ_ERR_NULL;
    return mmq::launch_q4K_sb(w, xa, ds, y, T, O, K, ksplit, part, counters, stream);
}

extern "C" int mmq_gemm_q4K_swiglu(const void *w_gu, const uint16_t *xa, const uint32_t *ds, uint16_t *h_xa,
                                   uint32_t *h_ds, int8_t *h_qs, int T, int F, int K, mmq_stream_t stream)
{
    if (F < 64 || F % 64 != 0 || F > (1 << 20)) return MMQ_ERR_SHAPE;
    if (!h_xa || !h_ds) return MMQ_ERR_NULL;
    return mmq::launch_q4K_sb(w_gu, xa, ds, nullptr, T, 2 * F, K, 1, nullptr, nullptr, stream, h_xa, h_ds, h_qs);
}

// Scratch of mmq_gemm_q4K_splitk_static: partial sums and tile counters in
// the library's own device memory (zero-initialised at module load; every
// completed launch leaves the counters at zero).
constexpr int64_t kStaticPartFloats = (int64_t)1 << 22;   // 16 MiB of f32 partial sums
constexpr int64_t kStaticCounters = 8192;                 // output tiles
static __device__ __align__(256) float g_splitk_part[kStaticPartFloats];
static __device__ __align__(256) int g_splitk_cnt[kStaticCounters];

extern "C" int mmq_gemm_q4K_splitk_static(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T,
                                          int O, int K, int ksplit, mmq_stream_t stream)
{
    if (T == 0) return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
    int64_t part_floats = 0, tiles = 0;
    const int rc = mmq_splitk_sizes(T, O, K, ksplit, &part_floats, &tiles);
    if (rc != MMQ_OK) return rc;
    // one split (ksplit == 1, or a single super-block per row) uses no scratch at all
    if (part_floats == 0) return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, 1, nullptr, nullptr, stream);
    if (part_floats > kStaticPartFloats || tiles > kStaticCounters) return MMQ_ERR_SCRATCH;
    // device addresses of the two arrays, looked up once per device (with that
    // device current) under a lock, so that concurrent first calls from several
    // host threads do not race on the table
    static float *part[64];
    static int *cnt[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= 64) return MMQ_ERR_DEVICE;
    float *pp = nullptr;
    int *cc = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!part[dev] || !cnt[dev]) {
            void *a = nullptr, *b = nullptr;
            if (cudaGetSymbolAddress(&a, g_splitk_part) != cudaSuccess ||
                cudaGetSymbolAddress(&b, g_splitk_cnt) != cudaSuccess)
                return mmq::launch_status();
            part[dev] = static_cast<float *>(a);
            cnt[dev] = static_cast<int *>(b);
        }
        pp = part[dev];
        cc = cnt[dev];
    }
    return mmq_gemm_q4K_splitk(w, xa, ds, y, T, O, K, ksplit, pp, cc, stream);
}

extern "C" int mmq_gemm_q4K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ4K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_gemm_q6K(const void *w, const uint16_t *xa, const uint32_t *ds, float *y, int T, int O, int K,
                            mmq_stream_t stream)
{
    return mmq::launch_q6K_sb(w, xa, ds, y, T, O, K, stream);
}

extern "C" int mmq_gemm_q6K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ6K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q4K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ4K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_gemm_q5K_subblock(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O,
                                     int K, mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ5K, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_gemm_q8_0(const void *w, const uint16_t *xh, const uint32_t *ds, float *y, int T, int O, int K,
                             mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ8_0, mmq::kFold>(w, xh, ds, y, nullptr, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q5K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ5K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q8_0(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                      mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ8_0, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_subdots_q6K(const void *w, const uint16_t *xh, int32_t *out, int T, int O, int K,
                                     mmq_stream_t stream)
{
    return mmq::launch<mmq::kQ6K, mmq::kSubdots>(w, xh, nullptr, nullptr, out, T, O, K, stream);
}

extern "C" int mmq_debug_fault_inject(int mode, int wait_limit_us)
{
    if (mode < 0 || mode > 1) return MMQ_ERR_SHAPE;
    const unsigned long long lim =
        wait_limit_us > 0 ? (unsigned long long)wait_limit_us * 1000ull : mmq::kWaitLimitNs;
    if (cudaMemcpyToSymbol(mmq::g_inject, &mode, sizeof(mode)) != cudaSuccess ||
        cudaMemcpyToSymbol(mmq::g_wait_limit_ns, &lim, sizeof(lim)) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return MMQ_OK;
}

// extra detail of the last failure reported by mmq_check_status (host side)
static int g_last_failure[4];

extern "C" int mmq_check_status(mmq_stream_t stream, int *detail)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        if (detail) detail[0] = detail[1] = detail[2] = detail[3] = 0;
        return MMQ_ERR_CUDA;
    }
    int h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(h, mmq::g_status, sizeof(h)) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    if (h[0] != 0) {
        const int zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        cudaMemcpyToSymbol(mmq::g_status, zero, sizeof(zero));
        for (int i = 0; i < 4; ++i) g_last_failure[i] = h[4 + i];
    }
    if (detail)
        for (int i = 0; i < 4; ++i) detail[i] = h[i];
    return h[0];
}

extern "C" int mmq_last_failure_info(int *info)
{
    if (!info) return MMQ_ERR_NULL;
    for (int i = 0; i < 4; ++i) info[i] = g_last_failure[i];
    return MMQ_OK;
}

// decode-shaped q4_K and q6_K products (mmq_gemv_q4K, mmq_gemv_q6K): in this unit for their bounded waits
// and the status word
#include "mmq_gemv.cuh"
#include "mmq_gemv_q6.cuh"
#include "mmq_decode.cuh"
