// mmq_host.cu -- status codes, architecture check, TMA tensor-map encoding
// (through the runtime's driver entry point, so the library does not link
// libcuda directly) and the device status word.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mmq_host.h"

namespace mmq {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDevices = 64;
int g_arch_ok[kMaxDevices];   // 0 unknown, 1 ok, -1 wrong arch
std::mutex g_arch_mu;

}  // namespace

int check_arch()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_ARCH;
    }
    if (dev < 0 || dev >= kMaxDevices) return MMQ_ERR_DEVICE;
    {
        std::lock_guard<std::mutex> lk(g_arch_mu);
        if (g_arch_ok[dev] == 0) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
                cudaGetLastError();
                return MMQ_ERR_ARCH;
            }
            g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        }
        return g_arch_ok[dev] == 1 ? MMQ_OK : MMQ_ERR_ARCH;
    }
}

int launch_status()
{
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return MMQ_OK;
    if (std::getenv("MMQ_DEBUG")) std::fprintf(stderr, "libmmq: launch failed: %s\n", cudaGetErrorString(e));
    return MMQ_ERR_LAUNCH;
}

int make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t inner,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return MMQ_ERR_DRIVER;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && std::getenv("MMQ_DEBUG"))
        std::fprintf(stderr, "libmmq: cuTensorMapEncodeTiled(2d) failed: %d\n", (int)r);
    return r == CUDA_SUCCESS ? MMQ_OK : MMQ_ERR_DRIVER;
}

int make_tmap_4d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, const uint64_t (&dims)[4],
                 const uint64_t (&strides_bytes)[3], const uint32_t (&box)[4], CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return MMQ_ERR_DRIVER;
    const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    const cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, dtype, 4, const_cast<void *>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && std::getenv("MMQ_DEBUG"))
        std::fprintf(stderr, "libmmq: cuTensorMapEncodeTiled(4d) failed: %d\n", (int)r);
    return r == CUDA_SUCCESS ? MMQ_OK : MMQ_ERR_DRIVER;
}

}  // namespace mmq

extern "C" int mmq_version(void) { return 8; }

extern "C" const char *mmq_status_str(int status)
{
    switch (status) {
    case MMQ_OK: return "ok";
    case MMQ_ERR_SHAPE: return "shape out of range";
    case MMQ_ERR_ALIGN: return "pointer or leading dimension not 16-byte aligned";
    case MMQ_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case MMQ_ERR_LAUNCH: return "kernel launch refused by the CUDA runtime";
    case MMQ_ERR_TIMEOUT: return "a kernel pipeline wait timed out; output invalid";
    case MMQ_ERR_NULL: return "required pointer is NULL";
    case MMQ_ERR_DRIVER: return "driver could not encode a TMA tensor map";
    case MMQ_ERR_CUDA: return "CUDA error pending on the stream";
    case MMQ_ERR_SCRATCH: return "split-K scratch needed exceeds the library's static scratch (4 Mi f32 partial sums, 8192 tiles)";
    case MMQ_ERR_DEVICE: return "current device index is beyond the library's per-device tables (64 devices)";
    default: return "unknown status";
    }
}
