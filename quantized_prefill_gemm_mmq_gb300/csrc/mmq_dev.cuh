// mmq_dev.cuh -- sm_103a device primitives used by the MMQ kernels:
// mbarriers with bounded waits, TMA tensor loads, tcgen05 (UMMA) issue,
// TMEM allocation and loads, and the library's device status word.
//
// All PTX here is hand-written from the public PTX ISA descriptions of
// mbarrier, cp.async.bulk.tensor and tcgen05.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mmq {

// ------------------------------------------------------------ status word --
// g_status[0] = first error code, [1] = kernel id, [2] = wait site,
// [3] = linear block index, [4] = time waited (us), [5] = polls,
// [6] = phase parity waited for, [7] = the barrier's shared-memory address.
// One copy per translation unit (internal linkage); the GEMM translation
// unit owns the one mmq_check_status reads.
static __device__ int g_status[8];

constexpr int kStatusTimeout = -5;            // == MMQ_ERR_TIMEOUT
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait (the default)

// Test-only knobs (mmq_debug_fault_inject): the time a pipeline wait may
// take before it gives up, and a mode in which a kernel withholds one copy so
// that a wait runs out (the production q4_K kernel skips the raw weight copy
// of its second super-block).  One copy per translation unit, like g_status.
static __device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;
static __device__ int g_inject;

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(int code, int kernel_id, int site, int waited_us = 0, int polls = 0,
                                             int parity = 0, int bar = 0)
{
    if (atomicCAS(&g_status[0], 0, code) == 0) {
        g_status[1] = kernel_id;
        g_status[2] = site;
        g_status[3] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        g_status[4] = waited_us;
        g_status[5] = polls;
        g_status[6] = parity;
        g_status[7] = bar;
    }
}

// ------------------------------------------------------------- addresses --
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    // make the initialised barriers visible to the async (TMA / tensor core) proxy
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware for up to hint_ns
// until the phase completes (it is woken by the completion), so that waiting
// warps do not take issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Longest single hardware sleep of a wait.  Every try_wait of mbar_wait
// passes this explicit hint, the first one included: measured on the
// production q4_K GEMM (T = 512, K = 4096 / 11008), a first try_wait
// without a hint (system-dependent suspend time) followed by 20 us hints
// made the kernel 2.5 % / 6 % slower than 100 ns hints, and any hint from
// 20 ns to 2 us gave the same times within 2 %.
constexpr uint32_t kWaitSleepNs = 100;

constexpr uint64_t kPollCreditNs = 1000000;    // most waiting time one poll may add (1 ms)

// Wait for the phase with the given parity to complete.  Gives up (and
// returns false) when *abort is set by another role, or after g_wait_limit_ns
// (2 s unless a test lowered it) of waiting, in which case it records MMQ_ERR_TIMEOUT and raises *abort
// itself.  The time waited is the sum of the global timer's steps between
// polls, each counted only if positive and at most kPollCreditNs, so that an
// adjustment of the global timer (backwards or a jump forwards) cannot end a
// wait on its own.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                          int kernel_id, int site)
{
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    uint64_t prev = globaltimer(), waited = 0;
    for (uint32_t polls = 1;; ++polls) {
        if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (*abort) return false;
        const uint64_t now = globaltimer();
        const int64_t step = (int64_t)(now - prev);
        prev = now;
        if (step > 0) waited += (uint64_t)step < kPollCreditNs ? (uint64_t)step : kPollCreditNs;
        if (waited > g_wait_limit_ns) {
            *abort = 1u;
            record_error(kStatusTimeout, kernel_id, site, (int)(waited / 1000u),
                         (int)(polls < 0x7FFFFFFFu ? polls : 0x7FFFFFFFu), (int)parity, (int)bar);
            return false;
        }
    }
}

// Warp-collective form: lane 0 polls, the result is broadcast, and the warp
// reconverges, so that warp-synchronous code after it never diverges (the
// other lanes are ordered after lane 0's acquire by the warp barrier).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                               int kernel_id, int site)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, kernel_id, site);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// barrier among `count` threads (whole warps) on hardware barrier `id` (1..15)
__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// as named_bar_sync, returning the AND of `v` over the participating threads
__device__ __forceinline__ bool named_bar_and(int id, int count, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %2, 0;\n\t"
        "bar.red.and.pred po, %1, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(v ? 1u : 0u), "r"(count)
        : "memory");
    return r != 0u;
}

// ---------------------------------------------------------------- cluster --
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// all threads of all CTAs of the cluster; shared-memory writes before it are
// visible to the cluster's reads after it
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// -------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}


__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, uint32_t bar, int c0, int c1, int c2,
                                            int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Tensor store shared -> global of one box, tracked by this thread's bulk
// async-groups.  The box may extend past the map's far edges (those elements
// are not written); coordinates are never negative.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(x),
                 "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's committed bulk async-groups have completed (writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Non-tensor bulk copy global -> shared, completing `bytes` of transaction
// on the mbarrier.  src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses with the async
// proxy (TMA, bulk copies, the tensor core): needed after writes the tensor
// core will read, and also after reads of a buffer that a TMA or bulk copy
// refills once it is released -- an mbarrier release alone did not order
// those reads before the copy's write (measured: a one-slot raw-weight ring
// released without it gave results that changed from run to run).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, f16 inputs, f32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, f16 inputs, f32 accumulate.  A (M = 128)
// lives in tensor memory: row m in lane m, column c holding the f16 pair
// (k = 2c, 2c + 1) with the even k in the low half; a 16-k step reads 8
// consecutive columns starting at a_tmem.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, tf32 inputs, f32 accumulate.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on an mbarrier once every previously issued tcgen05 op of this thread completes
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Instruction descriptor for kind::f16: f16 A and B (both K-major), f32 D,
// M = 128 rows (TMEM lanes), N columns.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N)
{
    return (1u << 4)                          // D format: f32
           | (0u << 7) | (0u << 10)           // A, B format: f16
           | (0u << 15) | (0u << 16)          // A, B K-major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Instruction descriptor for kind::tf32: tf32 A and B (K-major), f32 D.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N)
{
    return (1u << 4)                          // D format: f32
           | (2u << 7) | (2u << 10)           // A, B format: tf32
           | ((uint32_t)(N >> 3) << 17)
           | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand without swizzle:
// 8-row x 16-byte core matrices, `lbo` bytes apart along K and `sbo` bytes
// apart along M/N.
__device__ __forceinline__ uint64_t sdesc_k_none(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4)
           | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16)
           | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32)
           | ((uint64_t)1 << 46);                   // version; layout 0 = no swizzle
}

// f32 rounded to tf32 (round to nearest, ties away), low 13 bits cleared
__device__ __forceinline__ float to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO),
// group base 1024-byte aligned.  `addr` may be offset by multiples of 32
// bytes inside a row group to select a K slice of 16 f16 values.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4)      // start address >> 4
           | ((uint64_t)1 << 16)                    // leading byte offset (unused for SW128 K-major)
           | ((uint64_t)(1024 >> 4) << 32)          // stride byte offset: 8 rows x 128 B
           | ((uint64_t)1 << 46)                    // descriptor version (tcgen05)
           | ((uint64_t)2 << 61);                   // layout: 128-byte swizzle
}

// As sdesc_k_sw128 for the 64-byte swizzle layout: rows of 64 bytes (32 f16),
// 8-row groups 512 bytes apart, group base 512-byte aligned; `addr` may be
// offset by 32 bytes inside a row group for the second 16-value K slice.
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4)      // start address >> 4
           | ((uint64_t)1 << 16)                    // leading byte offset (unused for swizzled K-major)
           | ((uint64_t)(512 >> 4) << 32)           // stride byte offset: 8 rows x 64 B
           | ((uint64_t)1 << 46)                    // descriptor version (tcgen05)
           | ((uint64_t)4 << 61);                   // layout: 64-byte swizzle
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: register i of lane l holds
// column (taddr.col + i) of lane (taddr.lane + l).  Values are valid only
// after tmem_ld_wait() on the same registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 16-column variants of the TMEM load / store
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&a)[16], uint32_t (&b)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                   "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                   "+r"(b[14]), "+r"(b[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&a)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Wait for outstanding tcgen05.ld; the registers are tied in so that no use
// of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31])
                 :
                 : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns from registers (the inverse of
// tmem_ld32); complete with tmem_st_wait() before reading the columns back.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace mmq
