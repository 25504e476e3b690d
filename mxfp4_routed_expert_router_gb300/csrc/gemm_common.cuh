// gemm_common.cuh -- device helpers shared by the GEMM kernels: mbarrier
// waits with time bounds, bulk / tensor (TMA) copies, the work-item schedule
// over expert groups, and host-side tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "moe_internal.cuh"

namespace moe {
namespace gemm {
// internal linkage: every translation unit that includes this gets its own copy
namespace {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s
constexpr int MAX_GROUPS = 1088;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}


__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait (one thread) for the phase with the given parity.  Gives up
// after WAIT_LIMIT_NS, recording DEV_ERR_WAIT_TIMEOUT and raising the CTA's
// abort flag, or as soon as another role has raised it.  Returns true when
// the phase completed.  The first poll is inlined; only a phase that is not
// yet complete takes the out-of-line polling loop.
__device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err)
{
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 7u) == 0) {
            if (*abort_flag)
                return false;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                atomicCAS(err, 0, DEV_ERR_WAIT_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err)
{
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, err);
}

// Warp-wide wait: lane 0 polls, the outcome is broadcast so that the warp
// stays converged (warp-collective instructions that follow never run with a
// partial warp).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err,
                                               int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = mbar_wait(bar, parity, abort_flag, err);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// try_wait with a suspend-time hint: the thread sleeps (up to ns nanoseconds)
// until the phase completes instead of spinning, leaving issue slots to the
// warps that have work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded warp-wide wait for a role that waits long and has nothing else to
// do meanwhile (epilogue, copy issuers): sleeps in the barrier between polls.
__device__ __noinline__ bool mbar_wait_sleep_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000))
            return true;
        if (*abort_flag)
            return false;
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            atomicCAS(err, 0, DEV_ERR_WAIT_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait_sleep_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err,
                                                     int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = mbar_try_wait(bar, parity) || mbar_wait_sleep_slow(bar, parity, abort_flag, err);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Bounded wait used while tearing down: true when the phase completed.
__device__ __noinline__ bool mbar_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}


// ------------------------------------------------------------------ schedule

struct WorkItem {
    int g, rt, tok0, nvalid, n_mma;
};

// prefix[g] = first work item of group g; work items of a group are ordered
// row tile major, token tile minor, so that CTAs running neighbouring items
// share the weight chunk through L2.
__device__ __forceinline__ WorkItem decompose(int t, const int *prefix, const int *counts, int G, int row_tiles,
                                              int nmax)
{
    int lo = 0, hi = G;  // find g with prefix[g] <= t < prefix[g+1]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    WorkItem w;
    w.g = lo;
    const int cnt = counts[lo];
    const int ntiles = (cnt + nmax - 1) / nmax;
    const int local = t - prefix[lo];
    w.rt = local / ntiles;
    const int nt = local % ntiles;
    const int per = (((cnt + ntiles - 1) / ntiles) + 15) & ~15;
    w.tok0 = nt * per;
    w.nvalid = min(per, cnt - w.tok0);
    w.n_mma = (w.nvalid + 15) & ~15;
    return w;
}


// Work-item prefix over groups, computed by one warp (32 groups per step):
// prefix[g] = first work item of group g, prefix[G] = total.
__device__ __forceinline__ void schedule_prefix(const int *counts, int G, int row_tiles, int nmax, int *prefix,
                                                int lane)
{
    int run = 0;
    for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        const int cnt = g < G ? counts[g] : 0;
        const int v = ((cnt + nmax - 1) / nmax) * row_tiles;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += n;
        }
        if (g < G)
            prefix[g] = run + incl - v;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0)
        prefix[G] = run;
}

// ------------------------------------------------------------------ host side

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D BF16 tensor [rows][cols] (row stride cols*2 bytes), box 64 x box_rows, 128B swizzle.
inline cudaError_t make_map(CUtensorMap *m, const void *base, long long rows, int cols, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return cudaErrorNotSupported;
    if (rows < 1)
        rows = 1;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {HALF_K, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D view of a BF16 matrix [rows][cols] (cols a multiple of 64) as 64-wide K
// slices: dims {64, rows, cols/64}, strides {cols*2, 128} bytes, box {64,
// box_rows, box_slices}, 128B swizzle.  One copy then brings box_slices
// consecutive 64-wide K slices of box_rows rows, each slice landing as its own
// 128-byte-swizzled block of box_rows x 128 bytes.
inline cudaError_t make_map_3d(CUtensorMap *m, const void *base, long long rows, int cols, int box_rows,
                               int box_slices)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return cudaErrorNotSupported;
    if (rows < 1)
        rows = 1;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_slices};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

constexpr int MAX_DEVICES = 64;

inline int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        dev = 0;
    return dev;
}

// SM count of the current device, looked up once per device.
inline int sm_count()
{
    static std::atomic<int> cached[MAX_DEVICES];
    const int dev = current_device();
    int n = dev >= 0 && dev < MAX_DEVICES ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (n > 0)
        return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev >= 0 && dev < MAX_DEVICES)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: `done` is the kernel's own flag array, indexed by
// device ordinal.  Setting the attribute twice (two threads racing on a first
// launch) is harmless.
inline cudaError_t smem_limit_once(std::atomic<int> *done, const void *kern, int bytes)
{
    const int dev = current_device();
    const bool cacheable = dev >= 0 && dev < MAX_DEVICES;
    if (cacheable && done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cacheable)
        done[dev].store(1, std::memory_order_release);
    return e;
}


}  // namespace
}  // namespace gemm
}  // namespace moe
