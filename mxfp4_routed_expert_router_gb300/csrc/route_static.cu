// moe_route_static: the routing and grouping step of a routed layer (softmax
// top-k, expert histogram, prefix sum, stable permutation) for callers that
// cannot allocate device memory.  It runs the same router, histogram and
// permutation kernels as moe_forward, but the kernels' scratch (expert counts,
// group table, position -> token map) lives in the fixed file-scope array
// g_route_scratch below instead of a caller-supplied workspace, and the call
// allocates nothing.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.cuh"

namespace {

constexpr int STATIC_MAX_EXPERTS = MOE_ROUTE_STATIC_MAX_EXPERTS;
constexpr int STATIC_MAX_SLOTS = MOE_ROUTE_STATIC_MAX_SLOTS;

// Scratch of the router / histogram / permutation kernels that is not an output
// of this call.  counts must read zero before the histogram adds to it: the
// router kernel zeroes it at the start of every call.  The other members are
// written before they are read within a call.  err is the kernels' first-error
// flag: every call clears it on its stream before its kernels run, and
// moe_route_static_status() reads it back.
struct RouteScratch {
    int counts[STATIC_MAX_EXPERTS];
    int grp_start[STATIC_MAX_EXPERTS];
    int grp_count[STATIC_MAX_EXPERTS];
    int row_token[STATIC_MAX_SLOTS];
    int err;
};

// One copy per device, for the life of the process; every call on that device
// shares it.  sizeof(RouteScratch) = 274,436 bytes.
static __device__ __align__(256) unsigned char g_route_scratch[sizeof(RouteScratch)];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[MAX_DEVICES];  // device address of g_route_scratch per device; nullptr until set up

MoeStatus report(MoeStatus s, const char *fmt, long long a = 0, long long b = 0)
{
    char msg[256];
    snprintf(msg, sizeof msg, fmt, a, b);
    return (MoeStatus)moe::set_last_error((int)s, msg);
}

}  // namespace

extern "C" MoeStatus moe_route_static(const float *router_logits, int T, int E, int k, int *topk_ids, float *topk_w,
                                      int *expert_offsets, int *sorted_slot, int *slot_pos, void *cuda_stream)
{
    if (E < 1 || E > STATIC_MAX_EXPERTS)
        return report(MOE_EINVAL, "moe_route_static: E = %lld outside [1, %lld]", E, STATIC_MAX_EXPERTS);
    if (k < 1 || k > E || k > 32)
        return report(MOE_EINVAL, "moe_route_static: k = %lld outside [1, min(E, 32)] (E = %lld)", k, E);
    if (T < 0)
        return report(MOE_EINVAL, "moe_route_static: T = %lld < 0", T);
    if ((long long)T * k > STATIC_MAX_SLOTS)
        return report(MOE_EINVAL, "moe_route_static: T*k = %lld exceeds the fixed scratch limit of %lld slots",
                      (long long)T * k, STATIC_MAX_SLOTS);
    if (T == 0)
        return MOE_OK;
    if (!router_logits || !topk_ids || !topk_w || !expert_offsets || !sorted_slot || !slot_pos)
        return report(MOE_EINVAL, "moe_route_static: NULL pointer");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return report(MOE_ECUDA, "moe_route_static: cudaGetDevice failed (error %lld)", (long long)e);
    if (dev < 0 || dev >= MAX_DEVICES)
        return report(MOE_EDEVICE, "moe_route_static: device ordinal %lld not supported", dev);

    void *base;
    {
        // Set-up, once per device, on the first call made with that device
        // current: host code needs the array's device address.
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_scratch_addr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_route_scratch);
            if (e != cudaSuccess || !p)
                return report(MOE_ECUDA, "moe_route_static: cudaGetSymbolAddress failed (error %lld)", (long long)e);
            g_scratch_addr[dev] = p;
        }
        base = g_scratch_addr[dev];
    }
    RouteScratch *sc = static_cast<RouteScratch *>(base);
    cudaStream_t st = (cudaStream_t)cuda_stream;

    moe::Plan p{};
    p.T = T;
    p.k = k;
    p.E = E;
    p.S = 0;
    p.G = E;
    p.P = T * k;
    p.topk_ids = topk_ids;
    p.topk_w = topk_w;
    p.counts = sc->counts;
    p.expert_offsets = expert_offsets;
    p.sorted_slot = sorted_slot;
    p.slot_pos = slot_pos;
    p.grp_start = sc->grp_start;
    p.grp_count = sc->grp_count;
    p.row_token = sc->row_token;
    p.err = &sc->err;
    // this call's device-side checks start from a clear flag
    e = cudaMemsetAsync(&sc->err, 0, sizeof(int), st);
    if (e == cudaSuccess)
        e = moe::launch_router(router_logits, T, E, k, topk_ids, topk_w, sc->counts, E, st);
    if (e == cudaSuccess)
        e = moe::launch_permute(p, st);
    if (e != cudaSuccess)
        return report(MOE_ECUDA, "moe_route_static: kernel launch failed (error %lld)", (long long)e);
    return MOE_OK;
}

extern "C" MoeStatus moe_route_static_status(void *cuda_stream)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return report(MOE_ECUDA, "moe_route_static_status: cudaGetDevice failed (error %lld)", (long long)e);
    if (dev < 0 || dev >= MAX_DEVICES)
        return report(MOE_EDEVICE, "moe_route_static_status: device ordinal %lld not supported", dev);
    void *base;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        base = g_scratch_addr[dev];
    }
    if (!base)
        return MOE_OK;  // no call has run on this device
    if ((e = cudaStreamSynchronize((cudaStream_t)cuda_stream)) != cudaSuccess)
        return report(MOE_ECUDA, "moe_route_static_status: cudaStreamSynchronize failed (error %lld)", (long long)e);
    int flag = 0;
    e = cudaMemcpy(&flag, &static_cast<RouteScratch *>(base)->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return report(MOE_ECUDA, "moe_route_static_status: reading the error flag failed (error %lld)", (long long)e);
    if (flag != 0)
        return report(MOE_EDEVICE, "moe_route_static: a kernel reported device error %lld", flag);
    return MOE_OK;
}
