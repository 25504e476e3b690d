// routing.cu -- router top-k / renormalisation, expert histogram, prefix sum and
// the stable token permutation.
//
// Routing follows "Cascadia: Resident 975B MoE Inference on Eleven AI PCs"
// §3.1: routing results enter the expert computation as expert IDs plus
// weights, and the expert work is arranged expert-major.  The selection is a
// softmax top-k with renormalisation over the k kept experts.
#include "moe_internal.cuh"

namespace moe {

// Order key of a logit: larger float -> larger key; +0 and -0 equal; NaN
// below every number (key 0, while -inf maps to 0x007FFFFF).
__device__ __forceinline__ uint32_t logit_order_key(float f)
{
    if (isnan(f))
        return 0u;
    if (f == 0.0f)
        f = 0.0f;
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One warp per token.  Lane l owns experts e = l + 32*i, i < NV.  A 64-bit
// key (order key << 32 | ~e) makes every entry distinct, so the warp maximum
// is unique and "larger value, then lower index" falls out of one compare.
// Selected entries are set to key 0, which is below every real entry.
template <int NV>
__global__ void router_kernel(const float *__restrict__ logits, int T, int E, int k, int *__restrict__ ids,
                              float *__restrict__ w, int *__restrict__ counts, int n_counts)
{
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_counts; i += blockDim.x)
            counts[i] = 0;
    int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (warp >= T)
        return;
    const float *row = logits + (long long)warp * E;
    unsigned long long key[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        int e = lane + 32 * i;
        key[i] = 0ull;
        if (e < E)
            key[i] = ((unsigned long long)logit_order_key(row[e]) << 32) | (unsigned long long)(0xFFFFFFFFu - e);
    }
    int my_id = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            best = key[i] > best ? key[i] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (key[i] == best)
                key[i] = 0ull;
        if (lane == j) {
            my_id = e;
            my_v = row[e];
        }
    }
    // w_j = exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0); l_0 is the largest kept logit.
    float l0 = __shfl_sync(0xffffffffu, my_v, 0);
    float ex = (lane < k) ? expf(my_v - l0) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
        ids[(long long)warp * k + lane] = my_id;
        w[(long long)warp * k + lane] = ex / sum;
    }
}

cudaError_t launch_router(const float *logits, int T, int E, int k, int *ids, float *w, int *counts, int n_counts,
                          cudaStream_t st)
{
    int threads = 256;
    int blocks = (T * 32 + threads - 1) / threads;
    int nv = (E + 31) / 32;
#define MOE_ROUTER_CASE(N)                                                                                       \
    if (nv <= N) {                                                                                               \
        router_kernel<N><<<blocks, threads, 0, st>>>(logits, T, E, k, ids, w, counts, n_counts);                 \
        return cudaGetLastError();                                                                               \
    }
    MOE_ROUTER_CASE(1)
    MOE_ROUTER_CASE(2)
    MOE_ROUTER_CASE(4)
    MOE_ROUTER_CASE(8)
    MOE_ROUTER_CASE(16)
    MOE_ROUTER_CASE(32)
#undef MOE_ROUTER_CASE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- histogram

// counts[e] = number of slots routed to expert e (integer atomics: the result
// does not depend on their order).
__global__ void histogram_kernel(const int *__restrict__ ids, int n, int E, int *__restrict__ counts)
{
    extern __shared__ int sh_hist[];
    for (int i = threadIdx.x; i < E; i += blockDim.x)
        sh_hist[i] = 0;
    __syncthreads();
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < n; s += gridDim.x * blockDim.x)
        atomicAdd(&sh_hist[ids[s]], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x)
        if (sh_hist[i])
            atomicAdd(&counts[i], sh_hist[i]);
}

// ---------------------------------------------------------------- permutation
//
// CTA e < E collects the slots of expert e in ascending slot order (a stable
// compaction): position = off[e] + (number of earlier slots with id e).  The
// block-wide rank comes from warp ballots and a scan of per-warp totals, so it
// is deterministic.  CTA E writes expert_offsets and the shared groups.
constexpr int PERM_THREADS = 512;

__global__ void permute_kernel(const int *__restrict__ ids, int T, int k, int E, int S,
                               const int *__restrict__ counts, int *__restrict__ expert_offsets,
                               int *__restrict__ sorted_slot, int *__restrict__ slot_pos, int *__restrict__ grp_start,
                               int *__restrict__ grp_count, int *__restrict__ row_token, int *err)
{
    __shared__ int warp_tot[PERM_THREADS / 32];
    __shared__ int red[PERM_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = T * k;
    const int e = blockIdx.x;

    if (e == E) {
        // expert_offsets[0..E]: exclusive scan of counts, one thread (E <= 1024)
        if (tid == 0) {
            int acc = 0;
            for (int i = 0; i < E; ++i) {
                expert_offsets[i] = acc;
                acc += counts[i];
            }
            expert_offsets[E] = acc;
            if (acc != n)
                atomicCAS(err, 0, DEV_ERR_PERMUTE_COUNT);
        }
        for (int s = tid; s < S; s += blockDim.x) {
            grp_start[E + s] = n + s * T;
            grp_count[E + s] = T;
        }
        for (long long i = tid; i < (long long)S * T; i += blockDim.x)
            row_token[n + i] = (int)(i % T);
        return;
    }

    // off = sum of counts of experts below e
    int part = 0;
    for (int i = tid; i < e; i += blockDim.x)
        part += counts[i];
    for (int o = 16; o > 0; o >>= 1)
        part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0)
        red[wid] = part;
    __syncthreads();
    int off = 0;
    for (int i = 0; i < PERM_THREADS / 32; ++i)
        off += red[i];
    const int cnt = counts[e];
    if (tid == 0) {
        grp_start[e] = off;
        grp_count[e] = cnt;
    }
    if (cnt == 0)
        return;

    int running = 0;
    for (int base = 0; base < n; base += PERM_THREADS) {
        int s = base + tid;
        bool mine = s < n && ids[s] == e;
        unsigned bal = __ballot_sync(0xffffffffu, mine);
        int rank = __popc(bal & ((1u << lane) - 1u));
        if (lane == 0)
            warp_tot[wid] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
        for (int i = 0; i < PERM_THREADS / 32; ++i) {
            int v = warp_tot[i];
            before += (i < wid) ? v : 0;
            total += v;
        }
        if (mine) {
            int pos = off + running + before + rank;
            if (pos < off + cnt) {
                sorted_slot[pos] = s;
                slot_pos[s] = pos;
                row_token[pos] = s / k;
            } else {
                atomicCAS(err, 0, DEV_ERR_PERMUTE_COUNT);
            }
        }
        running += total;
        __syncthreads();
    }
    if (tid == 0 && running != cnt)
        atomicCAS(err, 0, DEV_ERR_PERMUTE_COUNT);
}

cudaError_t launch_permute(const Plan &p, cudaStream_t st)
{
    const int n = p.T * p.k;
    if (p.E > 0 && n > 0) {
        int blocks = (n + 1023) / 1024;
        if (blocks > 296)
            blocks = 296;
        histogram_kernel<<<blocks, 256, p.E * sizeof(int), st>>>(p.topk_ids, n, p.E, p.counts);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    permute_kernel<<<p.E + 1, PERM_THREADS, 0, st>>>(p.topk_ids, p.T, p.k, p.E, p.S, p.counts, p.expert_offsets,
                                                     p.sorted_slot, p.slot_pos, p.grp_start, p.grp_count,
                                                     p.row_token, p.err);
    return cudaGetLastError();
}

}  // namespace moe
