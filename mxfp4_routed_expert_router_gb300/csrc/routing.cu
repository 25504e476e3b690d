// routing.cu -- router top-k / renormalisation, expert histogram, prefix sum and
// the stable token permutation.
//
// Routing follows "Cascadia: Resident 975B MoE Inference on Eleven AI PCs"
// §3.1: the expert computation sees the routing only as one expert id and one
// weight per selection, and the expert work is arranged expert-major.  The selection is a
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

// ---------------------------------------------------------------- routing given by the caller
//
// "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1: the router
// hands the expert computation expert ids and their weights.  The caller's
// arrays are copied into the call's routing arrays.  The ids are global: the
// layer holds experts [ebase, ebase + E) of etotal, which become its groups
// 0..E-1.  An ID of -1, or of an expert held elsewhere, marks an empty slot
// (ID -1, weight 0: it is not grouped and adds nothing); any other ID outside
// [0, etotal) records DEV_ERR_BOUNDS (reported by moe_sync_status) and is
// replaced by group 0 with weight 0, so that everything after it stays in
// bounds.
__device__ __forceinline__ void route_in(int &e, float &wv, int E, int ebase, int etotal, int *err)
{
    if (e == -1) {
        wv = 0.f;
    } else if (e < 0 || e >= etotal) {
        atomicCAS(err, 0, DEV_ERR_BOUNDS);
        e = 0;
        wv = 0.f;
    } else if (e < ebase || e - ebase >= E) {
        e = -1;
        wv = 0.f;
    } else {
        e -= ebase;
    }
}

__global__ void routing_copy_kernel(const int *__restrict__ ids_in, const float *__restrict__ w_in, int n, int E,
                                    int ebase, int etotal, int *__restrict__ ids, float *__restrict__ w,
                                    int *__restrict__ counts, int n_counts, int *err)
{
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_counts; i += blockDim.x)
            counts[i] = 0;
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < n; s += gridDim.x * blockDim.x) {
        int e = ids_in[s];
        float wv = w_in[s];
        route_in(e, wv, E, ebase, etotal, err);
        ids[s] = e;
        w[s] = wv;
    }
}

cudaError_t launch_routing_copy(const int *ids_in, const float *w_in, int n, int E, int ebase, int etotal, int *ids,
                                float *w, int *counts, int n_counts, int *err, cudaStream_t st)
{
    int blocks = (n + 255) / 256;
    if (blocks < 1)
        blocks = 1;
    if (blocks > 1024)
        blocks = 1024;
    routing_copy_kernel<<<blocks, 256, 0, st>>>(ids_in, w_in, n, E, ebase, etotal, ids, w, counts, n_counts, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- sigmoid routing
//
// The routing of "Cascadia" §3.1: sigmoid scores s_e = 1 / (1 + exp(-l_e)),
// selection of the k largest keys s_e + b_e (the bias decides only the
// selection), weights w_j = scale * s_j / sum of the selected scores.  Scores
// and keys are FP64, so that the selection matches an FP64 reference except
// for keys less than an FP64 ulp apart.  One warp per token; lane l holds the
// keys of experts l, l+32, ... as order keys + 1 (0: absent or taken).  Each
// round takes the warp's largest key and, among the experts holding it, the
// lowest index.

// total order of doubles as unsigned integers: larger value, larger key; +0
// and -0 equal; NaN below every number
__device__ __forceinline__ unsigned long long double_order_key(double d)
{
    if (isnan(d))
        return 0ull;
    if (d == 0.0)
        d = 0.0;
    const unsigned long long b = (unsigned long long)__double_as_longlong(d);
    return (b & 0x8000000000000000ull) ? ~b : (b | 0x8000000000000000ull);
}

template <int NV>
__global__ void router_sigmoid_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E,
                                      int k, float scale, int *__restrict__ ids, float *__restrict__ w)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= T)
        return;
    const float *row = logits + (long long)warp * E;
    unsigned long long key[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0ull;
        if (e < E) {
            const double sc = 1.0 / (1.0 + exp(-(double)row[e]));
            key[i] = double_order_key(sc + (bias ? (double)bias[e] : 0.0)) + 1ull;
        }
    }
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        unsigned long long best = 0ull;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (key[i] > best) {  // strict: the lowest expert of the lane among equals
                best = key[i];
                bi = i;
            }
        unsigned long long m = best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, m, o);
            m = other > m ? other : m;
        }
        const unsigned mine = (unsigned)(lane + 32 * bi);
        const unsigned ew = __reduce_min_sync(0xffffffffu, best == m ? mine : 0xFFFFFFFFu);
        if (mine == ew) {
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if (i == bi)
                    key[i] = 0ull;
        }
        if (lane == j)
            my_e = (int)ew;
    }
    const double my_s = lane < k ? 1.0 / (1.0 + exp(-(double)row[my_e])) : 0.0;
    double sum = my_s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
        ids[(long long)warp * k + lane] = my_e;
        w[(long long)warp * k + lane] = (float)((double)scale * my_s / sum);
    }
}

cudaError_t launch_router_sigmoid(const float *logits, const float *bias, int T, int E, int k, float scale, int *ids,
                                  float *w, cudaStream_t st)
{
    const int threads = 256;
    const int blocks = (T * 32 + threads - 1) / threads;
    const int nv = (E + 31) / 32;
#define MOE_SIGMOID_CASE(N)                                                                                      \
    if (nv <= N) {                                                                                               \
        router_sigmoid_kernel<N><<<blocks, threads, 0, st>>>(logits, bias, T, E, k, scale, ids, w);              \
        return cudaGetLastError();                                                                               \
    }
    MOE_SIGMOID_CASE(1)
    MOE_SIGMOID_CASE(2)
    MOE_SIGMOID_CASE(4)
    MOE_SIGMOID_CASE(8)
    MOE_SIGMOID_CASE(16)
    MOE_SIGMOID_CASE(32)
#undef MOE_SIGMOID_CASE
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
        if ((unsigned)ids[s] < (unsigned)E)
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

// Chunked stable counting sort (moe_forward's path): the slots are cut into
// chunks of PERM_CHUNK; one kernel counts each chunk's slots per expert (and,
// in column E, its empty slots: ID -1 from caller routing), a second gives
// every chunk its starting position per expert (slots of the experts below,
// then of the same expert in earlier chunks) and places the chunk's slots in
// slot order.  Integer counts only: the result equals the one-CTA-per-expert
// kernel above, bit for bit.  Empty slots get no position (slot_pos -1); the
// positions from expert_offsets[E] to T*k are left unused (sorted_slot -1,
// token 0).
constexpr int PERM_CHUNK = 1024;
constexpr int PERM_CT = 256;                    // threads of the chunked kernels
constexpr int PERM_CW = PERM_CT / 32;           // warps
constexpr int PERM_WSLOTS = PERM_CHUNK / PERM_CW;  // consecutive slots per warp

__global__ void chunk_hist_kernel(const int *__restrict__ ids, int n, int E, int *__restrict__ chunk_cnt)
{
    extern __shared__ int h[];  // [E + 1]: per expert, then the empty slots
    for (int i = threadIdx.x; i <= E; i += blockDim.x)
        h[i] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * PERM_CHUNK, s1 = min(n, s0 + PERM_CHUNK);
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
        const int e = ids[s];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&h[e], 1);
        else if (e == -1)
            atomicAdd(&h[E], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i <= E; i += blockDim.x)
        chunk_cnt[(size_t)blockIdx.x * (E + 1) + i] = h[i];
}

__global__ void chunk_scatter_kernel(const int *__restrict__ ids, int T, int k, int E, int S, int nchunks,
                                     const int *__restrict__ chunk_cnt, int *__restrict__ counts,
                                     int *__restrict__ expert_offsets, int *__restrict__ sorted_slot,
                                     int *__restrict__ slot_pos, int *__restrict__ grp_start,
                                     int *__restrict__ grp_count, int *__restrict__ row_token, int *err)
{
    extern __shared__ int sm[];
    int *base = sm;            // [E]  first position of this chunk's slots of expert e
    int *wc = sm + E;          // [PERM_CW][E]  per-warp counts, then per-warp running positions
    __shared__ int wsum[PERM_CW];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = T * k, c = blockIdx.x;
    // per expert: all slots (tot) and those of earlier chunks (pre); this thread
    // takes experts [e0, e1) for the scan
    const int per = (E + PERM_CT - 1) / PERM_CT;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int mytot = 0;
    for (int e = e0; e < e1; ++e) {
        int tot = 0, pre = 0;
        for (int cc = 0; cc < nchunks; ++cc) {
            const int v = chunk_cnt[(size_t)cc * (E + 1) + e];
            tot += v;
            pre += cc < c ? v : 0;
        }
        base[e] = tot;
        wc[e] = pre;
        mytot += tot;
    }
    // exclusive scan of the totals over experts
    int incl = mytot;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        wsum[wid] = incl;
    __syncthreads();
    int run = incl - mytot;
    for (int w = 0; w < wid; ++w)
        run += wsum[w];
    int grand = 0;
    for (int w = 0; w < PERM_CW; ++w)
        grand += wsum[w];
    for (int e = e0; e < e1; ++e) {
        const int tot = base[e];
        if (c == 0) {
            counts[e] = tot;
            expert_offsets[e] = run;
            grp_start[e] = run;
            grp_count[e] = tot;
        }
        base[e] = run + wc[e];
        run += tot;
    }
    if (c == 0 && tid == 0) {
        expert_offsets[E] = grand;
        int empty = 0;
        for (int cc = 0; cc < nchunks; ++cc)
            empty += chunk_cnt[(size_t)cc * (E + 1) + E];
        if (grand + empty != n)
            atomicCAS(err, 0, DEV_ERR_PERMUTE_COUNT);
    }
    if (c == 0)  // positions left unused by empty slots
        for (int p = grand + tid; p < n; p += blockDim.x) {
            sorted_slot[p] = -1;
            row_token[p] = 0;
        }
    if (c == 0)
        for (int s = tid; s < S; s += blockDim.x) {
            grp_start[E + s] = n + s * T;
            grp_count[E + s] = T;
        }
    for (long long i = (long long)c * blockDim.x + tid; i < (long long)S * T; i += (long long)nchunks * blockDim.x)
        row_token[n + i] = (int)(i % T);
    __syncthreads();
    // per-warp counts of the chunk, then each warp's first position per expert
    const int ws0 = c * PERM_CHUNK + wid * PERM_WSLOTS, ws1 = min(n, ws0 + PERM_WSLOTS);
    int *my = wc + wid * E;
    for (int e = lane; e < E; e += 32)
        my[e] = 0;
    __syncwarp();
    for (int s = ws0 + lane; s < ws1; s += 32) {
        const int e = ids[s];
        if ((unsigned)e < (unsigned)E)
            atomicAdd(&my[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int r = base[e];
        for (int w = 0; w < PERM_CW; ++w) {
            const int v = wc[w * E + e];
            wc[w * E + e] = r;
            r += v;
        }
    }
    __syncthreads();
    // each warp places its slots in order, 32 at a time
    for (int b = ws0; b < ws1; b += 32) {
        const int s = b + lane;
        const bool act = s < ws1;
        const int e = act ? ids[s] : -1;
        const bool ok = act && (unsigned)e < (unsigned)E;
        const unsigned m = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok) {
            const int pos = my[e] + __popc(m & ((1u << lane) - 1u));
            sorted_slot[pos] = s;
            slot_pos[s] = pos;
            row_token[pos] = s / k;
        } else if (act && e == -1) {
            slot_pos[s] = -1;  // an empty slot
        } else if (act) {
            atomicCAS(err, 0, DEV_ERR_PERMUTE_COUNT);
        }
        __syncwarp();
        if (ok && lane == 31 - __clz(m))
            my[e] += __popc(m);
        __syncwarp();
    }
}

cudaError_t launch_permute(const Plan &p, cudaStream_t st)
{
    const int n = p.T * p.k;
    if (p.chunk_cnt && p.E > 0 && n > 0) {
        const int nchunks = (n + PERM_CHUNK - 1) / PERM_CHUNK;
        chunk_hist_kernel<<<nchunks, PERM_CT, (p.E + 1) * sizeof(int), st>>>(p.topk_ids, n, p.E, p.chunk_cnt);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        chunk_scatter_kernel<<<nchunks, PERM_CT, (1 + PERM_CW) * p.E * sizeof(int), st>>>(
            p.topk_ids, p.T, p.k, p.E, p.S, nchunks, p.chunk_cnt, p.counts, p.expert_offsets, p.sorted_slot,
            p.slot_pos, p.grp_start, p.grp_count, p.row_token, p.err);
        return cudaGetLastError();
    }
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
