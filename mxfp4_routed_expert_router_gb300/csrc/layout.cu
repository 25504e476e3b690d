// layout.cu -- load-time weight repack, dense-layer plan, and the weighted
// unpermute-combine of expert outputs into the FP32 result.
#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "mx_decode.cuh"

namespace moe {

// ---------------------------------------------------------------- repack
//
// Source element / scale lookups on the caller's row-major matrices; values
// past the logical end read as code 0 / scale 127.  An E8M0 byte of 255 (NaN
// in the OCP MX format) sets *bad_scale.
__device__ __forceinline__ uint32_t src_code(const SrcMat *src, int srow, int k, int K)
{
    if (srow < 0 || k >= K)
        return 0;
    uint8_t byte = src->codes[srow * src->code_stride + k / 2];
    return (k & 1) ? (byte >> 4) : (byte & 0xFu);
}

__device__ __forceinline__ uint8_t src_scale(const SrcMat *src, int srow, int k, int K, int *bad_scale)
{
    if (srow < 0 || k >= K)
        return 127;
    uint8_t e = src->scales[srow * src->scale_stride + k / 32];
    if (e == 255)
        atomicOr(bad_scale, 1);
    return e;
}

__device__ __forceinline__ uint16_t src_bf16(const SrcMat *src, int srow, int k, int K)
{
    if (srow < 0 || k >= K)
        return 0;
    return reinterpret_cast<const uint16_t *>(src->codes + srow * src->code_stride)[k];
}

// Source matrix and row of tile row r of row tile `tile` (row order in moe_internal.cuh).
__device__ __forceinline__ const SrcMat *tile_row_source(int gate_up, const SrcMat *gate, const SrcMat *up,
                                                         int tile, int r, int logical_rows, int *srow)
{
    int row;
    const SrcMat *src = gate;
    if (gate_up) {
        row = gu_row_feature(tile, r);
        if (gu_row_is_up(r))
            src = up;
    } else {
        row = tile * TILE_ROWS + r;
    }
    *srow = row < logical_rows ? row : -1;
    return src;
}

__device__ __forceinline__ uint32_t pack_word(const uint32_t codes[8])
{
    uint32_t w = 0;
    for (int i = 0; i < 8; ++i) {
        w |= (codes[i] & 7u) << (4 * i);
        w |= (codes[i] >> 3) << repacked_sign_bit(i);
    }
    return w;
}

// TILE layout: one thread builds one row of one chunk.
__global__ void repack_tile_kernel(int fmt, int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles,
                                   int kchunks, int chunk_bytes, int logical_rows, int K, int *bad_scale)
{
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)row_tiles * kchunks * TILE_ROWS)
        return;
    const int r = (int)(idx % TILE_ROWS);
    const long long tk = idx / TILE_ROWS;
    const int kc = (int)(tk % kchunks), tile = (int)(tk / kchunks);
    int srow;
    const SrcMat *src = tile_row_source(gate_up, &gate, &up, tile, r, logical_rows, &srow);
    uint8_t *chunk = dst + ((long long)tile * kchunks + kc) * chunk_bytes;
    const int k0 = kc * CHUNK_K;
    if (fmt == FMT_MXFP4) {
        for (int b = 0; b < CHUNK_K / 32; ++b) {
            uint32_t *words =
                reinterpret_cast<uint32_t *>(chunk + (b / 2) * (CHUNK_MX_CODE_BYTES / 2) + r * 32 + (b % 2) * 16);
            for (int c = 0; c < 4; ++c) {
                uint32_t codes[8];
                for (int i = 0; i < 8; ++i)
                    codes[i] = src_code(src, srow, k0 + 32 * b + 8 * c + i, K);
                words[c] = pack_word(codes);
            }
            chunk[CHUNK_MX_CODE_BYTES + r * (CHUNK_K / 32) + b] = src_scale(src, srow, k0 + 32 * b, K, bad_scale);
        }
    } else {
        for (int h = 0; h < 2; ++h) {
            uint16_t *vals = reinterpret_cast<uint16_t *>(chunk + h * (CHUNK_BF16_BYTES / 2) + r * HALF_K * 2);
            for (int j = 0; j < HALF_K; ++j)
                vals[j] = src_bf16(src, srow, k0 + h * HALF_K + j, K);
        }
    }
}

// FRAG layout: one thread builds the fragments of thread t of row group w of
// one chunk (all 8 K steps), plus the group's scales when t % 4 == 0.
__global__ void repack_frag_kernel(int fmt, int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles,
                                   int kchunks, int chunk_bytes, int logical_rows, int K, int *bad_scale)
{
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)row_tiles * kchunks * 256)
        return;
    const int t = (int)(idx % 32), w = (int)((idx / 32) % 8);
    const long long tk = idx / 256;
    const int kc = (int)(tk % kchunks), tile = (int)(tk / kchunks);
    const int g = t / 4, q = t % 4;
    int srow0, srow1;
    const SrcMat *src0 = tile_row_source(gate_up, &gate, &up, tile, 16 * w + g, logical_rows, &srow0);
    const SrcMat *src1 = tile_row_source(gate_up, &gate, &up, tile, 16 * w + g + 8, logical_rows, &srow1);
    uint8_t *chunk = dst + ((long long)tile * kchunks + kc) * chunk_bytes;
    const int k0 = kc * CHUNK_K;
    for (int j = 0; j < 8; ++j) {
        const int ka = k0 + 16 * j + 2 * q, kb = ka + 8;
        if (fmt == FMT_MXFP4) {
            uint32_t codes[8] = {src_code(src0, srow0, ka, K), src_code(src0, srow0, ka + 1, K),
                                 src_code(src1, srow1, ka, K), src_code(src1, srow1, ka + 1, K),
                                 src_code(src0, srow0, kb, K), src_code(src0, srow0, kb + 1, K),
                                 src_code(src1, srow1, kb, K), src_code(src1, srow1, kb + 1, K)};
            reinterpret_cast<uint32_t *>(chunk)[((w * 2 + j / 4) * 32 + t) * 4 + j % 4] = pack_word(codes);
        } else {
            uint16_t *v = reinterpret_cast<uint16_t *>(chunk + ((w * 8 + j) * 32 + t) * 16);
            v[0] = src_bf16(src0, srow0, ka, K);
            v[1] = src_bf16(src0, srow0, ka + 1, K);
            v[2] = src_bf16(src1, srow1, ka, K);
            v[3] = src_bf16(src1, srow1, ka + 1, K);
            v[4] = src_bf16(src0, srow0, kb, K);
            v[5] = src_bf16(src0, srow0, kb + 1, K);
            v[6] = src_bf16(src1, srow1, kb, K);
            v[7] = src_bf16(src1, srow1, kb + 1, K);
        }
    }
    if (fmt == FMT_MXFP4 && q == 0) {
        uint8_t *sc = chunk + CHUNK_MX_CODE_BYTES + (w * 8 + g) * 8;
        for (int b = 0; b < 4; ++b) {
            sc[b] = src_scale(src0, srow0, k0 + 32 * b, K, bad_scale);
            sc[4 + b] = src_scale(src1, srow1, k0 + 32 * b, K, bad_scale);
        }
    }
}

// R_row of every tile row of one group: (largest E8M0 of the row) - 140, 0
// for padding rows.
__global__ void row_rfac_kernel(int gate_up, SrcMat gate, SrcMat up, int16_t *rfac, int row_tiles, int logical_rows,
                                int K)
{
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= row_tiles * TILE_ROWS)
        return;
    int srow;
    const SrcMat *src = tile_row_source(gate_up, &gate, &up, idx / TILE_ROWS, idx % TILE_ROWS, logical_rows, &srow);
    int emax = -1;
    if (srow >= 0)
        for (int b = 0; b < K / 32; ++b) {
            const int e = src->scales[srow * src->scale_stride + b];
            emax = e > emax ? e : emax;
        }
    rfac[idx] = (int16_t)(emax < 0 ? 0 : emax - F16_ROW_HEADROOM);
}

// FRAG_F16 layout (see moe_internal.cuh); rfac of the group filled beforehand.
__global__ void repack_frag_f16_kernel(int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, const int16_t *rfac,
                                       int row_tiles, int kchunks, int chunk_bytes, int logical_rows, int K,
                                       int *bad_scale)
{
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)row_tiles * kchunks * 256)
        return;
    const int t = (int)(idx % 32), w = (int)((idx / 32) % 8);
    const long long tk = idx / 256;
    const int kc = (int)(tk % kchunks), tile = (int)(tk / kchunks);
    const int g = t / 4, q = t % 4;
    int srow0, srow1;
    const SrcMat *src0 = tile_row_source(gate_up, &gate, &up, tile, 16 * w + g, logical_rows, &srow0);
    const SrcMat *src1 = tile_row_source(gate_up, &gate, &up, tile, 16 * w + g + 8, logical_rows, &srow1);
    uint8_t *chunk = dst + ((long long)tile * kchunks + kc) * chunk_bytes;
    const int k0 = kc * CHUNK_K;
    for (int j = 0; j < 8; ++j) {
        const int ka = k0 + 16 * j + 2 * q, kb = ka + 8;
        const uint32_t b0 = src_code(src0, srow0, ka, K) | src_code(src0, srow0, ka + 1, K) << 4;
        const uint32_t b1 = src_code(src1, srow1, ka, K) | src_code(src1, srow1, ka + 1, K) << 4;
        const uint32_t b2 = src_code(src0, srow0, kb, K) | src_code(src0, srow0, kb + 1, K) << 4;
        const uint32_t b3 = src_code(src1, srow1, kb, K) | src_code(src1, srow1, kb + 1, K) << 4;
        reinterpret_cast<uint32_t *>(chunk)[((w * 2 + j / 4) * 32 + t) * 4 + j % 4] = b0 | b1 << 8 | b2 << 16 | b3 << 24;
    }
    if (q == 0) {
        const int r0 = rfac[tile * TILE_ROWS + 16 * w + g], r1 = rfac[tile * TILE_ROWS + 16 * w + g + 8];
        uint8_t *sc = chunk + CHUNK_MX_CODE_BYTES + (w * 8 + g) * 8;
        for (int b = 0; b < 4; ++b) {
            const int e0 = src_scale(src0, srow0, k0 + 32 * b, K, bad_scale) - r0 - 112;
            const int e1 = src_scale(src1, srow1, k0 + 32 * b, K, bad_scale) - r1 - 112;
            sc[b] = (uint8_t)(4 * (e0 < 0 ? 0 : (e0 > 30 ? 30 : e0)));
            sc[4 + b] = (uint8_t)(4 * (e1 < 0 ? 0 : (e1 > 30 ? 30 : e1)));
        }
    }
}

cudaError_t launch_repack(int fmt, int layout, bool gate_up, const SrcMat &gate, const SrcMat &up,
                          const WeightStore &ws, int group, int I, int H, int *bad_scale, cudaStream_t st)
{
    if (layout == LAYOUT_FRAG_F16) {
        const int logical_rows = gate_up ? I : H;
        int16_t *rf = ws.rfac + (size_t)group * ws.row_tiles * TILE_ROWS;
        row_rfac_kernel<<<(ws.row_tiles * TILE_ROWS + 127) / 128, 128, 0, st>>>(gate_up ? 1 : 0, gate, up, rf,
                                                                              ws.row_tiles, logical_rows, ws.cols);
        const long long total = (long long)ws.row_tiles * ws.kchunks * 256;
        repack_frag_f16_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(
            gate_up ? 1 : 0, gate, up, ws.base + (size_t)group * ws.group_bytes, rf, ws.row_tiles, ws.kchunks,
            ws.chunk_bytes, logical_rows, ws.cols, bad_scale);
        return cudaGetLastError();
    }
    const int per_chunk = layout == LAYOUT_TILE ? TILE_ROWS : 256;
    const long long total = (long long)ws.row_tiles * ws.kchunks * per_chunk;
    const int threads = 128;
    const long long blocks = (total + threads - 1) / threads;
    uint8_t *dst = ws.base + (size_t)group * ws.group_bytes;
    const int logical_rows = gate_up ? I : H;
    if (layout == LAYOUT_TILE)
        repack_tile_kernel<<<(unsigned)blocks, threads, 0, st>>>(fmt, gate_up ? 1 : 0, gate, up, dst, ws.row_tiles,
                                                                  ws.kchunks, ws.chunk_bytes, logical_rows, ws.cols,
                                                                  bad_scale);
    else
        repack_frag_kernel<<<(unsigned)blocks, threads, 0, st>>>(fmt, gate_up ? 1 : 0, gate, up, dst, ws.row_tiles,
                                                                  ws.kchunks, ws.chunk_bytes, logical_rows, ws.cols,
                                                                  bad_scale);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- dense plan
//
// A dense layer is G shared groups with every token in every group
// (all-active slices with unit weight): group s covers positions
// [s*T, (s+1)*T) and position s*T + t reads token t.
__global__ void dense_plan_kernel(int T, int G, int *grp_start, int *grp_count, int *row_token)
{
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < G) {
        grp_start[i] = (int)(i * T);
        grp_count[i] = T;
    }
    if (i < (long long)G * T)
        row_token[i] = (int)(i % T);
}

cudaError_t launch_dense_plan(const Plan &p, cudaStream_t st)
{
    long long n = (long long)p.G * p.T;
    if (n < p.G)
        n = p.G;
    dense_plan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p.T, p.G, p.grp_start, p.grp_count,
                                                                  p.row_token);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- FP16 token prep
//
// One CTA per token: xs[t] = floor(log2(max|x_t|)) - 14 (0 for an all-zero
// row, clamped to [-100, 100]), and the FP16 row fp16(x[t][k] * 2^-xs[t]) is
// written to x16[t] and to every routed position of the token
// (x_perm[slot_pos[t*k + j]], j < k).  A BF16 value has 8 significant bits and
// FP16 11, so the conversion is exact for every element within 2^17 of the
// row's largest (and off by at most 2^-25 * 2^xs[t] below that).
constexpr int PREP_THREADS = 256;

__global__ void __launch_bounds__(PREP_THREADS) prep_x16_kernel(const uint16_t *__restrict__ x, int H, int k,
                                                                const int *__restrict__ slot_pos,
                                                                uint16_t *__restrict__ x16, uint16_t *__restrict__ x_perm,
                                                                int *__restrict__ xs)
{
    __shared__ uint32_t red[PREP_THREADS / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    const int nvec = H / 8;  // 8 BF16 per 16-byte vector (H is a multiple of 32)
    uint32_t mx = 0;         // max |x| as BF16 bits without sign (monotonic for finite values)
    for (int i = tid; i < nvec; i += PREP_THREADS) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    }
    for (int o = 16; o > 0; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0)
        red[tid >> 5] = mx;
    __syncthreads();
    mx = 0;
    for (int i = 0; i < PREP_THREADS / 32; ++i)
        mx = max(mx, red[i]);
    int sc = mx == 0 ? 0 : (int)(mx >> 7) - 127 - 14;
    sc = sc < -100 ? -100 : (sc > 100 ? 100 : sc);  // keep 2^-sc a finite float
    if (tid == 0)
        xs[t] = sc;
    const float mul = ldexpf(1.0f, -sc);
    // 16-element groups (two 16-byte vectors), written in the x16 K order
    for (int gi = tid; gi < nvec / 2; gi += PREP_THREADS) {
        const uint4 v0 = row[2 * gi], v1 = row[2 * gi + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint16_t hv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t b = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
            hv[k] = __half_as_ushort(__float2half_rn(__uint_as_float(b << 16) * mul));
        }
        uint32_t o[8];
#pragma unroll
        for (int p2 = 0; p2 < 8; ++p2)
            o[p2] = (uint32_t)hv[x16_logical_k(2 * p2)] | (uint32_t)hv[x16_logical_k(2 * p2 + 1)] << 16;
        const uint4 o0 = make_uint4(o[0], o[1], o[2], o[3]), o1 = make_uint4(o[4], o[5], o[6], o[7]);
        uint4 *dst = reinterpret_cast<uint4 *>(x16 + (size_t)t * H);
        dst[2 * gi] = o0;
        dst[2 * gi + 1] = o1;
        for (int j = 0; j < k; ++j) {
            uint4 *pd = reinterpret_cast<uint4 *>(x_perm + (size_t)slot_pos[t * k + j] * H);
            pd[2 * gi] = o0;
            pd[2 * gi + 1] = o1;
        }
    }
}

cudaError_t launch_prep_x16(const Plan &p, const uint16_t *x, cudaStream_t st)
{
    prep_x16_kernel<<<p.T, PREP_THREADS, 0, st>>>(x, p.H, p.k, p.slot_pos, p.x16, p.x_perm, p.xs);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
//
// out[t] (+)= sum_{j<k} w[t,j] * y[slot_pos[t*k+j]] + sum_{s<S} y[T*k + s*T + t]
// in FP32, in that fixed order (j ascending, then shared groups ascending), so
// the result does not depend on scheduling.  One thread per 4 consecutive
// features of one token (float4 loads/stores; H is a multiple of 32).
__global__ void combine_kernel(const float *__restrict__ y, const float *__restrict__ w,
                               const int *__restrict__ slot_pos, int T, int k, int S, int H, float *__restrict__ out,
                               int accumulate)
{
    int h4 = H / 4;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * h4)
        return;
    int t = (int)(i / h4);
    int c = (int)(i % h4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (accumulate)
        acc = reinterpret_cast<const float4 *>(out)[(long long)t * h4 + c];
    for (int j = 0; j < k; ++j) {
        float wj = w[t * k + j];
        int p = slot_pos[t * k + j];
        float4 v = reinterpret_cast<const float4 *>(y)[(long long)p * h4 + c];
        acc.x = fmaf(wj, v.x, acc.x);
        acc.y = fmaf(wj, v.y, acc.y);
        acc.z = fmaf(wj, v.z, acc.z);
        acc.w = fmaf(wj, v.w, acc.w);
    }
    for (int s = 0; s < S; ++s) {
        long long p = (long long)T * k + (long long)s * T + t;
        float4 v = reinterpret_cast<const float4 *>(y)[p * h4 + c];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4 *>(out)[(long long)t * h4 + c] = acc;
}

cudaError_t launch_combine(const Plan &p, float *out, int accumulate, cudaStream_t st)
{
    long long n = (long long)p.T * (p.H / 4);
    combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p.y, p.topk_w, p.slot_pos, p.T, p.k, p.S, p.H, out,
                                                               accumulate);
    return cudaGetLastError();
}

}  // namespace moe
