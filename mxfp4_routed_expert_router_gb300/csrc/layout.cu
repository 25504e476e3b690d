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

// Group-32 INT4: the FP16 scale bits and the zero point of element k's group.
// Past the logical end the scale is 0 and the zero point 8 (weight 0).  A scale
// with exponent bits 31 (Inf or NaN) or a zero point above 15 sets *bad_scale.
__device__ __forceinline__ uint16_t src_i4_scale(const SrcMat *src, int srow, int k, int K, int *bad_scale)
{
    if (srow < 0 || k >= K)
        return 0;
    const uint16_t s = reinterpret_cast<const uint16_t *>(src->scales)[srow * src->scale_stride + k / 32];
    if ((s & 0x7C00u) == 0x7C00u)
        atomicOr(bad_scale, 1);
    return s;
}

__device__ __forceinline__ uint8_t src_i4_zero(const SrcMat *src, int srow, int k, int K, int *bad_scale)
{
    if (srow < 0 || k >= K || !src->zeros)
        return 8;
    const uint8_t z = src->zeros[srow * src->scale_stride + k / 32];
    if (z > 15)
        atomicOr(bad_scale, 1);
    return z;
}

__device__ __forceinline__ uint16_t src_bf16(const SrcMat *src, int srow, int k, int K)
{
    if (srow < 0 || k >= K)
        return 0;
    return reinterpret_cast<const uint16_t *>(src->codes + srow * src->code_stride)[k];
}

// One warp per row n of a pair of MXFP4 matrices (gate and up rows of one
// feature; or a down row twice): log2 |a_n|^2 and log2 |b_n|^2 of the decoded
// rows, in FP32 against the row's largest exponent among blocks with a nonzero
// code (that block alone contributes at least 1/4, so the blocks too small to
// register below it change the sum by less than 2^-100 of it); `scale` times
// their sum, rounded up by 2^-10, goes into out as an order-preserving key with
// atomicMax (scale 1/2: log2 |a_n| |b_n|; 1/4 with a = b: log2 |a_n|).  An
// all-zero row counts as log2 = -2000.
__device__ __forceinline__ float row_log2_sq(const SrcMat &src, int n, int K, int lane)
{
    const uint8_t *sc = src.scales + (long long)n * src.scale_stride;
    const uint8_t *cd = src.codes + (long long)n * src.code_stride;
    // (2v)^2 of the magnitude indices 0..7, one byte each: 0, 1, 4, 9, 16, 36, 64, 144
    constexpr unsigned long long SQ = 0x9040241009040100ull;
    float acc = 0.f;  // sum of the lane's blocks of q * 4^(e - lmax), q = sum (2v)^2
    int lmax = -1;    // largest exponent of the lane's blocks with a nonzero code
    for (int b = lane; b < K / 32; b += 32) {
        int q = 0;
        for (int i = 0; i < 16; ++i) {
            const uint32_t byte = cd[b * 16 + i];
            q += (int)((SQ >> (8 * (byte & 7u))) & 0xFFu) + (int)((SQ >> (8 * ((byte >> 4) & 7u))) & 0xFFu);
        }
        if (q == 0)
            continue;
        const int e = sc[b];
        if (e > lmax) {
            acc = lmax < 0 ? 0.f : ldexpf(acc, 2 * (lmax - e));
            lmax = e;
        }
        acc += ldexpf((float)q, 2 * (e - lmax));
    }
    int wmax = lmax;
    for (int o = 16; o > 0; o >>= 1)
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
    float v = lmax < 0 ? 0.f : ldexpf(acc, 2 * (lmax - wmax));
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    // sum v(c)^2 = q / 4 at 4^(wmax - 127)
    return wmax < 0 ? -2000.f : log2f(v) - 2.f + 2.f * (float)(wmax - 127);
}

// log2 |w_n|^2 of a group-32 INT4 row: sum over blocks of s_b^2 * sum (q - z_b)^2
// in FP32 (s^2 of an FP16 scale lies in [2^-48, 2^32]: no under- or overflow).
__device__ __forceinline__ float i4_row_log2_sq(const SrcMat &src, int n, int K, int lane)
{
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(src.scales) + (long long)n * src.scale_stride;
    const uint8_t *zp = src.zeros ? src.zeros + (long long)n * src.scale_stride : nullptr;
    const uint8_t *cd = src.codes + (long long)n * src.code_stride;
    float acc = 0.f;
    for (int b = lane; b < K / 32; b += 32) {
        const int z = zp ? zp[b] : 8;
        int q2 = 0;
        for (int i = 0; i < 16; ++i) {
            const int byte = cd[b * 16 + i];
            const int d0 = (byte & 15) - z, d1 = (byte >> 4) - z;
            q2 += d0 * d0 + d1 * d1;
        }
        const float s = __half2float(__ushort_as_half(sc[b]));
        acc = fmaf(s * s, (float)q2, acc);
    }
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc > 0.f ? log2f(acc) : -2000.f;
}

__global__ void gu_norm_kernel(int fmt, SrcMat gate, SrcMat up, int I, int K, float scale, unsigned *out)
{
    const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= I)
        return;
    const float l0 = fmt == FMT_INT4 ? i4_row_log2_sq(gate, n, K, lane) : row_log2_sq(gate, n, K, lane);
    const float l1 = fmt == FMT_INT4 ? i4_row_log2_sq(up, n, K, lane) : row_log2_sq(up, n, K, lane);
    if (lane == 0) {
        const float v = scale * (l0 + l1) + 0.001f;
        const uint32_t b = __float_as_uint(v);
        atomicMax(out, (b & 0x80000000u) ? ~b : (b | 0x80000000u));
    }
}

cudaError_t launch_gu_norm(int fmt, const SrcMat &gate, const SrcMat &up, int group, int I, int H, int *out,
                           cudaStream_t st)
{
    gu_norm_kernel<<<(unsigned)((I + 7) / 8), 256, 0, st>>>(fmt, gate, up, I, H, 0.5f,
                                                            reinterpret_cast<unsigned *>(out) + group);
    return cudaGetLastError();
}

cudaError_t launch_dn_norm(int fmt, const SrcMat &dn, int group, int I, int H, int *out, cudaStream_t st)
{
    gu_norm_kernel<<<(unsigned)((H + 7) / 8), 256, 0, st>>>(fmt, dn, dn, H, I, 0.25f,
                                                            reinterpret_cast<unsigned *>(out) + group);
    return cudaGetLastError();
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

// FRAG_F16 layout (see moe_internal.cuh), MXFP4 or group-32 INT4 codes.
__global__ void repack_frag_f16_kernel(int fmt, int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles,
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
        uint32_t word;
        if (fmt == FMT_INT4) {
            // pair p: first element in nibble p, second in nibble p + 4
            const uint32_t first[4] = {src_code(src0, srow0, ka, K), src_code(src1, srow1, ka, K),
                                       src_code(src0, srow0, kb, K), src_code(src1, srow1, kb, K)};
            const uint32_t second[4] = {src_code(src0, srow0, ka + 1, K), src_code(src1, srow1, ka + 1, K),
                                        src_code(src0, srow0, kb + 1, K), src_code(src1, srow1, kb + 1, K)};
            word = 0;
            for (int p = 0; p < 4; ++p)
                word |= first[p] << (4 * p) | second[p] << (4 * p + 16);
        } else {
            const uint32_t b0 = src_code(src0, srow0, ka, K) | src_code(src0, srow0, ka + 1, K) << 4;
            const uint32_t b1 = src_code(src1, srow1, ka, K) | src_code(src1, srow1, ka + 1, K) << 4;
            const uint32_t b2 = src_code(src0, srow0, kb, K) | src_code(src0, srow0, kb + 1, K) << 4;
            const uint32_t b3 = src_code(src1, srow1, kb, K) | src_code(src1, srow1, kb + 1, K) << 4;
            word = b0 | b1 << 8 | b2 << 16 | b3 << 24;
        }
        reinterpret_cast<uint32_t *>(chunk)[((w * 2 + j / 4) * 32 + t) * 4 + j % 4] = word;
    }
    if (fmt == FMT_INT4 && q == 0) {
        uint16_t *sc = reinterpret_cast<uint16_t *>(chunk + CHUNK_MX_CODE_BYTES + (w * 8 + g) * 16);
        uint8_t *zp = chunk + CHUNK_MX_CODE_BYTES + CHUNK_I4_SCALE_BYTES + (w * 8 + g) * 8;
        for (int b = 0; b < 4; ++b) {
            sc[b] = src_i4_scale(src0, srow0, k0 + 32 * b, K, bad_scale);
            sc[4 + b] = src_i4_scale(src1, srow1, k0 + 32 * b, K, bad_scale);
            zp[b] = src_i4_zero(src0, srow0, k0 + 32 * b, K, bad_scale);
            zp[4 + b] = src_i4_zero(src1, srow1, k0 + 32 * b, K, bad_scale);
        }
    } else if (q == 0) {
        uint8_t *sc = chunk + CHUNK_MX_CODE_BYTES + (w * 8 + g) * 8;
        for (int b = 0; b < 4; ++b) {
            sc[b] = src_scale(src0, srow0, k0 + 32 * b, K, bad_scale);
            sc[4 + b] = src_scale(src1, srow1, k0 + 32 * b, K, bad_scale);
        }
    }
}

// TILE_F16 layout (MXFP4 only; see moe_internal.cuh): one thread builds one
// row of one chunk -- plain pack4 code bytes per 32-value block and the raw
// E8M0 bytes (127 past K, whose codes are 0).
__global__ void repack_tile_f16_kernel(int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles, int kchunks,
                                       int chunk_bytes, int logical_rows, int K, int *bad_scale)
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
    for (int b = 0; b < CHUNK_K / 32; ++b) {
        uint32_t words[4];
        for (int c = 0; c < 4; ++c) {
            uint32_t wv = 0;
            for (int i = 0; i < 8; ++i)
                wv |= src_code(src, srow, k0 + 32 * b + 8 * c + i, K) << (4 * i);
            words[c] = wv;
        }
        *reinterpret_cast<uint4 *>(chunk + (b * TILE_ROWS + r) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
        chunk[CHUNK_MX_CODE_BYTES + b * TILE_ROWS + r] = src_scale(src, srow, k0 + 32 * b, K, bad_scale);
    }
}

// TILE_I4 layout (group-32 INT4; see moe_internal.cuh): one thread builds one
// row of one chunk -- per 32-value block, the codes with pair (2p, 2p + 1) of
// each 8-value word in nibbles p and p + 4, the FP16 scale bits and the zero
// point (scale 0 and zero point 8 past K, a weight of 0).
__global__ void repack_tile_i4_kernel(int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles, int kchunks,
                                      int chunk_bytes, int logical_rows, int K, int *bad_scale)
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
    for (int b = 0; b < CHUNK_K / 32; ++b) {
        uint32_t words[4];
        for (int c = 0; c < 4; ++c) {
            uint32_t wv = 0;
            for (int p = 0; p < 4; ++p) {
                const int k = k0 + 32 * b + 8 * c + 2 * p;
                wv |= src_code(src, srow, k, K) << (4 * p);
                wv |= src_code(src, srow, k + 1, K) << (4 * p + 16);
            }
            words[c] = wv;
        }
        *reinterpret_cast<uint4 *>(chunk + (b * TILE_ROWS + r) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
        reinterpret_cast<uint16_t *>(chunk + CHUNK_MX_CODE_BYTES)[b * TILE_ROWS + r] =
            src_i4_scale(src, srow, k0 + 32 * b, K, bad_scale);
        chunk[CHUNK_MX_CODE_BYTES + CHUNK_I4_SCALE_BYTES + b * TILE_ROWS + r] =
            src_i4_zero(src, srow, k0 + 32 * b, K, bad_scale);
    }
}

// Row bases of a TILE_I4 store: one warp per tile row, b_row + 127 with b_row =
// floor(log2 max|s|) - TILE_I4_BASE_SHIFT over the row's nonzero FP16 scales
// (127 for a row with none, or past the logical end).
__global__ void row_base_i4_kernel(int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles, int logical_rows,
                                   int K)
{
    const long long idx = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (idx >= (long long)row_tiles * TILE_ROWS)
        return;
    const int r = (int)(idx % TILE_ROWS), tile = (int)(idx / TILE_ROWS);
    int srow;
    const SrcMat *src = tile_row_source(gate_up, &gate, &up, tile, r, logical_rows, &srow);
    int mx = -1000;
    if (srow >= 0) {
        const uint16_t *sc = reinterpret_cast<const uint16_t *>(src->scales) + (long long)srow * src->scale_stride;
        for (int b = lane; b < K / 32; b += 32) {
            const float s = fabsf(__half2float(__ushort_as_half(sc[b])));
            if (s > 0.f && s <= 65504.f)
                mx = max(mx, ilogbf(s));
        }
    }
    for (int o = 16; o > 0; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0)
        dst[idx] = (uint8_t)(mx == -1000 ? 127 : mx - TILE_I4_BASE_SHIFT + 127);
}

// Row bases of a TILE_F16 store: one thread per tile row; rows past the
// logical end get 127 (their codes are 0).
__global__ void row_base_kernel(int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles, int logical_rows,
                                int K, int *wide)
{
    // one warp per tile row; lanes read the row's scale bytes side by side
    const long long idx = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (idx >= (long long)row_tiles * TILE_ROWS)
        return;
    const int r = (int)(idx % TILE_ROWS), tile = (int)(idx / TILE_ROWS);
    int srow;
    const SrcMat *src = tile_row_source(gate_up, &gate, &up, tile, r, logical_rows, &srow);
    if (srow < 0) {
        if (lane == 0)
            dst[idx] = 127;
        return;
    }
    const uint8_t *sc = src->scales + srow * src->scale_stride;
    int mx = 0, mn = 255;
    for (int b = lane; b < K / 32; b += 32) {
        const int e = sc[b];
        mx = e > mx ? e : mx;
        mn = e < mn ? e : mn;
    }
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        dst[idx] = (uint8_t)mx;
        if (mx - mn > TILE_F16_MAX_SPREAD)
            atomicOr(wide, 1);
    }
}

cudaError_t launch_row_base(int fmt, bool gate_up, const SrcMat &gate, const SrcMat &up, const WeightStore &ws,
                            int group, int I, int H, int *wide, cudaStream_t st)
{
    const int logical_rows = gate_up ? I : H;
    const long long total = (long long)ws.row_tiles * TILE_ROWS;
    if (fmt == FMT_INT4)
        row_base_i4_kernel<<<(unsigned)((total + 7) / 8), 256, 0, st>>>(
            gate_up ? 1 : 0, gate, up, ws.row_base + (size_t)group * total, ws.row_tiles, logical_rows, ws.cols);
    else
        row_base_kernel<<<(unsigned)((total + 7) / 8), 256, 0, st>>>(
            gate_up ? 1 : 0, gate, up, ws.row_base + (size_t)group * total, ws.row_tiles, logical_rows, ws.cols,
            wide);
    return cudaGetLastError();
}

cudaError_t launch_repack(int fmt, int layout, bool gate_up, const SrcMat &gate, const SrcMat &up,
                          const WeightStore &ws, int group, int I, int H, int *bad_scale, cudaStream_t st)
{
    if (layout == LAYOUT_FRAG_F16) {
        const int logical_rows = gate_up ? I : H;
        const long long total = (long long)ws.row_tiles * ws.kchunks * 256;
        repack_frag_f16_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(
            fmt, gate_up ? 1 : 0, gate, up, ws.base + (size_t)group * ws.group_bytes, ws.row_tiles, ws.kchunks,
            ws.chunk_bytes, logical_rows, ws.cols, bad_scale);
        return cudaGetLastError();
    }
    if (layout == LAYOUT_TILE_I4) {
        const int logical_rows = gate_up ? I : H;
        const long long total = (long long)ws.row_tiles * ws.kchunks * TILE_ROWS;
        repack_tile_i4_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(
            gate_up ? 1 : 0, gate, up, ws.base + (size_t)group * ws.group_bytes, ws.row_tiles, ws.kchunks,
            ws.chunk_bytes, logical_rows, ws.cols, bad_scale);
        return cudaGetLastError();
    }
    if (layout == LAYOUT_TILE_F16) {
        const int logical_rows = gate_up ? I : H;
        const long long total = (long long)ws.row_tiles * ws.kchunks * TILE_ROWS;
        repack_tile_f16_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(
            gate_up ? 1 : 0, gate, up, ws.base + (size_t)group * ws.group_bytes, ws.row_tiles, ws.kchunks,
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
        if (p < 0)  // an empty slot of caller routing
            continue;
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

// The same over FP16 rows: y[p] = y16[p] * 2^ys[p], in the same fixed order.
__global__ void combine_f16_kernel(const uint16_t *__restrict__ y16, const int *__restrict__ ys,
                                   const float *__restrict__ w, const int *__restrict__ slot_pos, int T, int k, int S,
                                   int H, float *__restrict__ out, int accumulate)
{
    const int h4 = H / 4;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * h4)
        return;
    const int t = (int)(i / h4);
    const int c = (int)(i % h4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (accumulate)
        acc = reinterpret_cast<const float4 *>(out)[(long long)t * h4 + c];
    auto row = [&](long long p, float f) {
        const uint2 v = reinterpret_cast<const uint2 *>(y16)[p * h4 + c];
        const float sc = f * __int_as_float((127 + ys[p]) << 23);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        acc.x = fmaf(sc, a.x, acc.x);
        acc.y = fmaf(sc, a.y, acc.y);
        acc.z = fmaf(sc, b.x, acc.z);
        acc.w = fmaf(sc, b.y, acc.w);
    };
    for (int j = 0; j < k; ++j) {
        const int p = slot_pos[t * k + j];
        if (p >= 0)  // (-1: an empty slot of caller routing)
            row(p, w[t * k + j]);
    }
    for (int s = 0; s < S; ++s)
        row((long long)T * k + (long long)s * T + t, 1.0f);
    reinterpret_cast<float4 *>(out)[(long long)t * h4 + c] = acc;
}

cudaError_t launch_combine_f16(const Plan &p, float *out, int accumulate, cudaStream_t st)
{
    long long n = (long long)p.T * (p.H / 4);
    combine_f16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(reinterpret_cast<const uint16_t *>(p.y), p.ys,
                                                                   p.topk_w, p.slot_pos, p.T, p.k, p.S, p.H, out,
                                                                   accumulate);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Plan &p, float *out, int accumulate, cudaStream_t st)
{
    long long n = (long long)p.T * (p.H / 4);
    combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p.y, p.topk_w, p.slot_pos, p.T, p.k, p.S, p.H, out,
                                                               accumulate);
    return cudaGetLastError();
}

}  // namespace moe
