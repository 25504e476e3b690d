// gemm_simt.cu -- straightforward CUDA-core grouped expert GEMMs (gate|up with
// fused SwiGLU, and down), decoding MXFP4 inside the reduction.
//
// The decode is the one of "DeepSeek-V4-Flash on a four-GPU Ampere
// workstation", section "MXFP4 is not NVFP4, and the difference matters on
// Ampere": z_n = sum_k a_k v(c_nk) 2^(e_{n, k/32} - 127), FP32 accumulation, no
// decoded copy of the expert written anywhere.  The SwiGLU expert is the one of
// "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1.
//
// One CTA of 128 threads per (row tile, expert group); thread r owns tile row
// r and walks the group's tokens 8 at a time.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "mx_decode.cuh"

namespace moe {

namespace {

struct SimtArgs {
    const uint8_t *wbase;
    size_t group_bytes;
    int kchunks, chunk_bytes, K;
    const int *grp_start, *grp_count, *row_token;
    const uint16_t *in;
    const uint16_t *in_lo;  // down: low BF16 plane of h (h = hi + lo), else nullptr
    int in_ld;
    uint16_t *h_out;        // gate|up: hi plane; the lo plane follows at h_out + h_plane
    long long h_plane;
    float *y_out;
    int I, H, gate_up, fmt;
};

__device__ __forceinline__ float bf16_to_float(uint16_t b) { return __int_as_float((int)((uint32_t)b << 16)); }

constexpr int TOK = 8;
constexpr int TOK_PER_CTA = 64;  // tokens of a group handled by one CTA (blockIdx.z)

__global__ void __launch_bounds__(TILE_ROWS) gemm_simt_kernel(SimtArgs a)
{
    const int g = blockIdx.y, tile = blockIdx.x, r = threadIdx.x, lane = r & 31, q = r >> 5;
    const int cnt = a.grp_count[g];
    if ((int)blockIdx.z * TOK_PER_CTA >= cnt)
        return;
    const int start = a.grp_start[g];
    const uint8_t *wtile = a.wbase + (size_t)g * a.group_bytes + (size_t)tile * a.kchunks * a.chunk_bytes;

    const int c_end = min(cnt, (int)(blockIdx.z + 1) * TOK_PER_CTA);
    for (int c0 = blockIdx.z * TOK_PER_CTA; c0 < c_end; c0 += TOK) {
        float acc[TOK];
        const uint16_t *xrow[TOK];
        const uint16_t *xlo[TOK];
#pragma unroll
        for (int tt = 0; tt < TOK; ++tt) {
            acc[tt] = 0.f;
            int pos = start + min(c0 + tt, c_end - 1);
            int src = a.gate_up ? a.row_token[pos] : pos;
            xrow[tt] = a.in + (size_t)src * a.in_ld;
            xlo[tt] = a.in_lo ? a.in_lo + (size_t)src * a.in_ld : nullptr;
        }
        for (int kc = 0; kc < a.kchunks; ++kc) {
            const uint8_t *chunk = wtile + (size_t)kc * a.chunk_bytes;
            for (int b = 0; b < CHUNK_K / 32; ++b) {
                const int k0 = kc * CHUNK_K + 32 * b;
                if (k0 >= a.K)
                    break;
                float w[32];
                if (a.fmt == FMT_MXFP4) {
                    const uint32_t *words = reinterpret_cast<const uint32_t *>(
                        chunk + (b / 2) * (CHUNK_MX_CODE_BYTES / 2) + r * 32 + (b % 2) * 16);
                    const uint32_t s2 = e8m0_to_bf16x2(chunk[CHUNK_MX_CODE_BYTES + r * (CHUNK_K / 32) + b]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[4];
                        decode_word(words[c], s2, o);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            w[8 * c + 2 * j] = bf16_to_float((uint16_t)(o[j] & 0xFFFFu));
                            w[8 * c + 2 * j + 1] = bf16_to_float((uint16_t)(o[j] >> 16));
                        }
                    }
                } else {
                    const uint16_t *vals = reinterpret_cast<const uint16_t *>(
                        chunk + (b / 2) * (CHUNK_BF16_BYTES / 2) + r * HALF_K * 2) + (b % 2) * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        w[j] = bf16_to_float(vals[j]);
                }
#pragma unroll
                for (int tt = 0; tt < TOK; ++tt) {
                    float s = 0.f;
                    if (xlo[tt]) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            s = fmaf(bf16_to_float(xrow[tt][k0 + j]) + bf16_to_float(xlo[tt][k0 + j]), w[j], s);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            s = fmaf(bf16_to_float(xrow[tt][k0 + j]), w[j], s);
                    }
                    acc[tt] += s;
                }
            }
        }
        if (a.gate_up) {
            const int n = tile * GU_FEATURES_PER_TILE + q * 16 + (lane & 15);
#pragma unroll
            for (int tt = 0; tt < TOK; ++tt) {
                float u = __shfl_sync(0xffffffffu, acc[tt], lane | 16);
                if (lane < 16 && n < a.I && c0 + tt < c_end) {
                    float gt = acc[tt];
                    float hv = gt / (1.0f + expf(-gt)) * u;
                    // h is kept as hi + lo, two BF16 values: hi = bf16(h), lo = bf16(h - hi)
                    __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                    __nv_bfloat16 lb = __float2bfloat16_rn(hv - __bfloat162float(hb));
                    size_t o = (size_t)(start + c0 + tt) * a.I + n;
                    a.h_out[o] = *reinterpret_cast<uint16_t *>(&hb);
                    a.h_out[o + a.h_plane] = *reinterpret_cast<uint16_t *>(&lb);
                }
            }
        } else {
            const int m = tile * TILE_ROWS + r;
            if (m < a.H) {
#pragma unroll
                for (int tt = 0; tt < TOK; ++tt)
                    if (c0 + tt < c_end)
                        a.y_out[(size_t)(start + c0 + tt) * a.H + m] = acc[tt];
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm_gate_up(const Plan &p, const WeightStore &w, int fmt, const uint16_t *x, cudaStream_t st)
{
    SimtArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.cols, p.grp_start, p.grp_count, p.row_token,
               x, nullptr, p.H, p.h, (long long)p.P * p.I, nullptr, p.I, p.H, 1, fmt};
    dim3 grid(w.row_tiles, p.G, (p.T + TOK_PER_CTA - 1) / TOK_PER_CTA);
    gemm_simt_kernel<<<grid, TILE_ROWS, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gemm_down(const Plan &p, const WeightStore &w, int fmt, cudaStream_t st)
{
    SimtArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.cols, p.grp_start, p.grp_count, p.row_token,
               p.h, p.h + (size_t)p.P * p.I, p.I, nullptr, 0, p.y, p.I, p.H, 0, fmt};
    dim3 grid(w.row_tiles, p.G, (p.T + TOK_PER_CTA - 1) / TOK_PER_CTA);
    gemm_simt_kernel<<<grid, TILE_ROWS, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
