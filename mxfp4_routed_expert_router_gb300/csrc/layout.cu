// layout.cu -- load-time weight repack, dense-layer plan, and the weighted
// unpermute-combine of expert outputs into the FP32 result.
#include "moe_internal.cuh"
#include "mx_decode.cuh"

namespace moe {

// ---------------------------------------------------------------- repack
//
// One thread builds one row of one chunk: 64 code bytes + 4 scale bytes
// (MXFP4) or 128 BF16 values (BF16).  The destination row is tile row r of
// row tile `tile`; its source row follows the row order documented in
// moe_internal.cuh.  An E8M0 byte of 255 (NaN in the OCP MX format) sets
// *bad_scale.
__global__ void repack_kernel(int fmt, int gate_up, SrcMat gate, SrcMat up, uint8_t *dst, int row_tiles,
                              int kchunks, int chunk_bytes, int logical_rows, int K, int *bad_scale)
{
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    long long total = (long long)row_tiles * kchunks * TILE_ROWS;
    if (idx >= total)
        return;
    int r = (int)(idx % TILE_ROWS);
    long long tk = idx / TILE_ROWS;
    int kc = (int)(tk % kchunks);
    int tile = (int)(tk / kchunks);

    const SrcMat *src = &gate;
    int srow;
    if (gate_up) {
        int q = r >> 5, l = r & 31;
        srow = tile * GU_FEATURES_PER_TILE + q * 16 + (l & 15);
        if (l >= 16)
            src = &up;
        if (srow >= logical_rows)
            srow = -1;
    } else {
        srow = tile * TILE_ROWS + r;
        if (srow >= logical_rows)
            srow = -1;
    }
    uint8_t *chunk = dst + ((long long)tile * kchunks + kc) * chunk_bytes;
    int k0 = kc * CHUNK_K;
    if (fmt == FMT_MXFP4) {
        // 4 blocks of 32 elements; block b lives in half b/2 at 16*(b%2)
        for (int b = 0; b < CHUNK_K / 32; ++b) {
            uint32_t *words = reinterpret_cast<uint32_t *>(chunk + (b / 2) * (CHUNK_MX_CODE_BYTES / 2) + r * 32 +
                                                           (b % 2) * 16);
            for (int c = 0; c < 4; ++c) {
                uint32_t w = 0;
                for (int i = 0; i < 8; ++i) {
                    int k = k0 + 32 * b + 8 * c + i;
                    uint32_t code = 0;
                    if (srow >= 0 && k < K) {
                        uint8_t byte = src->codes[srow * src->code_stride + k / 2];
                        code = (k & 1) ? (byte >> 4) : (byte & 0xF);
                    }
                    w |= (code & 7u) << (4 * i);
                    w |= (code >> 3) << repacked_sign_bit(i);
                }
                words[c] = w;
            }
            int k = k0 + 32 * b;
            uint8_t e = 127;
            if (srow >= 0 && k < K) {
                e = src->scales[srow * src->scale_stride + k / 32];
                if (e == 255)
                    atomicOr(bad_scale, 1);
            }
            chunk[CHUNK_MX_CODE_BYTES + r * (CHUNK_K / 32) + b] = e;
        }
    } else {
        for (int h = 0; h < 2; ++h) {
            uint16_t *vals = reinterpret_cast<uint16_t *>(chunk + h * (CHUNK_BF16_BYTES / 2) + r * HALF_K * 2);
            for (int j = 0; j < HALF_K; ++j) {
                int k = k0 + h * HALF_K + j;
                uint16_t v = 0;
                if (srow >= 0 && k < K)
                    v = reinterpret_cast<const uint16_t *>(src->codes + srow * src->code_stride)[k];
                vals[j] = v;
            }
        }
    }
}

cudaError_t launch_repack(int fmt, bool gate_up, const SrcMat &gate, const SrcMat &up, const WeightStore &ws,
                          int group, int I, int H, int *bad_scale, cudaStream_t st)
{
    long long total = (long long)ws.row_tiles * ws.kchunks * TILE_ROWS;
    int threads = 128;
    long long blocks = (total + threads - 1) / threads;
    uint8_t *dst = ws.base + (size_t)group * ws.group_bytes;
    int logical_rows = gate_up ? I : H;
    repack_kernel<<<(unsigned)blocks, threads, 0, st>>>(fmt, gate_up ? 1 : 0, gate, up, dst, ws.row_tiles,
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
