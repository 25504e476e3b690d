// gemm_stream.cu -- register-streaming grouped expert GEMMs for decode-sized
// batches (a handful of tokens per expert), where the layer is bound by
// reading each selected expert's weights once from HBM.
//
// Same operations as gemm_tc.cu (gate|up with fused SwiGLU, and down; SwiGLU
// expert of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1,
// MXFP4 decoded inside the reduction as in "DeepSeek-V4-Flash on a four-GPU
// Ampere workstation", section "MXFP4 is not NVFP4, and the difference matters
// on Ampere").  Design for the HBM-bound regime:
//   * one CTA per SM walks a static schedule of (group, 128-row tile, token
//     tile of <= 8*NT tokens) work items;
//   * warp 0 streams CH consecutive 128-row x 128-K weight chunks (FRAG
//     layouts, contiguous, one bulk async copy of up to 34.8 KB) together with
//     the matching token rows (one 3-D TMA copy per 8-token tile and operand,
//     128-byte swizzle) into a ring of shared-memory stages: one mbarrier
//     handshake per stage;
//   * 16 compute warps: warp pair (w, w+8) owns 16 weight rows, warp w the
//     first and warp w+8 the second 64-wide half of every chunk; each decodes
//     its weights straight into warp-level MMA A fragments and runs m16n8k16
//     MMAs with FP32 accumulators in registers -- no decoded tile is written
//     anywhere, not even to shared memory;
//   * the pair sums its accumulators through shared memory and the epilogue
//     runs on registers.
// MXFP4 weights run on FP16 operands: the hardware E2M1 -> FP16 conversion
// decodes two weights per instruction, each block multiplier is rebased per
// weight row into FP16 range (FRAG_F16 layout), x enters as x16 (FP16, scaled
// per token) and h as FP16 hi + lo scaled per (position, 64-feature block);
// every power of two is undone exactly in FP32.  BF16 weights run on BF16
// operands (BF16 x, h as BF16 hi + lo).
// Every mbarrier wait is bounded (gemm_common.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "mx_decode.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int ST_COMPUTE_WARPS = 16;
constexpr int ST_THREADS = (1 + ST_COMPUTE_WARPS) * 32;
constexpr int BBOX_ROWS = 8;
constexpr int BBOX_BYTES = BBOX_ROWS * HALF_K * 2;  // 1 KB: 8 token rows x 64 BF16, one 128-byte-swizzle atom
constexpr int ST_SMEM_LIMIT = 232448;

template <bool GU, int WFMT, int NT, int CH>
struct StreamLayout {
    static constexpr int NB = GU ? 1 : 2;  // token operands (down: hi and lo planes of h)
    static constexpr int W_CHUNK = WFMT == FMT_MXFP4 ? CHUNK_MX_BYTES : CHUNK_BF16_BYTES;
    static constexpr int KS = 2 * CH;                          // 64-wide K slices per stage
    static constexpr int B_BYTES = NB * NT * KS * BBOX_BYTES;  // [operand][n tile][K slice] boxes
    static constexpr int STAGE = ((B_BYTES + CH * W_CHUNK) + 1023) / 1024 * 1024;
    static constexpr int RED_BYTES = 8 * NT * 4 * 32 * 4 + 8 * NT * 8 * 4;  // pair sums + h block maxima
    static constexpr int FIXED = RED_BYTES + (MAX_GROUPS + 1) * 4 + 16 + 64 + 1024 + 2 * 16 * 8;
    static constexpr int R_FIT = (ST_SMEM_LIMIT - FIXED) / STAGE;
    static constexpr int R = R_FIT > 12 ? 12 : R_FIT;
    static constexpr int RED_OFF = R * STAGE;
    static constexpr int BAR_OFF = RED_OFF + RED_BYTES;
    static constexpr int SCHED_OFF = BAR_OFF + 2 * R * 8;
    static constexpr int MISC_OFF = SCHED_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int PAIR_OFF = MISC_OFF + 16;
    static constexpr int TOTAL = PAIR_OFF + 64 + 1024;
};

// the largest stage (chunks per stage) that still leaves a ring of >= 3 stages
template <bool GU, int WFMT, int NT>
struct StreamCfg {
    static constexpr int CH = StreamLayout<GU, WFMT, NT, 4>::R >= 3   ? 4
                              : StreamLayout<GU, WFMT, NT, 2>::R >= 3 ? 2
                                                                       : 1;
    using L = StreamLayout<GU, WFMT, NT, CH>;
    static_assert(L::R >= 2, "stage ring");
    static_assert(L::TOTAL <= ST_SMEM_LIMIT, "shared memory");
};

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// FRAG_F16 word -> A fragment: each byte (two OCP E2M1 codes) converts to an
// FP16 pair in hardware, then takes its row's FP16 block multiplier.
__device__ __forceinline__ void decode_word_f16(uint32_t w, uint32_t sa, uint32_t sb, uint32_t out[4])
{
    uint32_t r0, r1, r2, r3;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[0]) : "r"(r0), "r"(sa));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[1]) : "r"(r1), "r"(sb));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[2]) : "r"(r2), "r"(sa));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[3]) : "r"(r3), "r"(sb));
}

// FP16 pair {m, m} of the block multiplier m whose high byte is scale byte b of
// the FRAG_F16 scale word: a byte permute with selector (b<<12)|0x400|(b<<4)|4
// (zero low bytes, byte b in both high bytes)
__device__ __forceinline__ uint32_t f16_scale_sel(int b) { return (uint32_t)((b << 12) | 0x400 | (b << 4) | 4); }

// B fragment of the FP16 path: x16 K order makes the lane's two registers the
// adjacent 8 bytes at logical k 2q..2q+1, 2q+8..2q+9 of K step jj
__device__ __forceinline__ void load_b16(const uint8_t *box, int g, int q, int jj, uint32_t &b0, uint32_t &b1)
{
    const uint2 v = *reinterpret_cast<const uint2 *>(box + g * 128 + (((2 * jj + (q >> 1)) ^ g) << 4) + 8 * (q & 1));
    b0 = v.x;
    b1 = v.y;
}

// 2^k as a float for |k| <= 126
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

// B fragment (k 2q..2q+1 and 2q+8..2q+9 of K step jj inside a 64-wide slice,
// token row g) from a 128-byte-swizzled 8-row box.
__device__ __forceinline__ void load_b(const uint8_t *box, int g, int q, int jj, uint32_t &b0, uint32_t &b1)
{
    const uint8_t *row = box + g * 128 + 4 * q;
    b0 = *reinterpret_cast<const uint32_t *>(row + (((2 * jj) ^ g) << 4));
    b1 = *reinterpret_cast<const uint32_t *>(row + (((2 * jj + 1) ^ g) << 4));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <bool GU, int WFMT, int NT>
__global__ void __launch_bounds__(ST_THREADS, 1)
    gemm_stream_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_b2, const int b3d)
{
    using Cfg = StreamCfg<GU, WFMT, NT>;
    using L = typename Cfg::L;
    constexpr int CH = Cfg::CH, KS = L::KS, R = L::R, NB = L::NB;
    constexpr int NMAX = 8 * NT;
    // MXFP4 weights run on FP16 operands (hardware E2M1 decode), BF16 weights on BF16
    constexpr bool F16 = WFMT == FMT_MXFP4;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF), *empty = full + R;
    float *red = reinterpret_cast<float *>(smem + L::RED_OFF);
    int *prefix = reinterpret_cast<int *>(smem + L::SCHED_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF);
    volatile int *pair_ok = reinterpret_cast<volatile int *>(smem + L::PAIR_OFF);  // [16]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], ST_COMPUTE_WARPS);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 0) {
        schedule_prefix(a.grp_count, a.G, a.row_tiles, NMAX, prefix, lane);
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b2)) : "memory");
        }
    }
    __syncthreads();
    const int total = prefix[a.G];
    const int nst = (a.kchunks + CH - 1) / CH;  // stages per work item

    if (warp == 0) {
        // ---------------------------------------------------------- loader
        uint32_t rc = 0, armed = 0, armed_par = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, a.row_tiles, NMAX);
            const int nt_used = (w.nvalid + 7) / 8;
            int row0 = a.grp_start[w.g] + w.tok0;
            const CUtensorMap *m0 = &map_b;
            if (GU && w.g >= a.E) {  // shared groups read x by token index
                row0 = w.tok0;
                m0 = &map_b2;
            }
            const uint8_t *wsrc =
                a.wbase + (size_t)w.g * a.group_bytes + (size_t)w.rt * a.kchunks * (size_t)a.chunk_bytes;
            for (int s = 0; s < nst; ++s, ++rc) {
                const int slot = rc % R;
                const uint32_t ph = (rc / R) & 1;
                if (!(ok = mbar_wait_warp(&empty[slot], ph ^ 1, abort_flag, a.err, lane)))
                    break;
                if (lane == 0) {
                    uint8_t *st = smem + slot * L::STAGE;
                    const int ch_n = min(CH, a.kchunks - s * CH);
                    const uint32_t wbytes = (uint32_t)(ch_n * a.chunk_bytes);
                    mbar_arrive_expect_tx(&full[slot], wbytes + (uint32_t)(nt_used * NB * KS * BBOX_BYTES));
                    bulk_g2s(st + L::B_BYTES, wsrc + (size_t)s * CH * a.chunk_bytes, wbytes, &full[slot]);
                    for (int nb = 0; nb < NB; ++nb) {
                        const CUtensorMap *m = nb ? &map_b2 : m0;
                        for (int nt = 0; nt < nt_used; ++nt) {
                            uint8_t *dst = st + ((nb * NT + nt) * KS) * BBOX_BYTES;
                            if (b3d) {
                                tma_3d(dst, m, 0, row0 + nt * BBOX_ROWS, s * KS, &full[slot]);
                            } else {
                                for (int ks = 0; ks < KS; ++ks)
                                    tma_2d(dst + ks * BBOX_BYTES, m, (s * KS + ks) * HALF_K, row0 + nt * BBOX_ROWS,
                                           &full[slot]);
                            }
                        }
                    }
                }
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (ph << slot);
            }
        }
        if (lane == 0)
            for (int s = 0; s < R; ++s)
                if (armed & (1u << s))
                    mbar_drain(&full[s], (armed_par >> s) & 1);
        __syncwarp();
    } else {
        // ---------------------------------------------------------- compute warps
        const int cw = warp - 1;
        const int wg = cw & 7, kh = cw >> 3;  // 16-row group, 64-wide half of each chunk
        const int g = lane >> 2, q = lane & 3;
        const uint32_t sel_s0 = f16_scale_sel(2 * kh), sel_s1 = f16_scale_sel(2 * kh + 1);
        float *hmax = red + 8 * NT * 4 * 32;  // [8 warps][8*NT tokens] block maxima of h (FP16 gate|up)
        uint32_t rc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, a.row_tiles, NMAX);
            const int nt_used = NT == 1 ? 1 : (w.nvalid + 7) / 8;
            const int pos0 = a.grp_start[w.g] + w.tok0;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            for (int s = 0; s < nst; ++s, ++rc) {
                const int slot = rc % R;
                if (!(ok = mbar_wait_warp(&full[slot], (rc / R) & 1, abort_flag, a.err, lane)))
                    break;
                const uint8_t *st = smem + slot * L::STAGE;
                const int ch_n = min(CH, a.kchunks - s * CH);
                for (int c = 0; c < ch_n; ++c) {
                    const uint8_t *wch = st + L::B_BYTES + c * L::W_CHUNK;
                    const int ks = 2 * c + kh;  // K slice of this warp inside the stage
                    if (F16) {
                        const uint2 sc =
                            *reinterpret_cast<const uint2 *>(wch + CHUNK_MX_CODE_BYTES + (wg * 8 + g) * 8);
                        const uint4 wv = *reinterpret_cast<const uint4 *>(wch + ((wg * 2 + kh) * 32 + lane) * 16);
                        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
                        // the two 32-element blocks of this warp's half: bytes 2kh, 2kh+1 of each row's scales
                        const uint32_t s_a0 = prmt(sc.x, 0u, sel_s0), s_a1 = prmt(sc.x, 0u, sel_s1);
                        const uint32_t s_b0 = prmt(sc.y, 0u, sel_s0), s_b1 = prmt(sc.y, 0u, sel_s1);
                        // down: h blocks carry their own scale, so each 64-wide slice accumulates apart
                        float part[NT][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            part[nt][0] = part[nt][1] = part[nt][2] = part[nt][3] = 0.f;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            uint32_t af[4];
                            decode_word_f16(words[jj], jj < 2 ? s_a0 : s_a1, jj < 2 ? s_b0 : s_b1, af);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if (nt < nt_used) {
                                    uint32_t b0, b1;
                                    load_b16(st + (nt * KS + ks) * BBOX_BYTES, g, q, jj, b0, b1);
                                    mma_f16(GU ? acc[nt] : part[nt], af, b0, b1);
                                    if (!GU) {
                                        load_b16(st + ((NT + nt) * KS + ks) * BBOX_BYTES, g, q, jj, b0, b1);
                                        mma_f16(part[nt], af, b0, b1);
                                    }
                                }
                            }
                        }
                        if (!GU) {
                            // fold in the scale of this 64-feature block of h for each token column
                            const int slice = 2 * (s * CH + c) + kh;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if (nt < nt_used) {
                                    const int t0 = 8 * nt + 2 * q;
                                    const float f0 = t0 < w.nvalid ? pow2i(a.hs[(size_t)(pos0 + t0) * a.row_tiles_h + slice]) : 0.f;
                                    const float f1 = t0 + 1 < w.nvalid ? pow2i(a.hs[(size_t)(pos0 + t0 + 1) * a.row_tiles_h + slice]) : 0.f;
                                    acc[nt][0] = fmaf(part[nt][0], f0, acc[nt][0]);
                                    acc[nt][1] = fmaf(part[nt][1], f1, acc[nt][1]);
                                    acc[nt][2] = fmaf(part[nt][2], f0, acc[nt][2]);
                                    acc[nt][3] = fmaf(part[nt][3], f1, acc[nt][3]);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const uint4 av =
                                *reinterpret_cast<const uint4 *>(wch + ((wg * 8 + 4 * kh + jj) * 32 + lane) * 16);
                            const uint32_t af[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if (nt < nt_used) {
                                    uint32_t b0, b1;
                                    load_b(st + (nt * KS + ks) * BBOX_BYTES, g, q, jj, b0, b1);
                                    mma_bf16(acc[nt], af, b0, b1);
                                    if (!GU) {
                                        load_b(st + ((NT + nt) * KS + ks) * BBOX_BYTES, g, q, jj, b0, b1);
                                        mma_bf16(acc[nt], af, b0, b1);
                                    }
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[slot]);
            }
            // ------------------------------------------------------ pair reduction (second half -> first)
            // one barrier over all 16 compute warps: the exit decision below is then the
            // same for every compute warp, even after an abort (a warp waiting alone at a
            // named barrier would never be released)
            float *rbuf = red + (size_t)wg * NT * 4 * 32;
            if (lane == 0)
                pair_ok[cw] = ok ? 1 : 0;
            if (kh == 1) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        rbuf[(nt * 4 + i) * 32 + lane] = acc[nt][i];
            }
            named_bar_sync(1, ST_COMPUTE_WARPS * 32);
            if (kh == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[nt][i] += rbuf[(nt * 4 + i) * 32 + lane];
            }
            ok = true;
#pragma unroll
            for (int i = 0; i < ST_COMPUTE_WARPS; ++i)
                ok = ok && pair_ok[i];
            named_bar_sync(1, ST_COMPUTE_WARPS * 32);
            if (!ok)
                break;
            if (kh == 1)
                continue;
            // ------------------------------------------------------ epilogue on the accumulators
            // acc[nt]: [0],[1] = row g, tokens 8nt+2q, +1; [2],[3] = row g+8, same tokens.
            float rf0 = 1.f, rf1 = 1.f;  // undo the per-row rebasing of FP16 weights
            if (F16) {
                const int16_t *rf = a.rfac + ((size_t)w.g * a.row_tiles + w.rt) * TILE_ROWS + 16 * wg + g;
                rf0 = pow2i(rf[0]);
                rf1 = pow2i(rf[8]);
            }
            if (GU) {
                const int n = gu_row_feature(w.rt, 16 * wg + g);  // row g: gate, row g+8: up of feature n
                float hv[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float gv = acc[nt][e], uv = acc[nt][2 + e];
                        const int tok = 8 * nt + 2 * q + e;
                        if (F16) {  // ... and the per-token scaling of x16
                            const float fx = tok < w.nvalid ? pow2i(a.xs[a.row_token[pos0 + tok]]) : 0.f;
                            gv = gv * rf0 * fx;
                            uv = uv * rf1 * fx;
                        }
                        hv[nt][e] = (tok < w.nvalid && n < a.I) ? gv / (1.0f + __expf(-gv)) * uv : 0.f;
                    }
                if (F16) {
                    // h leaves as FP16 hi + lo scaled by 2^-hs, hs per (position, 64-feature block):
                    // block maximum over the 8 features of each warp (lanes g), then over the 8 warps
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float m = fabsf(hv[nt][e]);
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            if (g == 0)
                                hmax[wg * 8 * NT + 8 * nt + 2 * q + e] = m;
                        }
                    named_bar_sync(9, 8 * 32);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = 8 * nt + 2 * q + e;
                            float m = 0.f;
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                m = fmaxf(m, hmax[i * 8 * NT + tok]);
                            const int mb = (int)((__float_as_uint(m) >> 23) & 0xFFu);
                            int hsc = m > 0.f ? mb - 127 - 14 : 0;
                            hsc = hsc < -100 ? -100 : (hsc > 100 ? 100 : hsc);
                            if (tok < w.nvalid) {
                                const float v = hv[nt][e] * pow2i(-hsc);
                                const __half hb = __float2half_rn(v);
                                const __half lb = __float2half_rn(v - __half2float(hb));
                                if (n < a.I) {
                                    const size_t o = (size_t)(pos0 + tok) * a.I + (n & ~15) + x16_phys_k(n & 15);
                                    a.h_out[o] = __half_as_ushort(hb);
                                    a.h_out[o + a.h_plane] = __half_as_ushort(lb);
                                }
                                if (wg == 0 && g == 0)
                                    a.hs[(size_t)(pos0 + tok) * a.row_tiles + w.rt] = hsc;
                            }
                        }
                    named_bar_sync(9, 8 * 32);  // hmax is reused by the next work item
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = 8 * nt + 2 * q + e;
                            if (tok < w.nvalid && n < a.I) {
                                const float v = hv[nt][e];
                                const __nv_bfloat16 hb = __float2bfloat16_rn(v);
                                const __nv_bfloat16 lb = __float2bfloat16_rn(v - __bfloat162float(hb));
                                const size_t o = (size_t)(pos0 + tok) * a.I + n;
                                a.h_out[o] = __bfloat16_as_ushort(hb);
                                a.h_out[o + a.h_plane] = __bfloat16_as_ushort(lb);
                            }
                        }
                }
            } else {
                const int m = w.rt * TILE_ROWS + 16 * wg + g;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = 8 * nt + 2 * q + e;
                        if (tok < w.nvalid) {
                            float *yrow = a.y_out + (size_t)(pos0 + tok) * a.H;
                            if (m < a.H)
                                yrow[m] = acc[nt][e] * rf0;
                            if (m + 8 < a.H)
                                yrow[m + 8] = acc[nt][2 + e] * rf1;
                        }
                    }
            }
        }
    }
    __syncthreads();
}

template <bool GU, int WFMT, int NT>
cudaError_t launch_stream_cfg(const GemmArgs &a, const void *b1, long long rows1, const void *b2, long long rows2,
                              int K, cudaStream_t st)
{
    using Cfg = StreamCfg<GU, WFMT, NT>;
    using L = typename Cfg::L;
    // token rows: a 3-D map (one copy per 8-token tile per stage) when the row
    // pitch is a whole number of 64-wide slices, else 2-D boxes per slice
    const int b3d = K % 64 == 0;
    CUtensorMap m1, m2;
    cudaError_t e = b3d ? make_map_3d(&m1, b1, rows1, K, BBOX_ROWS, L::KS) : make_map(&m1, b1, rows1, K, BBOX_ROWS);
    if (e != cudaSuccess)
        return e;
    e = b3d ? make_map_3d(&m2, b2, rows2, K, BBOX_ROWS, L::KS) : make_map(&m2, b2, rows2, K, BBOX_ROWS);
    if (e != cudaSuccess)
        return e;
    auto kern = gemm_stream_kernel<GU, WFMT, NT>;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    kern<<<sm_count(), ST_THREADS, L::TOTAL, st>>>(a, m1, m2, b3d);
    return cudaGetLastError();
}

// token tile: 8*NT tokens, NT the smallest power of two covering min(T, 64)
template <bool GU, int WFMT>
cudaError_t launch_stream_nt(const GemmArgs &a, int T, const void *b1, long long rows1, const void *b2,
                             long long rows2, int K, cudaStream_t st)
{
    const int t = T < STREAM_MAX_T ? T : STREAM_MAX_T;
    if (t <= 8)
        return launch_stream_cfg<GU, WFMT, 1>(a, b1, rows1, b2, rows2, K, st);
    if (t <= 16)
        return launch_stream_cfg<GU, WFMT, 2>(a, b1, rows1, b2, rows2, K, st);
    if (t <= 32)
        return launch_stream_cfg<GU, WFMT, 4>(a, b1, rows1, b2, rows2, K, st);
    return launch_stream_cfg<GU, WFMT, 8>(a, b1, rows1, b2, rows2, K, st);
}

}  // namespace

cudaError_t launch_gemm_gate_up_stream(const Plan &p, const WeightStore &w, int fmt, const uint16_t *x,
                                       cudaStream_t st)
{
    GemmArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.row_tiles, p.grp_start, p.grp_count, p.E, p.G,
               p.I, p.H, p.h, (long long)p.P * p.I, nullptr, p.err, w.rfac, p.xs, p.row_token, p.hs, w.row_tiles};
    // MXFP4 weights: FP16 tokens (x16 / its gathered rows); BF16 weights: BF16 tokens
    const void *xt = fmt == FMT_MXFP4 ? (const void *)p.x16 : (const void *)x;
    const long long routed = (long long)p.T * p.k;
    const void *b1 = routed > 0 ? (const void *)p.x_perm : xt;
    const long long r1 = routed > 0 ? routed : p.T;
    return fmt == FMT_MXFP4 ? launch_stream_nt<true, FMT_MXFP4>(a, p.T, b1, r1, xt, p.T, p.H, st)
                            : launch_stream_nt<true, FMT_BF16>(a, p.T, b1, r1, xt, p.T, p.H, st);
}

cudaError_t launch_gemm_down_stream(const Plan &p, const WeightStore &w, int fmt, cudaStream_t st)
{
    GemmArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.row_tiles, p.grp_start, p.grp_count, p.E, p.G,
               p.I, p.H, nullptr, 0, p.y, p.err, w.rfac, nullptr, nullptr, p.hs, (p.I + 63) / 64};
    const void *lo = p.h + (size_t)p.P * p.I;
    return fmt == FMT_MXFP4 ? launch_stream_nt<false, FMT_MXFP4>(a, p.T, p.h, p.P, lo, p.P, p.I, st)
                            : launch_stream_nt<false, FMT_BF16>(a, p.T, p.h, p.P, lo, p.P, p.I, st);
}

}  // namespace moe
