// layer_stream.cu -- the whole MoE layer (routed or dense-as-slices) for
// decode-sized batches in one persistent kernel: routing, grouping, gate|up
// with SwiGLU, down and the weighted combine.  At a handful of tokens per
// expert the layer is bound by reading each active expert's weights once from
// HBM, so the kernel is built around one uninterrupted weight stream per SM.
//
// Operations (SwiGLU experts, shared experts with unit weight and the weighted
// reduction of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1
// and §3.3 Eq. 1; dense FFN as all-active slices, §3.4 Eq. 2; MXFP4 decoded
// inside the reduction as in "DeepSeek-V4-Flash on a four-GPU Ampere
// workstation", section "MXFP4 is not NVFP4, and the difference matters on
// Ampere"; group-32 INT4 with FP16 group scales and zero points, the format of
// the same Cascadia paper's §3.1, decoded the same way):
//
//  phase 0a  tokens are routed (softmax top-k, renormalised; or the caller's
//            ids and weights are copied and checked) and their FP16 rows x16
//            written (per-token power-of-two scale).  With at most 8 tokens
//            every CTA routes every token itself; otherwise each CTA routes
//            its own and a grid-wide counter tells every CTA when all are done.
//  phase 0b  every CTA builds the expert histogram, positions and the stable
//            permutation in shared memory (CTA 0 also publishes them), then
//            the work list: (gate|up, group, 128-row tile, token tile) items
//            followed by (down, ...) items.
//  stream    warp 0 takes items from a grid-wide counter and streams each
//            item's weight chunks (one bulk copy per stage) plus its token
//            rows (one bulk copy per row and plane) into a ring of
//            shared-memory stages sized by the item's tile class; 8 compute
//            warps (16 weight rows each, the full K) decode MXFP4 or INT4 in
//            registers straight into warp-level MMA fragments (FP16 operands,
//            FP32 accumulation, the E8M0 or FP16 block scales applied in FP32
//            to each 32-wide block's partial sum).  gate|up epilogues write h
//            (one FP16 plane, scaled by a power of two per 64-feature block;
//            BF16 hi + lo planes for BF16 weights) and hand the item to warp
//            9, which publishes it to the other CTAs with one release; a
//            down item's token rows are copied only once its group's h is
//            complete, while its weights are already streaming.
//  combine   once every CTA has counted its items done, all warps of the
//            grid sum (token, 128-feature) blocks of y into out in a fixed
//            order (j ascending, then shared groups), so the result does not
//            depend on which CTA did what.
//
// The grid is one CTA per SM, launched cooperatively so that all CTAs are
// resident: CTAs wait on each other only through counters in the caller's
// workspace, and every such wait -- like every mbarrier wait -- is bounded in
// time; on expiry the kernel records DEV_ERR_WAIT_TIMEOUT and leaves.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "gemm_common.cuh"
#include "mx_decode.cuh"

namespace moe {

namespace {

using namespace gemm;

// warp 0 streams, warps 1..8 compute (one 16-row group each), warp 9 publishes
// finished gate|up items to the other CTAs
constexpr int LS_WARPS = 10;
constexpr int LS_THREADS = LS_WARPS * 32;
constexpr int LS_COMPUTE_WARPS = 8;
constexpr int LS_PUB_R = 4;  // hand-off slots between the compute warps and the publisher
// CTAs per SM.  Two CTAs (two independent streams, four compute warps per
// sub-partition, 112 registers, half the ring each) measured slower than one
// CTA with 168 registers for every token tile, so all tiles run one.
__host__ __device__ constexpr int ls_ctas_per_sm(int /*nt*/) { return 1; }
__host__ __device__ constexpr int ls_smem_limit(int ctas) { return ctas == 1 ? 232448 : 114688; }
__host__ __device__ constexpr int ls_stage_target(int ctas) { return ctas == 1 ? 52224 : 26624; }
constexpr int LS_R_MAX = 16;
// stage target of the kernel for batches of at most two tokens (NT = 0): its
// stages reserve two token rows, which leaves room for one more ring slot.
// Group-32 INT4 chunks are larger (9,728 B against 8,704); its target still
// takes four of them per gate|up stage.
constexpr int LS_TINY_TARGET = 40960;
constexpr int LS_TINY_TARGET_I4 = 41088;
constexpr int LS_HS_ROW = 16;  // ints of h block scales kept per token row and stage
// L2 prefetch at kernel entry of the leading shared groups' gate|up weights:
// at most this many bytes over the grid, in pieces of LS_PF_PIECE
constexpr size_t LS_PF_BYTES = 24u << 20;
constexpr uint32_t LS_PF_PIECE = 32768;

// ------------------------------------------------------------------ stage geometry
//
// A stage holds, in this order: NB token operands of ROWS rows each, row r at
// r * rowb(CH) bytes (CH*2 64-wide K slices of 128 bytes, then 32 bytes of
// padding so that the 8 rows an MMA fragment reads fall on distinct banks);
// for the FP16 down GEMM the rows' h block scales (LS_HS_ROW ints per row);
// then CH weight chunks.
__host__ __device__ constexpr int ls_rowb(int ch) { return ch * 256 + 32; }
__host__ __device__ constexpr int ls_stage_bytes(int nb, int rows, int hsb, int ch, int wchunk)
{
    return nb * rows * ls_rowb(ch) + hsb + ch * wchunk;
}
__host__ __device__ constexpr int ls_pick_ch(int nb, int rows, int hsb, int wchunk, int target)
{
    return ls_stage_bytes(nb, rows, hsb, 4, wchunk) <= target   ? 4
           : ls_stage_bytes(nb, rows, hsb, 2, wchunk) <= target ? 2
                                                                : 1;
}
__host__ __device__ constexpr int ls_max(int a, int b) { return a > b ? a : b; }

// Items hold up to 8 * NT tokens (NT = the kernel's token tiles; NT = 0 is the
// kernel for batches of at most two tokens, with one tile).  An item of c
// tokens runs the code and stage geometry of its own tile class NTI (the
// smallest power of two with 8 * NTI >= c): a token operand of res_rows(NTI)
// reserved rows (8 * NTI; two in the NT = 0 kernel, whose MMAs read the other
// six rows of their 8-token tile from the bytes that follow, in the same
// stage, and discard those columns) and as many weight chunks per stage as
// then fit the stage target.
template <int WFMT, int NT>
struct LsCfg {
    static constexpr bool F16 = WFMT != FMT_BF16;  // MXFP4 and INT4 codes run FP16 MMAs
    static constexpr int W_CHUNK = WFMT == FMT_MXFP4  ? CHUNK_MX_BYTES
                                   : WFMT == FMT_INT4 ? CHUNK_I4_BYTES
                                                      : CHUNK_BF16_BYTES;
    static constexpr int NTK = NT == 0 ? 1 : NT;  // token tiles of the largest item
    static constexpr int ROWS = 8 * NTK;          // token rows of the largest item
    static constexpr int CTAS = ls_ctas_per_sm(NT);
    static constexpr int SMEM_LIMIT = ls_smem_limit(CTAS);
    static constexpr int TARGET = NT == 0 ? (WFMT == FMT_INT4 ? LS_TINY_TARGET_I4 : LS_TINY_TARGET)
                                          : ls_stage_target(CTAS);
    // token operands of a down stage: one FP16 plane of h (MXFP4, INT4), or the
    // BF16 hi and lo planes (BF16 weights)
    static constexpr int NB_DN = F16 ? 1 : 2;
    __host__ __device__ static constexpr int res_rows(int nti) { return NT == 0 ? 2 : 8 * nti; }
    __host__ __device__ static constexpr int hsb_dn(int nti) { return F16 ? res_rows(nti) * LS_HS_ROW * 4 : 0; }
    __host__ __device__ static constexpr int ch_gu(int nti)
    {
        return ls_pick_ch(1, res_rows(nti), 0, W_CHUNK, TARGET);
    }
    __host__ __device__ static constexpr int ch_dn(int nti)
    {
        return ls_pick_ch(NB_DN, res_rows(nti), hsb_dn(nti), W_CHUNK, TARGET);
    }
    __host__ __device__ static constexpr int stage_of(int nti)
    {
        return ls_max(ls_stage_bytes(1, res_rows(nti), 0, ch_gu(nti), W_CHUNK),
                      ls_stage_bytes(NB_DN, res_rows(nti), hsb_dn(nti), ch_dn(nti), W_CHUNK));
    }
    static constexpr int STAGE = (ls_max(ls_max(stage_of(1), NT >= 2 ? stage_of(2) : 0),
                                         ls_max(NT >= 4 ? stage_of(4) : 0, NT >= 8 ? stage_of(8) : 0)) +
                                  127) / 128 * 128;
    static constexpr int RED_BYTES = 0;
    static constexpr int HMAX_BYTES = 2 * 8 * ROWS * 4;    // block maxima of h, double-buffered
};

// tile class of an item of c tokens in a kernel of NT token tiles
template <int NT>
__device__ __forceinline__ int ls_nti(int c)
{
    if (NT <= 1)
        return 1;
    const int t = (c + 7) >> 3;
    return t <= 1 ? 1 : t <= 2 ? (NT < 2 ? NT : 2) : t <= 4 ? (NT < 4 ? NT : 4) : NT;
}

// Shared-memory carve-up (bytes from the 1024-aligned base).  The ring comes
// first; phase 0 uses it as scratch before the first copy is issued.
struct LsSmem {
    int hdr, bars, pbars, misc, red, hmax, gcnt, gstart, tpre, sorted, xs, gdone, total;
};

__host__ __device__ inline LsSmem ls_smem(int R, int G, int n, int T, int stage, int red_bytes, int hmax_bytes)
{
    LsSmem s;
    int o = R * stage;
    s.hdr = o;
    o += LS_R_MAX * 8;
    s.bars = o;
    o += 2 * LS_R_MAX * 8;
    s.pbars = o;
    o += 24 * 8;
    s.misc = o;
    o += 64;
    s.red = o;
    o += red_bytes;
    s.hmax = o;
    o += hmax_bytes;
    s.gcnt = o;
    o += G * 4;
    s.gstart = o;
    o += G * 4;
    s.tpre = o;
    o += (G + 1) * 4;
    s.sorted = o;
    o += (n > 0 ? n : 1) * 4;
    s.xs = o;
    o += T * 4;
    s.gdone = o;
    o += ((G + 31) / 32) * 4;
    s.total = o + 1024;  // room to align the dynamic base to 1024
    return s;
}

// sync block (ints of the caller's workspace, zeroed before every launch)
constexpr int SY_ROUTED = 0;  // tokens routed and prepared
constexpr int SY_PERM = 1;    // 1 once CTA 0 has published the permutation
constexpr int SY_WORK = 2;    // next work item
constexpr int SY_DONE = 3;    // CTAs whose items are all finished
constexpr int SY_GRP = 16;    // [G] gate|up warps finished per group

struct LayerArgs {
    const uint8_t *wgu, *wdn;
    size_t gu_group_bytes, dn_group_bytes;
    int gu_kchunks, dn_kchunks, gu_row_tiles, dn_row_tiles, chunk_bytes;
    int T, k, E, S, G, H, I, n;
    const uint16_t *x;
    const float *logits;
    const int *ids_in;   // routing given by the caller (ids, weights) instead of logits, or NULL
    int ebase, etotal;   // caller routing: the groups 0..E-1 are expert ids [ebase, ebase + E) of etotal
    const float *w_in;
    int *topk_ids;
    float *topk_w;
    int *expert_offsets, *sorted_slot, *slot_pos;
    uint16_t *x16;
    int *xs;
    uint16_t *h;
    long long h_plane;
    int *hs;
    int hs_pitch;
    float *y, *out;
    int accumulate;
    int *sync;
    int *err;
    int R;
    // the grid-wide completion wait before the combine: extra count on its
    // target and its time limit (0 and WAIT_LIMIT_NS in every normal launch;
    // a test of the expiry path raises the target past reach)
    int done_extra;
    unsigned long long done_wait_ns;
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// m16n8k16 FP16 MMA with a zero C operand: d = A * B
__device__ __forceinline__ void mma_f16_z(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// Two E8M0 block scales (bytes 2H and 2H+1 of w) -> the BF16 pair of 2^(e-127)
// (e = 0 gives the subnormal 2^-127, exactly), low byte in the low half.
template <int H>
__device__ __forceinline__ uint32_t ue8m0x2_bf16x2(uint32_t w)
{
    uint32_t d;
    if (H == 0)
        asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.bf16x2.ue8m0x2 %0, lo;\n}" : "=r"(d) : "r"(w));
    else
        asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.bf16x2.ue8m0x2 %0, hi;\n}" : "=r"(d) : "r"(w));
    return d;
}

// FRAG_F16 word -> A fragment: each byte (two OCP E2M1 codes) converts to an
// FP16 pair in hardware; values are the unscaled v(c) (exact in FP16).
__device__ __forceinline__ void decode_e2m1(uint32_t w, uint32_t out[4])
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// FRAG_F16 word of group-32 INT4 codes -> A fragment.  Pair p holds its first
// code in nibble p and its second in nibble p + 4; 0x6400 | q is the FP16
// value 1024 + q (ulp 1 there), so subtracting 1024 + z leaves q - z exactly.
// Pairs 0 and 2 belong to row g (zero point za), pairs 1 and 3 to row g + 8 (zb).
__device__ __forceinline__ void decode_i4(uint32_t w, uint32_t za, uint32_t zb, uint32_t out[4])
{
    const uint32_t ma = (0x6400u + za) * 0x10001u, mb = (0x6400u + zb) * 0x10001u;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t v = ((w >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(out[p]) : "r"(v), "r"((p & 1) ? mb : ma));
    }
}

// FP16 half H of w (H = 0: low) widened to FP32, exactly.
template <int H>
__device__ __forceinline__ float f16_half_to_f32(uint32_t w)
{
    float f;
    if (H == 0)
        asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, lo;\n}" : "=f"(f) : "r"(w));
    else
        asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, hi;\n}" : "=f"(f) : "r"(w));
    return f;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// B fragment: token rows hold K in the x16 order, so a lane's two registers
// (logical k 2q..2q+1 and 2q+8..2q+9 of a 16-wide K step) are 8 adjacent bytes
__device__ __forceinline__ void load_b(const uint8_t *p, uint32_t &b0, uint32_t &b1)
{
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    b0 = v.x;
    b1 = v.y;
}

// 2^k as a float for |k| <= 126
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// bring [p, p + bytes) into L2 (16-byte aligned address, size a multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_release(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add(int *p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (one thread) until *p >= target, with acquire semantics.
// Gives up after limit_ns (recording DEV_ERR_WAIT_TIMEOUT) or when the CTA's
// abort flag is raised.
__device__ __noinline__ bool wait_geq(const int *p, int target, volatile int *abort_flag, int *err,
                                      uint64_t limit_ns = WAIT_LIMIT_NS)
{
    if (ld_acquire(p) >= target)
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (ld_acquire(p) >= target)
            return true;
        if ((i & 15u) == 0) {
            if (abort_flag && *abort_flag)
                return false;
            if (global_ns() - t0 > limit_ns) {
                atomicCAS(err, 0, DEV_ERR_WAIT_TIMEOUT);
                if (abort_flag)
                    *abort_flag = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ phase 0a
//
// Warps 0..3 route (one warp per token, no barrier) while warps 4..8 prepare
// token rows (LS_PREP_THREADS threads, named barrier 2).  Token t belongs to
// CTA t mod gridDim.x, which writes its routing outputs and its x16 row.
// With few tokens (T <= LS_LOCAL_ROUTE_T) every CTA routes every token itself
// so that it can build the schedule without waiting for the other CTAs; only
// the token rows are then awaited, by the loader, before its first token copy.
constexpr int LS_ROUTE_WARPS = 4;
constexpr int LS_ROUTE_THREADS = LS_ROUTE_WARPS * 32;
constexpr int LS_PREP_THREADS = LS_THREADS - LS_ROUTE_THREADS;
constexpr int LS_SCRATCH_PREP = 9216;  // byte offset of the prep scratch (after the schedule's slot ids)
constexpr int LS_LOCAL_ROUTE_T = 8;
constexpr int LS_KEYS_PER_LANE = LS_MAX_EXPERTS / 32;

// Order key of a logit: larger float -> larger key; +0 and -0 equal; NaN
// below every number.
__device__ __forceinline__ uint32_t ls_logit_key(float f)
{
    if (isnan(f))
        return 0u;
    if (f == 0.0f)
        f = 0.0f;
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// the logit of an order key (a NaN key gives a NaN)
__device__ __forceinline__ float ls_key_logit(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Route token t with one warp: softmax top-k, renormalised over the kept k.
// Lane l holds experts e = l + 32 i as order key + 1 (0: absent or taken).
// Round j takes the largest key of the warp (redux max) and, among the
// experts holding it, the lowest index (redux min), so "larger logit, then
// lower index" is the selection order.  Weights: w_j = exp(l_j - l_0) /
// sum_{j' < k} exp(l_j' - l_0), l_0 the largest kept logit.  The expert ids
// go to ids_s[t * k + j] when ids_s is given, and the owner CTA writes both
// outputs to the caller's arrays.
__device__ void ls_route_warp(const LayerArgs &a, int t, int lane, int *ids_s, bool owner)
{
    const float *row = a.logits + (size_t)t * a.E;
    uint32_t key[LS_KEYS_PER_LANE];
#pragma unroll
    for (int i = 0; i < LS_KEYS_PER_LANE; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < a.E ? ls_logit_key(__ldg(row + e)) + 1u : 0u;
    }
    int my_e = 0;
    uint32_t my_key = 0;
    for (int j = 0; j < a.k; ++j) {
        uint32_t best = 0;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < LS_KEYS_PER_LANE; ++i)
            if (key[i] > best) {  // strict: the lowest i (lowest expert of the lane) among equals
                best = key[i];
                bi = i;
            }
        const uint32_t m = __reduce_max_sync(0xffffffffu, best);
        const uint32_t mine = lane + 32 * bi;
        const uint32_t ew = __reduce_min_sync(0xffffffffu, best == m ? mine : 0xFFFFFFFFu);
        if (mine == ew) {
#pragma unroll
            for (int i = 0; i < LS_KEYS_PER_LANE; ++i)
                if (i == bi)
                    key[i] = 0;
        }
        if (lane == j) {
            my_e = (int)ew;
            my_key = m - 1u;
        }
    }
    const float my_v = lane < a.k ? ls_key_logit(my_key) : 0.f;
    const float l0 = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < a.k ? expf(my_v - l0) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < a.k) {
        if (ids_s)
            ids_s[t * a.k + lane] = my_e;
        if (owner) {
            a.topk_ids[(size_t)t * a.k + lane] = my_e;
            a.topk_w[(size_t)t * a.k + lane] = ex / sum;
        }
    }
}

// Routing given by the caller for token t (one warp): lane j < k takes its id
// and weight.  Ids are global: the layer holds experts [ebase, ebase + E) of
// etotal as its groups 0..E-1.  Id -1, or an expert held elsewhere, is an
// empty slot (id -1, weight 0); any other id outside [0, etotal) records
// DEV_ERR_BOUNDS and becomes group 0 with weight 0, so that the layer stays in
// bounds.  The ids go to ids_s when
// given, and the owner CTA writes both to the call's routing arrays.
__device__ void ls_copy_route_warp(const LayerArgs &a, int t, int lane, int *ids_s, bool owner)
{
    if (lane < a.k) {
        int e = __ldg(a.ids_in + (size_t)t * a.k + lane);
        float wv = __ldg(a.w_in + (size_t)t * a.k + lane);
        if (e == -1) {
            wv = 0.f;
        } else if (e < 0 || e >= a.etotal) {
            atomicCAS(a.err, 0, DEV_ERR_BOUNDS);
            e = 0;
            wv = 0.f;
        } else if (e < a.ebase || e - a.ebase >= a.E) {
            e = -1;
            wv = 0.f;
        } else {
            e -= a.ebase;
        }
        if (ids_s)
            ids_s[t * a.k + lane] = e;
        if (owner) {
            a.topk_ids[(size_t)t * a.k + lane] = e;
            a.topk_w[(size_t)t * a.k + lane] = wv;
        }
    }
}

// Token row t for the GEMMs, in the x16 K order (physical element 4q + c of
// every 16-element group holds logical element 2q + (c & 1) + 8 * (c >> 1)),
// by threads LS_ROUTE_THREADS.. of the CTA.
// MXFP4 weights: FP16 x_t * 2^-xs[t] with xs[t] = floor(log2 max|x_t|) - 14
// (0 for an all-zero row, clamped to [-100, 100]); a BF16 value has 8
// significant bits and FP16 11, so the conversion is exact for every element
// within 2^17 of the row's largest.  BF16 weights: the BF16 row unchanged.
template <bool F16>
__device__ void ls_prep_token(const LayerArgs &a, int t, uint8_t *scratch)
{
    const int pt = threadIdx.x - LS_ROUTE_THREADS;
    const uint4 *row = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H);
    const int ngr = a.H / 16;  // 16-element groups (H is a multiple of 32)
    float mul = 1.f;
    if (F16) {
        uint32_t *red = reinterpret_cast<uint32_t *>(scratch);
        uint32_t mx = 0;  // max |x| as BF16 bits without sign (monotonic for finite values)
        for (int i = pt; i < 2 * ngr; i += LS_PREP_THREADS) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        }
        for (int o = 16; o > 0; o >>= 1)
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((pt & 31) == 0)
            red[pt >> 5] = mx;
        named_bar_sync(2, LS_PREP_THREADS);
        mx = 0;
        for (int i = 0; i < LS_PREP_THREADS / 32; ++i)
            mx = max(mx, red[i]);
        int sc = mx == 0 ? 0 : (int)(mx >> 7) - 127 - 14;
        sc = sc < -100 ? -100 : (sc > 100 ? 100 : sc);
        if (pt == 0)
            a.xs[t] = sc;
        mul = ldexpf(1.0f, -sc);
        named_bar_sync(2, LS_PREP_THREADS);  // red is reused by the next token
    }
    uint4 *dst = reinterpret_cast<uint4 *>(a.x16 + (size_t)t * a.H);
    for (int gi = pt; gi < ngr; gi += LS_PREP_THREADS) {
        const uint4 v0 = row[2 * gi], v1 = row[2 * gi + 1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint16_t hv[16];
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const uint32_t b = (w[kk >> 1] >> (16 * (kk & 1))) & 0xFFFFu;
            hv[kk] = F16 ? __half_as_ushort(__float2half_rn(__uint_as_float(b << 16) * mul)) : (uint16_t)b;
        }
        uint32_t o[8];
#pragma unroll
        for (int p2 = 0; p2 < 8; ++p2)
            o[p2] = (uint32_t)hv[x16_logical_k(2 * p2)] | (uint32_t)hv[x16_logical_k(2 * p2 + 1)] << 16;
        dst[2 * gi] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * gi + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ------------------------------------------------------------------ phase 0b

// Work-list order of the groups: the shared groups (or dense slices) first, then
// the routed experts in index order.  The shared groups' items do not depend on
// the routing, so their weights can start moving before it is done.
__device__ __forceinline__ int ls_group_of(int j, int E, int G) { return j < G - E ? E + j : j - (G - E); }

// Groups, positions, token tiles and (routed) the stable permutation, in
// shared memory.  Positions: routed slots 0..n-1 in expert-major order (slots
// of one expert in ascending slot order s = t*k + j), then shared group s at
// n + s*T + t.  An empty slot (id -1, from caller routing) takes no position;
// the routed positions from expert_offsets[E] to n are then left unused.  gcnt[g] / gstart[g]: tokens and first position of group g;
// tpre[j]: first token tile of the j-th group in work-list order (ls_group_of;
// a group of c tokens has ceil(c/ROWS) tiles); sorted[p]: slot at routed
// position p, replaced by its token once CTA 0 has published the permutation;
// xs_s[t]: the x16 scales.
template <int ROWS, bool F16>
__device__ void ls_schedule(const LayerArgs &a, uint8_t *scratch, int *gcnt, int *gstart, int *tpre, int *sorted,
                            int *xs_s, bool local)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, E = a.E, G = a.G;
    int *sid = reinterpret_cast<int *>(scratch);  // slot ids (local routing: already here)
    int *wtot = sid + ((n + 3) & ~3);     // [LS_WARPS][2] warp totals of the group scan
    int *wc = wtot + 2 * LS_WARPS;        // [LS_WARPS][E] per-warp running positions
    for (int g = tid; g < G; g += LS_THREADS)
        gcnt[g] = g < E ? 0 : a.T;
    if (!local) {
        for (int s = tid; s < n; s += LS_THREADS)
            sid[s] = __ldcg(a.topk_ids + s);
        // (local routing: the loader fills xs_s once the token rows are ready)
        if (F16)
            for (int t = tid; t < a.T; t += LS_THREADS)
                xs_s[t] = __ldcg(a.xs + t);
    }
    __syncthreads();
    for (int s = tid; s < n; s += LS_THREADS)
        if (sid[s] >= 0)
            atomicAdd(&gcnt[sid[s]], 1);
    __syncthreads();
    // group scan in work-list order: positions (routed groups only, which keeps
    // them in expert order) and token tiles, 32 groups per warp, LS_WARPS * 32
    // groups per round
    int base_pos = 0, base_tiles = 0;
    for (int g0 = 0; g0 < G; g0 += LS_WARPS * 32) {
        const int j = g0 + warp * 32 + lane;
        const int g = j < G ? ls_group_of(j, E, G) : G;
        const int c = j < G ? gcnt[g] : 0;
        const int cp = g < E ? c : 0;
        const int tl = (c + ROWS - 1) / ROWS;
        int ip = cp, it = tl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vp = __shfl_up_sync(0xffffffffu, ip, o), vt = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                ip += vp;
                it += vt;
            }
        }
        if (lane == 31) {
            wtot[2 * warp] = ip;
            wtot[2 * warp + 1] = it;
        }
        __syncthreads();
        int op = base_pos, ot = base_tiles, tp = 0, tt = 0;
        for (int w = 0; w < LS_WARPS; ++w) {
            if (w < warp) {
                op += wtot[2 * w];
                ot += wtot[2 * w + 1];
            }
            tp += wtot[2 * w];
            tt += wtot[2 * w + 1];
        }
        if (j < G) {
            gstart[g] = g < E ? op + ip - cp : n + (g - E) * a.T;
            tpre[j] = ot + it - tl;
        }
        base_pos += tp;
        base_tiles += tt;
        __syncthreads();
    }
    if (tid == 0)
        tpre[G] = base_tiles;
    if (E == 0 || n == 0) {
        __syncthreads();
        return;
    }
    // stable permutation
    if (n <= 2048) {
        // one warp, 32 slots per step, a running position per expert
        for (int e = tid; e < E; e += LS_THREADS)
            wc[e] = gstart[e];
        __syncthreads();
        if (warp == 0) {
            for (int base = 0; base < n; base += 32) {
                const int s = base + lane;
                const int e = s < n ? sid[s] : -1;
                const bool act = e >= 0;
                const unsigned m = __match_any_sync(0xffffffffu, e);
                if (act)
                    sorted[wc[e] + __popc(m & ((1u << lane) - 1u))] = s;
                __syncwarp();
                if (act && lane == 31 - __clz(m))
                    wc[e] += __popc(m);
                __syncwarp();
            }
        }
    } else {
        // every warp owns slots [lo, hi): per-warp counts per expert, turned
        // into each warp's first position per expert, then every warp places
        // its slots in order
        const int lo = (int)((long long)warp * n / LS_WARPS), hi = (int)((long long)(warp + 1) * n / LS_WARPS);
        int *my = wc + warp * E;
        for (int e = lane; e < E; e += 32)
            my[e] = 0;
        __syncwarp();
        for (int s = lo + lane; s < hi; s += 32)
            if (sid[s] >= 0)
                atomicAdd(&my[sid[s]], 1);
        __syncthreads();
        for (int e = tid; e < E; e += LS_THREADS) {
            int run = gstart[e];
            for (int w = 0; w < LS_WARPS; ++w) {
                const int c = wc[w * E + e];
                wc[w * E + e] = run;
                run += c;
            }
        }
        __syncthreads();
        for (int base = lo; base < hi; base += 32) {
            const int s = base + lane;
            const int e = s < hi ? sid[s] : -1;
            const bool act = e >= 0;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (act)
                sorted[my[e] + __popc(m & ((1u << lane) - 1u))] = s;
            __syncwarp();
            if (act && lane == 31 - __clz(m))
                my[e] += __popc(m);
            __syncwarp();
        }
    }
    // (base_pos: the routed positions taken, n less the empty slots)
    for (int p = base_pos + tid; p < n; p += LS_THREADS)
        sorted[p] = -1;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = tid; e <= E; e += LS_THREADS)
            a.expert_offsets[e] = e < E ? gstart[e] : base_pos;
        for (int p = tid; p < n; p += LS_THREADS) {
            const int s = sorted[p];
            a.sorted_slot[p] = s;
            if (s >= 0)
                a.slot_pos[s] = p;
        }
        for (int s = tid; s < n; s += LS_THREADS)
            if (sid[s] < 0)
                a.slot_pos[s] = -1;
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            st_release(&a.sync[SY_PERM], 1);
        }
    }
    // from here on the GEMMs need only each routed position's token
    __syncthreads();
    for (int p = tid; p < n; p += LS_THREADS)
        sorted[p] = sorted[p] < 0 ? 0 : sorted[p] / a.k;
}

// ------------------------------------------------------------------ work items

struct LsItem {
    bool gu;
    int g, rt, tok0, nvalid, pos0;
    int ntl;  // token tiles of the group
};

// Item u: gate|up items u < total_gu, then down items, groups in work-list
// order.  Items of one group are ordered row tile major, token tile minor; a
// group of c tokens in ntiles tiles gives each tile ceil(c / ntiles) tokens
// rounded up to 8.
template <int ROWS>
__device__ __forceinline__ LsItem ls_item(int u, int total_gu, int rt_gu, int rt_dn, int E, int G, const int *gcnt,
                                          const int *gstart, const int *tpre)
{
    LsItem it;
    it.gu = u < total_gu;
    if (!it.gu)
        u -= total_gu;
    const int rtn = it.gu ? rt_gu : rt_dn;
    const int v = u / rtn;
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tpre[mid] <= v)
            lo = mid;
        else
            hi = mid;
    }
    it.g = ls_group_of(lo, E, G);
    const int ntiles = tpre[lo + 1] - tpre[lo];
    it.ntl = ntiles;
    const int local = u - tpre[lo] * rtn;
    it.rt = local / ntiles;
    const int tt = local % ntiles;
    const int cnt = gcnt[it.g];
    const int per = ((cnt + ntiles - 1) / ntiles + 7) & ~7;
    it.tok0 = tt * per;
    it.nvalid = min(per, cnt - it.tok0);
    it.pos0 = gstart[it.g] + it.tok0;
    return it;
}

// tile class of an item
template <int WFMT, int NT>
__device__ __forceinline__ int ls_nti_item(const LsItem &it)
{
    return ls_nti<NT>(it.nvalid);
}

// token of row r of an item: routed positions look it up (tokp: token of each
// routed position); a shared group or dense slice holds every token in order
__device__ __forceinline__ int ls_row_token(const LayerArgs &a, const int *tokp, const LsItem &it, int r)
{
    return it.g < a.E ? tokp[it.pos0 + r] : it.tok0 + r;
}

// out[t][f..f+3] (+)= sum_{j<k} w_tj y[slot_pos[t*k+j]][f..] + sum_s y[n+s*T+t][f..],
// in that order (an empty slot, slot_pos -1, adds nothing); loads in batches
// of 8 so that their latencies overlap.
__device__ __forceinline__ void ls_combine(const LayerArgs &a, int tt, int f, int lane)
{
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 *po = reinterpret_cast<float4 *>(a.out + (size_t)tt * a.H + f);
    const bool on = f < a.H;
    if (on && a.accumulate)
        acc = *po;
    for (int j0 = 0; j0 < a.k; j0 += 8) {
        const int jn = min(8, a.k - j0);
        float wl = 0.f;
        int pl = 0;
        if (lane < jn) {
            wl = __ldcg(a.topk_w + (size_t)tt * a.k + j0 + lane);
            pl = __ldcg(a.slot_pos + (size_t)tt * a.k + j0 + lane);
        }
        float4 v[8];
        int pv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            pv[u] = __shfl_sync(0xffffffffu, pl, u);
            if (u < jn && on && pv[u] >= 0)
                v[u] = __ldcg(reinterpret_cast<const float4 *>(a.y + (size_t)pv[u] * a.H + f));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float wj = __shfl_sync(0xffffffffu, wl, u);
            if (u < jn && on && pv[u] >= 0) {
                acc.x = fmaf(wj, v[u].x, acc.x);
                acc.y = fmaf(wj, v[u].y, acc.y);
                acc.z = fmaf(wj, v[u].z, acc.z);
                acc.w = fmaf(wj, v[u].w, acc.w);
            }
        }
    }
    const int S = a.G - a.E;
    for (int s0 = 0; s0 < S; s0 += 8) {
        const int sn = min(8, S - s0);
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < sn && on)
                v[u] = __ldcg(reinterpret_cast<const float4 *>(
                    a.y + ((size_t)a.n + (size_t)(s0 + u) * a.T + tt) * a.H + f));
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < sn && on) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
    }
    if (on)
        *po = acc;
}

// ------------------------------------------------------------------ one item's stages
//
// The compute warps' work on one item of tile class NTI: every stage of the
// item, from the ring.  Compute warp wg owns weight rows 16*wg .. 16*wg+15 of
// the 128-row tile over the whole K.  acc[nt]: [0],[1] = row g, token columns
// 8nt+2q, +1; [2],[3] = row g+8, same columns.  Returns false when a wait gave
// up.
template <int WFMT, int NT, int NTI, bool GU>
__device__ __forceinline__ bool ls_item_stages(const LayerArgs &a, const LsItem &it, uint8_t *smem,
                                               uint64_t *full, uint64_t *empty, uint32_t &rc,
                                               volatile int *abort_flag, float (&acc)[NTI][4])
{
    using C = LsCfg<WFMT, NT>;
    constexpr bool F16 = C::F16;
    constexpr int RES = C::res_rows(NTI);  // token rows reserved in the stage (per plane)
    constexpr int CH = GU ? C::ch_gu(NTI) : C::ch_dn(NTI);
    constexpr int ROWB = ls_rowb(CH);
    constexpr int HS_OFF = (GU ? 1 : C::NB_DN) * RES * ROWB;
    constexpr int W_OFF = HS_OFF + (GU ? 0 : C::hsb_dn(NTI));
    const int R = a.R;
    const int lane = threadIdx.x & 31, cw = (threadIdx.x >> 5) - 1;
    const int wg = cw, g = lane >> 2, q = lane & 3;
    const int kch = GU ? a.gu_kchunks : a.dn_kchunks;
    const int nst = (kch + CH - 1) / CH;
    const int K = GU ? a.H : a.I;
    const int nt_used = (it.nvalid + 7) >> 3;  // 8-token tiles holding the item's tokens
#pragma unroll
    for (int nt = 0; nt < NTI; ++nt)
        acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    for (int s = 0; s < nst; ++s, ++rc) {
        const int slot = rc % R;
        if (s > 0 && !mbar_wait_warp(&full[slot], (rc / R) & 1, abort_flag, a.err, lane))
            return false;
        const uint8_t *st = smem + (size_t)slot * C::STAGE;
        const uint8_t *brow = st + g * ROWB + q * 8;  // row g of token tile 0, this lane's 8 bytes
        const int ch_n = min(CH, kch - s * CH);
        const int sl0 = (s * 2 * CH) & ~3;
        // 64-wide half kh of chunk c; FULL: the whole chunk lies inside K
        auto half_chunk = [&](const int c, const int kh, auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const uint8_t *wch = st + W_OFF + c * C::W_CHUNK;
            const int ks = 2 * c + kh;                 // 64-wide K slice inside the stage
            const int slice = s * 2 * CH + ks;         // 64-wide K slice of the matrix
            const int kleft = K - slice * 64;          // K left from this slice on (a multiple of 32)
            if (!FULL && kleft <= 0)
                return;
            const int nblk = FULL || kleft >= 64 ? 2 : 1;  // 32-wide blocks of the slice inside K
            const uint8_t *bk = brow + ks * 128;
            if (F16) {
                // weights decode unscaled; each 32-wide block's partial sum takes the
                // row's block scale in FP32: MXFP4 2^(e-127) (a BF16 scale widened
                // exactly), INT4 the group's FP16 scale (widened exactly)
                const uint4 wv = *reinterpret_cast<const uint4 *>(wch + ((wg * 2 + kh) * 32 + lane) * 16);
                const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
                float sg[2], sg8[2];
                // the four A fragments of this half-chunk, decoded once for every token tile
                uint32_t af[4][4];
                if constexpr (WFMT == FMT_MXFP4) {
                    const uint2 sc = *reinterpret_cast<const uint2 *>(wch + CHUNK_MX_CODE_BYTES + (wg * 8 + g) * 8);
                    const uint32_t bx = kh ? ue8m0x2_bf16x2<1>(sc.x) : ue8m0x2_bf16x2<0>(sc.x);
                    const uint32_t by = kh ? ue8m0x2_bf16x2<1>(sc.y) : ue8m0x2_bf16x2<0>(sc.y);
                    sg[0] = __uint_as_float(bx << 16);
                    sg[1] = __uint_as_float(bx & 0xFFFF0000u);
                    sg8[0] = __uint_as_float(by << 16);
                    sg8[1] = __uint_as_float(by & 0xFFFF0000u);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (jj < 2 * nblk)
                            decode_e2m1(words[jj], af[jj]);
                } else {
                    // rows g and g+8: FP16 scales of blocks 0..3 each, then their zero points
                    const uint4 s4 = *reinterpret_cast<const uint4 *>(wch + CHUNK_MX_CODE_BYTES + (wg * 8 + g) * 16);
                    const uint2 z2 = *reinterpret_cast<const uint2 *>(wch + CHUNK_MX_CODE_BYTES + CHUNK_I4_SCALE_BYTES +
                                                                      (wg * 8 + g) * 8);
                    const uint32_t sa = kh ? s4.y : s4.x, sb = kh ? s4.w : s4.z;  // blocks 2kh, 2kh+1
                    sg[0] = f16_half_to_f32<0>(sa);
                    sg[1] = f16_half_to_f32<1>(sa);
                    sg8[0] = f16_half_to_f32<0>(sb);
                    sg8[1] = f16_half_to_f32<1>(sb);
                    const uint32_t za = kh ? z2.x >> 16 : z2.x, zb = kh ? z2.y >> 16 : z2.y;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (jj < 2 * nblk)
                            decode_i4(words[jj], (za >> (8 * (jj >> 1))) & 0xFFu, (zb >> (8 * (jj >> 1))) & 0xFFu,
                                      af[jj]);
                }
                const int *hs_st = reinterpret_cast<const int *>(st + HS_OFF) + (slice - sl0);
#pragma unroll
                for (int nt = 0; nt < NTI; ++nt) {
                    if (NTI == 1 || nt < nt_used) {
                        const uint8_t *pb = bk + nt * 8 * ROWB;
                        float part[4];  // down: this slice's sum before the h block scale
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            if (b < nblk) {
                                float t[4];  // one 32-wide block, before its weight scale
                                uint32_t b0, b1;
                                load_b(pb + (2 * b) * 32, b0, b1);
                                mma_f16_z(t, af[2 * b], b0, b1);
                                load_b(pb + (2 * b + 1) * 32, b0, b1);
                                mma_f16(t, af[2 * b + 1], b0, b1);
                                if (GU) {
                                    acc[nt][0] = fmaf(t[0], sg[b], acc[nt][0]);
                                    acc[nt][1] = fmaf(t[1], sg[b], acc[nt][1]);
                                    acc[nt][2] = fmaf(t[2], sg8[b], acc[nt][2]);
                                    acc[nt][3] = fmaf(t[3], sg8[b], acc[nt][3]);
                                } else if (b == 0) {
                                    part[0] = t[0] * sg[0];
                                    part[1] = t[1] * sg[0];
                                    part[2] = t[2] * sg8[0];
                                    part[3] = t[3] * sg8[0];
                                } else {
                                    part[0] = fmaf(t[0], sg[1], part[0]);
                                    part[1] = fmaf(t[1], sg[1], part[1]);
                                    part[2] = fmaf(t[2], sg8[1], part[2]);
                                    part[3] = fmaf(t[3], sg8[1], part[3]);
                                }
                            }
                        }
                        if (!GU) {
                            // fold in the scale of this 64-feature block of h for each token
                            // column (columns past the item's tokens hold stale data, discarded)
                            const int r0 = 8 * nt + 2 * q;
                            const float f0 = r0 < it.nvalid ? pow2i(hs_st[r0 * LS_HS_ROW]) : 0.f;
                            const float f1 = r0 + 1 < it.nvalid ? pow2i(hs_st[(r0 + 1) * LS_HS_ROW]) : 0.f;
                            acc[nt][0] = fmaf(part[0], f0, acc[nt][0]);
                            acc[nt][1] = fmaf(part[1], f1, acc[nt][1]);
                            acc[nt][2] = fmaf(part[2], f0, acc[nt][2]);
                            acc[nt][3] = fmaf(part[3], f1, acc[nt][3]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    if (jj >= 2 * nblk)
                        break;
                    const uint4 av = *reinterpret_cast<const uint4 *>(wch + ((wg * 8 + 4 * kh + jj) * 32 + lane) * 16);
                    const uint32_t af[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                    for (int nt = 0; nt < NTI; ++nt) {
                        if (NTI == 1 || nt < nt_used) {
                            const uint8_t *pb = bk + nt * 8 * ROWB + jj * 32;
                            uint32_t b0, b1;
                            load_b(pb, b0, b1);
                            mma_bf16(acc[nt], af, b0, b1);
                            if (!GU) {
                                load_b(pb + RES * ROWB, b0, b1);
                                mma_bf16(acc[nt], af, b0, b1);
                            }
                        }
                    }
                }
            }
                };
        if (ch_n == CH && (s + 1) * CH * 128 <= K) {
#pragma unroll(C::CTAS == 1 ? CH : 1)
            for (int c = 0; c < CH; ++c) {
                half_chunk(c, 0, std::true_type{});
                half_chunk(c, 1, std::true_type{});
            }
        } else {
#pragma unroll 1
            for (int c = 0; c < ch_n; ++c) {
                half_chunk(c, 0, std::false_type{});
                half_chunk(c, 1, std::false_type{});
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
    }
    return true;
}

// One item of tile class NTI on a compute warp: its stages, then the epilogue
// (gate|up: SwiGLU and h; down: y).  Returns false when a wait gave up.
template <int WFMT, int NT, int NTI>
__device__ __forceinline__ bool ls_compute_item(const LayerArgs &a, const LsItem &it, uint8_t *smem, uint64_t *full,
                                                uint64_t *empty, uint32_t &rc, volatile int *abort_flag,
                                                const int *sorted, const int *xs_s, float *hmaxb, uint64_t *hmax_bar,
                                                int gu_idx, uint64_t *pub_full, uint64_t *pub_empty, int *pub_g)
{
    using C = LsCfg<WFMT, NT>;
    constexpr bool F16 = C::F16;
    const int lane = threadIdx.x & 31, wg = (threadIdx.x >> 5) - 1;
    const int g = lane >> 2, q = lane & 3;
    const bool gu = it.gu;
    float acc[NTI][4];
    const bool ok = gu ? ls_item_stages<WFMT, NT, NTI, true>(a, it, smem, full, empty, rc, abort_flag, acc)
                       : ls_item_stages<WFMT, NT, NTI, false>(a, it, smem, full, empty, rc, abort_flag, acc);
    if (!ok)
        return false;

    // ------------------------------------------------------ epilogue
    // acc[nt]: [0],[1] = row g, tokens 8nt+2q, +1; [2],[3] = row g+8, same tokens.
    if (gu) {
        const int n = gu_row_feature(it.rt, 16 * wg + g);  // row g: gate, row g+8: up of feature n
        float hv[NTI][2];
#pragma unroll
        for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = 8 * nt + 2 * q + e;
                float gv = acc[nt][e], uv = acc[nt][2 + e];
                if (F16) {  // undo the per-token scaling of x16
                    const float fx = tok < it.nvalid ? pow2i(xs_s[ls_row_token(a, sorted, it, tok)]) : 0.f;
                    gv *= fx;
                    uv *= fx;
                }
                hv[nt][e] = (tok < it.nvalid && n < a.I) ? __fdividef(gv, 1.0f + __expf(-gv)) * uv : 0.f;
            }
        if (F16) {
            // h leaves as one FP16 plane scaled by 2^-hs, hs per (position, 64-feature
            // block): block maximum over the 8 features of each warp, then over the 8
            // warps; the block's largest value lands in [2^14, 2^15)
            float *hm = hmaxb + (gu_idx & 1) * 8 * C::ROWS;
#pragma unroll
            for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float m = fabsf(hv[nt][e]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    if (g == 0)
                        hm[wg * C::ROWS + 8 * nt + 2 * q + e] = m;
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(hmax_bar);
            if (!mbar_wait_warp(hmax_bar, gu_idx & 1, abort_flag, a.err, lane))
                return false;
#pragma unroll
            for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * nt + 2 * q + e;
                    float m = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m = fmaxf(m, hm[i * C::ROWS + tok]);
                    const int mb = (int)((__float_as_uint(m) >> 23) & 0xFFu);
                    int hsc = m > 0.f ? mb - 127 - 14 : 0;
                    hsc = hsc < -100 ? -100 : (hsc > 100 ? 100 : hsc);
                    if (tok < it.nvalid) {
                        if (n < a.I) {
                            const size_t o =
                                (size_t)(it.pos0 + tok) * a.I + (n & ~15) + x16_phys_k(n & 15);
                            a.h[o] = __half_as_ushort(__float2half_rn(hv[nt][e] * pow2i(-hsc)));
                        }
                        if (wg == 0 && g == 0)
                            a.hs[(size_t)(it.pos0 + tok) * a.hs_pitch + it.rt] = hsc;
                    }
                }
        } else {
#pragma unroll
            for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * nt + 2 * q + e;
                    if (tok < it.nvalid && n < a.I) {
                        const float v = hv[nt][e];
                        const __nv_bfloat16 hb = __float2bfloat16_rn(v);
                        const __nv_bfloat16 lb = __float2bfloat16_rn(v - __bfloat162float(hb));
                        const size_t o = (size_t)(it.pos0 + tok) * a.I + (n & ~15) + x16_phys_k(n & 15);
                        a.h[o] = __bfloat16_as_ushort(hb);
                        a.h[o + a.h_plane] = __bfloat16_as_ushort(lb);
                    }
                }
        }
        // hand the item to the publisher warp, whose release at GPU scope covers
        // this warp's h (ordered before it through the hand-off barrier)
        const int ps = gu_idx % LS_PUB_R;
        if (!mbar_wait_warp(&pub_empty[ps], ((gu_idx / LS_PUB_R) & 1) ^ 1, abort_flag, a.err, lane))
            return false;
        if (lane == 0) {
            if (wg == 0)
                pub_g[ps] = it.g;
            mbar_arrive(&pub_full[ps]);
        }
    } else {
        const int m = it.rt * TILE_ROWS + 16 * wg + g;
#pragma unroll
        for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = 8 * nt + 2 * q + e;
                if (tok < it.nvalid) {
                    float *yrow = a.y + (size_t)(it.pos0 + tok) * a.H;
                    if (m < a.H)
                        yrow[m] = acc[nt][e];
                    if (m + 8 < a.H)
                        yrow[m + 8] = acc[nt][2 + e];
                }
            }
    }
    return true;
}

// the wide tile classes out of line: they hold many accumulators and run only
// for the few groups with more than 8 tokens
template <int WFMT, int NT, int NTI>
__device__ __noinline__ bool ls_compute_item_wide(const LayerArgs &a, const LsItem &it, uint8_t *smem, uint64_t *full,
                                                  uint64_t *empty, uint32_t &rc, volatile int *abort_flag,
                                                  const int *sorted, const int *xs_s, float *hmaxb,
                                                  uint64_t *hmax_bar, int gu_idx, uint64_t *pub_full,
                                                  uint64_t *pub_empty, int *pub_g)
{
    return ls_compute_item<WFMT, NT, NTI>(a, it, smem, full, empty, rc, abort_flag, sorted, xs_s, hmaxb, hmax_bar,
                                          gu_idx, pub_full, pub_empty, pub_g);
}

// ------------------------------------------------------------------ the kernel

template <int WFMT, int NT>
__global__ void __launch_bounds__(LS_THREADS, ls_ctas_per_sm(NT)) layer_stream_kernel(const __grid_constant__ LayerArgs a)
{
    using C = LsCfg<WFMT, NT>;
    constexpr bool F16 = C::F16;
    constexpr int ROWS = C::ROWS;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    const LsSmem L = ls_smem(a.R, a.G, a.n, a.T, C::STAGE, C::RED_BYTES, C::HMAX_BYTES);
    int2 *hdr = reinterpret_cast<int2 *>(smem + L.hdr);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars), *empty = full + LS_R_MAX;
    uint64_t *hmax_bar = reinterpret_cast<uint64_t *>(smem + L.pbars);
    uint64_t *pub_full = hmax_bar + 1, *pub_empty = pub_full + LS_PUB_R;  // publisher hand-off
    int *pub_g = reinterpret_cast<int *>(smem + L.misc) + 4;
    int *misc = reinterpret_cast<int *>(smem + L.misc);
    volatile int *abort_flag = misc;
    float *hmaxb = reinterpret_cast<float *>(smem + L.hmax);
    int *gcnt = reinterpret_cast<int *>(smem + L.gcnt), *gstart = reinterpret_cast<int *>(smem + L.gstart);
    int *tpre = reinterpret_cast<int *>(smem + L.tpre), *sorted = reinterpret_cast<int *>(smem + L.sorted);
    int *xs_s = reinterpret_cast<int *>(smem + L.xs);
    uint32_t *gdone = reinterpret_cast<uint32_t *>(smem + L.gdone);  // loader: groups whose h is complete
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = a.R;

    if (tid == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], LS_COMPUTE_WARPS);
        }
        mbar_init(hmax_bar, LS_COMPUTE_WARPS);
        for (int i = 0; i < LS_PUB_R; ++i) {
            mbar_init(&pub_full[i], LS_COMPUTE_WARPS);
            mbar_init(&pub_empty[i], 1);
        }
        misc[0] = 0;
        for (int i = 0; i < (a.G + 31) / 32; ++i)
            gdone[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    // The shared groups (or dense slices) lead the work list and need no
    // routing, so their gate|up weights start moving into L2 now, while the
    // tokens are routed: CTA b prefetches the b-th share of the first
    // LS_PF_BYTES (group bytes and shares are multiples of 16).
    if (tid == LS_THREADS - 32 && a.E < a.G) {
        const size_t total = min((size_t)(a.G - a.E) * a.gu_group_bytes, LS_PF_BYTES);
        const size_t per = (total / gridDim.x + 15) & ~(size_t)15;
        const size_t lo = per * blockIdx.x, hi = min(lo + per, total);
        const uint8_t *base = a.wgu + (size_t)a.E * a.gu_group_bytes;
        for (size_t o = lo; o < hi; o += LS_PF_PIECE)
            prefetch_l2(base + o, (uint32_t)min((size_t)LS_PF_PIECE, hi - o));
    }

    // ---------------------------------------------------------- phase 0a
    // local: this CTA routes every token (slot ids straight into the
    // schedule's scratch); otherwise only its own tokens
    const bool local = a.T <= LS_LOCAL_ROUTE_T;
    const int mine = (int)blockIdx.x < a.T ? (a.T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (tid < LS_ROUTE_THREADS) {
        if (a.E > 0) {
            if (local) {
                for (int t = warp; t < a.T; t += LS_ROUTE_WARPS) {
                    const bool own = t % (int)gridDim.x == (int)blockIdx.x;
                    if (a.ids_in)
                        ls_copy_route_warp(a, t, lane, reinterpret_cast<int *>(smem), own);
                    else
                        ls_route_warp(a, t, lane, reinterpret_cast<int *>(smem), own);
                }
            } else {
                for (int i = warp; i < mine; i += LS_ROUTE_WARPS) {
                    const int t = (int)blockIdx.x + i * (int)gridDim.x;
                    if (a.ids_in)
                        ls_copy_route_warp(a, t, lane, nullptr, true);
                    else
                        ls_route_warp(a, t, lane, nullptr, true);
                }
            }
        }
    } else {
        for (int t = blockIdx.x; t < a.T; t += gridDim.x)
            ls_prep_token<F16>(a, t, smem + LS_SCRATCH_PREP);
    }
    fence_proxy_async_global();  // x16 is read by other CTAs' bulk copies
    __syncthreads();
    if (tid == 0) {
        if (mine > 0) {
            __threadfence();
            atomicAdd(&a.sync[SY_ROUTED], mine);
        }
        misc[1] = local || wait_geq(&a.sync[SY_ROUTED], a.T, nullptr, a.err) ? 1 : 0;
    }
    __syncthreads();
    if (!misc[1])
        return;

    // ---------------------------------------------------------- phase 0b
    ls_schedule<ROWS, F16>(a, smem, gcnt, gstart, tpre, sorted, xs_s, local);
    __syncthreads();

    const int rt_gu = a.gu_row_tiles, rt_dn = a.dn_row_tiles;
    const int tiles = tpre[a.G];
    const int total_gu = tiles * rt_gu, total = total_gu + tiles * rt_dn;
    int *grp_done = a.sync + SY_GRP;

    if (warp == 0) {
        // ------------------------------------------------------ loader
        uint32_t rc = 0, armed = 0, armed_par = 0;
        bool ok = true;
        fence_proxy_async_global();  // x16 of other CTAs, acquired above, is read by bulk copies
        // first item: blockIdx.x; the shared counter hands out the rest from gridDim.x on
        int u = blockIdx.x;
        // local routing: every CTA's token rows must be written before the first token copy
        bool x_ready = !local;
        while (ok && u < total) {
            int nxt = 0;
            if (lane == 0)
                nxt = (int)gridDim.x + atomicAdd(&a.sync[SY_WORK], 1);
            const LsItem it = ls_item<ROWS>(u, total_gu, rt_gu, rt_dn, a.E, a.G, gcnt, gstart, tpre);
            const int nti = ls_nti_item<WFMT, NT>(it);  // the item's tile class: its stage geometry
            const int irows = C::res_rows(nti);
            const int CH = it.gu ? C::ch_gu(nti) : C::ch_dn(nti);
            const int kch = it.gu ? a.gu_kchunks : a.dn_kchunks;
            const int nst = (kch + CH - 1) / CH;
            const int K = it.gu ? a.H : a.I;
            const int nb = it.gu ? 1 : C::NB_DN;
            const int rowb = ls_rowb(CH);
            const int hsb = it.gu ? 0 : C::hsb_dn(nti);
            const int w_off = nb * irows * rowb + hsb;
            const uint8_t *wsrc = (it.gu ? a.wgu + (size_t)it.g * a.gu_group_bytes
                                         : a.wdn + (size_t)it.g * a.dn_group_bytes) +
                                  (size_t)it.rt * kch * (size_t)a.chunk_bytes;
            // this lane's token rows (r = lane, lane + 32): source row starts
            const uint16_t *src[2] = {nullptr, nullptr};
            int pos_r[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = lane + 32 * i;
                if (r < it.nvalid) {
                    pos_r[i] = it.pos0 + r;
                    src[i] = it.gu ? a.x16 + (size_t)ls_row_token(a, sorted, it, r) * a.H
                                   : a.h + (size_t)pos_r[i] * a.I;
                }
            }
            for (int s = 0; s < nst; ++s, ++rc) {
                const int slot = rc % R;
                const uint32_t ph = (rc / R) & 1;
                // (a sleeping wait: the loader shares its sub-partition with compute warps)
                if (!(ok = mbar_wait_sleep_warp(&empty[slot], ph ^ 1, abort_flag, a.err, lane)))
                    break;
                uint8_t *st = smem + (size_t)slot * C::STAGE;
                const int ch_n = min(CH, kch - s * CH);
                const uint32_t wbytes = (uint32_t)(ch_n * a.chunk_bytes);
                const int k0 = s * CH * 128;
                const uint32_t vb = (uint32_t)min(CH * 128, K - k0) * 2;  // valid bytes of a token row
                int sl0 = 0, nh = 0;
                if (F16 && !it.gu) {
                    const int ks2 = 2 * CH;
                    sl0 = (s * ks2) & ~3;
                    nh = min(((s * ks2 + ks2 + 3) & ~3) - sl0, a.hs_pitch - sl0);
                }
                const uint32_t tbytes = (uint32_t)it.nvalid * (nb * vb + (uint32_t)nh * 4);
                const bool wait_h = !it.gu && s == 0;
                const bool wait_x = it.gu && s == 0 && !x_ready;
                if (lane == 0) {
                    hdr[slot] = make_int2(u, s);
                    if (wait_h || wait_x)
                        mbar_expect_tx(&full[slot], wbytes);
                    else
                        mbar_arrive_expect_tx(&full[slot], wbytes + tbytes);
                    bulk_g2s(st + w_off, wsrc + (size_t)s * CH * a.chunk_bytes, wbytes, &full[slot]);
                }
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (ph << slot);
                if (wait_h) {
                    // the group's h must be complete: 8 epilogue warps per gate|up item
                    int hok = 1;
                    if (lane == 0) {
                        const uint32_t bit = 1u << (it.g & 31);
                        if (!(gdone[it.g >> 5] & bit)) {
                            const int target = it.ntl * rt_gu * 8;
                            hok = wait_geq(&grp_done[it.g], target, abort_flag, a.err) ? 1 : 0;
                            if (hok)
                                gdone[it.g >> 5] |= bit;
                        }
                        if (hok)
                            fence_proxy_async_global();
                        // arrive in any case so that the weight copy can still complete the phase
                        mbar_arrive_expect_tx(&full[slot], hok ? tbytes : 0u);
                    }
                    if (!(ok = __shfl_sync(0xffffffffu, hok, 0) != 0))
                        break;
                }
                if (wait_x) {
                    // the token rows and scales of all tokens (written by their owner CTAs)
                    int xok = 1;
                    if (lane == 0) {
                        xok = wait_geq(&a.sync[SY_ROUTED], a.T, abort_flag, a.err) ? 1 : 0;
                        if (xok)
                            fence_proxy_async_global();
                    }
                    __syncwarp();
                    xok = __shfl_sync(0xffffffffu, xok, 0);
                    if (F16 && xok && lane < a.T)
                        xs_s[lane] = __ldcg(a.xs + lane);
                    __syncwarp();
                    // arrive in any case so that the weight copy can still complete the phase
                    if (lane == 0)
                        mbar_arrive_expect_tx(&full[slot], xok ? tbytes : 0u);
                    x_ready = true;
                    if (!(ok = xok != 0))
                        break;
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = lane + 32 * i;
                    if (r < it.nvalid) {
                        uint8_t *drow = st + r * rowb;
                        bulk_g2s(drow, src[i] + k0, vb, &full[slot]);
                        if (!it.gu) {
                            if (!F16)  // BF16: the lo plane of h
                                bulk_g2s(drow + irows * rowb, src[i] + a.h_plane + k0, vb, &full[slot]);
                            else
                                bulk_g2s(st + nb * irows * rowb + r * LS_HS_ROW * 4,
                                         a.hs + (size_t)pos_r[i] * a.hs_pitch + sl0, (uint32_t)nh * 4, &full[slot]);
                        }
                    }
                }
            }
            u = __shfl_sync(0xffffffffu, nxt, 0);
        }
        if (ok) {
            // terminal stage: tells the compute warps that the list is exhausted
            const int slot = rc % R;
            const uint32_t ph = (rc / R) & 1;
            if (mbar_wait_warp(&empty[slot], ph ^ 1, abort_flag, a.err, lane)) {
                // the slot's previous phase has been consumed, so its copies have landed;
                // the terminal phase carries no copy
                armed &= ~(1u << slot);
                if (lane == 0) {
                    hdr[slot] = make_int2(-1, 0);
                    mbar_arrive(&full[slot]);
                }
            }
        }
        if (lane == 0)
            for (int s = 0; s < R; ++s)
                if (armed & (1u << s))
                    mbar_drain(&full[s], (armed_par >> s) & 1);
        __syncwarp();
    } else if (warp <= LS_COMPUTE_WARPS) {
        // ------------------------------------------------------ compute warps
        uint32_t rc = 0;
        int gu_i = 0;
        bool ok = true;
        for (;;) {
            int slot = rc % R;
            if (!(ok = mbar_wait_warp(&full[slot], (rc / R) & 1, abort_flag, a.err, lane)))
                break;
            const int2 h0 = hdr[slot];
            if (h0.x < 0)
                break;
            const LsItem it = ls_item<ROWS>(h0.x, total_gu, rt_gu, rt_dn, a.E, a.G, gcnt, gstart, tpre);
            const int gu_idx = it.gu ? gu_i++ : 0;
            const int nti = ls_nti_item<WFMT, NT>(it);
#define LS_ITEM(F_, ...)                                                                                      \
    F_<WFMT, NT, __VA_ARGS__>(a, it, smem, full, empty, rc, abort_flag, sorted, xs_s, hmaxb, hmax_bar, gu_idx,   \
                              pub_full, pub_empty, pub_g)
            if (NT <= 1 || nti == 1)
                ok = LS_ITEM(ls_compute_item, 1);
            else if (NT == 2 || nti == 2)
                ok = LS_ITEM(ls_compute_item_wide, NT < 2 ? 1 : 2);
            else if (NT == 4 || nti == 4)
                ok = LS_ITEM(ls_compute_item_wide, NT < 4 ? 1 : 4);
            else
                ok = LS_ITEM(ls_compute_item_wide, NT < 8 ? 1 : 8);
#undef LS_ITEM
            if (!ok)
                break;
        }
        if (ok) {
            // terminal hand-off: no further item follows
            const int ps = gu_i % LS_PUB_R;
            if (mbar_wait_warp(&pub_empty[ps], ((gu_i / LS_PUB_R) & 1) ^ 1, abort_flag, a.err, lane) && lane == 0) {
                if (warp == 1)
                    pub_g[ps] = -1;
                mbar_arrive(&pub_full[ps]);
            }
        }
        __threadfence();  // y of this warp, before the CTA reports that it is done
    } else {
        // ------------------------------------------------------ publisher
        // For each finished gate|up item, in order: once all compute warps have
        // written their h, one release at GPU scope adds the item's warps to the
        // group's count, so a compute warp never waits for its own writes.
        for (int i = 0;; ++i) {
            const int ps = i % LS_PUB_R;
            if (!mbar_wait_sleep_warp(&pub_full[ps], (i / LS_PUB_R) & 1, abort_flag, a.err, lane))
                break;
            const int g = pub_g[ps];
            if (g < 0)
                break;
            if (lane == 0) {
                fence_acq_rel_gpu();
                atomicAdd(&grp_done[g], LS_COMPUTE_WARPS);
                mbar_arrive(&pub_empty[ps]);
            }
            __syncwarp();
        }
    }
    __syncthreads();

    // ---------------------------------------------------------- combine
    // once every CTA has finished its items: warp w of CTA b combines the
    // (token, 128-feature block)s w * gridDim.x + b, then every LS_WARPS * gridDim.x
    if (tid == 0) {
        red_release_add(&a.sync[SY_DONE], 1);
        bool okc = wait_geq(&a.sync[SY_DONE], (int)gridDim.x + a.done_extra, abort_flag, a.err, a.done_wait_ns);
        if (okc && a.E > 0 && a.n > 0)
            okc = wait_geq(&a.sync[SY_PERM], 1, abort_flag, a.err);
        misc[2] = okc ? 1 : 0;
    }
    __syncthreads();
    if (misc[2]) {
        const int nblk = a.T * rt_dn;
        for (int bk = warp * (int)gridDim.x + (int)blockIdx.x; bk < nblk; bk += LS_WARPS * (int)gridDim.x)
            ls_combine(a, bk / rt_dn, (bk % rt_dn) * TILE_ROWS + 4 * lane, lane);
    }
}

// ------------------------------------------------------------------ host side

template <int WFMT, int NT>
int ls_ring_depth(int G, int n, int E, int T)
{
    using C = LsCfg<WFMT, NT>;
    const LsSmem base = ls_smem(0, G, n, T, C::STAGE, C::RED_BYTES, C::HMAX_BYTES);
    int R = (C::SMEM_LIMIT - base.total) / C::STAGE;
    if (R > LS_R_MAX)
        R = LS_R_MAX;
    // phase-0 scratch lives in the ring: the slot ids of local routing and the
    // prep reduction; then the slot ids, group-scan totals and permutation counters
    const long long scratch0 = LS_SCRATCH_PREP + 128;
    const long long scratch1 = ((long long)((n + 3) & ~3) + 2 * LS_WARPS + (long long)LS_WARPS * E) * 4;
    const long long ring = (long long)R * C::STAGE;
    if (ring < scratch0 || ring < scratch1)
        return 0;
    return R >= 2 ? R : 0;
}

template <int WFMT, int NT>
cudaError_t ls_launch(LayerArgs a, cudaStream_t st)
{
    using C = LsCfg<WFMT, NT>;
    // the stages hold whole chunks of this format's size
    if (a.chunk_bytes != C::W_CHUNK)
        return cudaErrorInvalidValue;
    a.R = ls_ring_depth<WFMT, NT>(a.G, a.n, a.E, a.T);
    if (a.R < 2)
        return cudaErrorNotSupported;
    const LsSmem L = ls_smem(a.R, a.G, a.n, a.T, C::STAGE, C::RED_BYTES, C::HMAX_BYTES);
    auto kern = layer_stream_kernel<WFMT, NT>;
    static std::atomic<int> attr_set[MAX_DEVICES];
    cudaError_t e = smem_limit_once(attr_set, (const void *)kern, C::SMEM_LIMIT);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sm_count() * C::CTAS));
    cfg.blockDim = dim3(LS_THREADS);
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

int ls_nt(int T)
{
    const int t = T < STREAM_MAX_T ? T : STREAM_MAX_T;
    return t <= 2 ? 0 : t <= 8 ? 1 : t <= 16 ? 2 : t <= 32 ? 4 : 8;
}

template <int WFMT>
int ls_depth_fmt(int nt, int G, int n, int E, int T)
{
    switch (nt) {
    case 0: return ls_ring_depth<WFMT, 0>(G, n, E, T);
    case 1: return ls_ring_depth<WFMT, 1>(G, n, E, T);
    case 2: return ls_ring_depth<WFMT, 2>(G, n, E, T);
    case 4: return ls_ring_depth<WFMT, 4>(G, n, E, T);
    default: return ls_ring_depth<WFMT, 8>(G, n, E, T);
    }
}

template <int WFMT>
cudaError_t ls_launch_fmt(int nt, const LayerArgs &a, cudaStream_t st)
{
    switch (nt) {
    case 0: return ls_launch<WFMT, 0>(a, st);
    case 1: return ls_launch<WFMT, 1>(a, st);
    case 2: return ls_launch<WFMT, 2>(a, st);
    case 4: return ls_launch<WFMT, 4>(a, st);
    default: return ls_launch<WFMT, 8>(a, st);
    }
}

}  // namespace

size_t layer_stream_sync_bytes(int G)
{
    return (size_t)(SY_GRP + G) * sizeof(int);
}

bool layer_stream_fits(const Plan &p, int fmt)
{
    if (p.T < 1 || p.G < 1 || p.G > MAX_GROUPS || p.E > LS_MAX_EXPERTS || (long long)p.T * p.k > LS_MAX_SLOTS)
        return false;
    const int nt = ls_nt(p.T);
    const int n = p.T * p.k;
    const int R = fmt == FMT_MXFP4  ? ls_depth_fmt<FMT_MXFP4>(nt, p.G, n, p.E, p.T)
                  : fmt == FMT_INT4 ? ls_depth_fmt<FMT_INT4>(nt, p.G, n, p.E, p.T)
                                    : ls_depth_fmt<FMT_BF16>(nt, p.G, n, p.E, p.T);
    return R >= 2;
}

cudaError_t launch_layer_stream(const Plan &p, const WeightStore &gu, const WeightStore &dn, int fmt,
                                const uint16_t *x, const float *logits, const int *ids_in, const float *w_in,
                                float *out, int accumulate, cudaStream_t st, int expire_wait_us)
{
    cudaError_t e = cudaMemsetAsync(p.sync, 0, layer_stream_sync_bytes(p.G), st);
    if (e != cudaSuccess)
        return e;
    LayerArgs a{};
    a.wgu = gu.base;
    a.wdn = dn.base;
    a.gu_group_bytes = gu.group_bytes;
    a.dn_group_bytes = dn.group_bytes;
    a.gu_kchunks = gu.kchunks;
    a.dn_kchunks = dn.kchunks;
    a.gu_row_tiles = gu.row_tiles;
    a.dn_row_tiles = dn.row_tiles;
    a.chunk_bytes = gu.chunk_bytes;
    a.T = p.T;
    a.k = p.E > 0 ? p.k : 0;
    a.E = p.E;
    a.S = p.S;
    a.G = p.G;
    a.H = p.H;
    a.I = p.I;
    a.n = p.E > 0 ? p.T * p.k : 0;
    a.x = x;
    a.logits = logits;
    a.ids_in = ids_in;
    a.ebase = p.ebase;
    a.etotal = p.etotal;
    a.w_in = w_in;
    a.topk_ids = p.topk_ids;
    a.topk_w = p.topk_w;
    a.expert_offsets = p.expert_offsets;
    a.sorted_slot = p.sorted_slot;
    a.slot_pos = p.slot_pos;
    a.x16 = p.x16;
    a.xs = p.xs;
    a.h = p.h;
    a.h_plane = (long long)p.P * p.I;
    a.hs = p.hs;
    a.hs_pitch = p.hs_pitch;
    a.y = p.y;
    a.out = out;
    a.accumulate = accumulate;
    a.sync = p.sync;
    a.err = p.err;
    a.done_extra = expire_wait_us > 0 ? 1 : 0;
    a.done_wait_ns = expire_wait_us > 0 ? (unsigned long long)expire_wait_us * 1000ull : WAIT_LIMIT_NS;
    const int nt = ls_nt(p.T);
    return fmt == FMT_MXFP4  ? ls_launch_fmt<FMT_MXFP4>(nt, a, st)
           : fmt == FMT_INT4 ? ls_launch_fmt<FMT_INT4>(nt, a, st)
                             : ls_launch_fmt<FMT_BF16>(nt, a, st);
}

}  // namespace moe
