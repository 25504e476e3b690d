// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a): gate|up with fused SwiGLU, and down.
//
// Operation (per expert group g and token position p of the group):
//   gate|up:  g_n = x_p . W_g[n],  u_n = x_p . W_u[n],  h_pn = SiLU(g_n) * u_n
//   down:     y_pm = h_p . W_d[m]
// with the SwiGLU expert of "Cascadia: Resident 975B MoE Inference on Eleven
// AI PCs" §3.1 and MXFP4 weights decoded inside the reduction as in
// "DeepSeek-V4-Flash on a four-GPU Ampere workstation", section "MXFP4 is not
// NVFP4, and the difference matters on Ampere" (the block scale applied once
// per 32-value block, FP32 accumulation, no decoded copy of an expert in
// device memory).
//
// Mapping to the hardware ("swap-AB": weights are the M side):
//   D[128 weight rows, N tokens] (FP32, tensor memory) += A[128 rows, K] . B[N tokens, K]^T
//   A = weight rows, decoded by CUDA-core warps straight from the weight chunks
//       in global memory and written into TENSOR MEMORY (tcgen05.st); the MMA
//       reads A from there, so shared memory carries only the token operand;
//   B = token rows, loaded by TMA into 128-byte-swizzled K-major tiles;
//   MMA = tcgen05.mma kind::f16, M = 128, N = 16..256, K = 16, one thread.
// A work item is (group, 128-row tile, token tile of up to 192), and a pipeline
// stage is 128 values of K: eight long MMAs (up to 96 cycles each) per hand-off
// between the producers and the MMA thread.  (Measured: the tensor pipe idles
// when a stage's hand-off guards few or short MMAs -- two 128 x 128 tiles per
// 64-wide stage ran at about half rate; one 128 x 256 tile per 128-wide stage at
// full rate.)  Tensor memory holds two 192-column accumulators, so that the
// epilogue of one item overlaps the MMAs of the next, and two stages of A (64
// columns each); shared memory holds four 48 KB stages of B, a deeper ring
// with its own barriers, so that token tiles arrive ahead despite L2 latency.
//
// Two operand types (chosen per handle at load):
//   FP16: MXFP4 weights whose E8M0 exponents span at most 23 within every row.
//     A weight decodes to v(c) * 2^(e - b), b the row's largest exponent: one
//     hardware e2m1x2 -> f16x2 conversion per pair and one multiply by a power
//     of two, both exact (every value is a multiple of 2^-24 with at most two
//     significant bits).  The epilogue multiplies each row's accumulator by
//     2^(b - 127).  Token rows are FP16 x * 2^-xs (a power of two per token,
//     chosen so that the conversion of the BF16 values is exact); h leaves
//     gate|up as one FP16 plane h * 2^-hs with a power of two per position
//     fixed before the GEMM from a bound on |h| (token_prep_f16_kernel), and
//     down runs one MMA per K step and writes y as FP16 with a power of two
//     per position from a bound on |y| (half the bytes of FP32 y for the
//     combine to read).
//   FP16 hi + lo (group-32 INT4): w = s (q - z) relative to a power of two per
//     row, split into an exact FP16 pair; the decoders write hi and lo into the
//     two halves of an A slot, stages are 64 values of K, and the MMA thread
//     runs four MMAs on each half.  Tokens, h and y as for FP16.
//   BF16: BF16 weights, or MXFP4 whose exponents spread wider.  MXFP4 decodes
//     exactly to BF16 v(c) * 2^(e - 127); BF16 weights need no decode, and
//     their A tiles come by TMA into the token tiles' shared-memory stage,
//     the MMAs reading both operands from shared memory (the decoder warps
//     idle).  Tokens are the caller's BF16 rows; h is kept as BF16 hi + lo
//     planes (lo = bf16(h - hi)), so down runs two MMAs per K step (and its
//     stages hold 64 values of K, to keep 64 KB of B).
// One CTA per SM walks a static schedule of work items.  Warp roles:
//   warp 0      TMA-loads token tiles (B; with BF16 weights also the A tiles)
//               into the shared-memory stage ring and prefetches the weight
//               chunks ahead into L2
//   warp 1      allocates tensor memory, issues the MMAs, commits to mbarriers
//   warps 2-9   decode weights into the tensor-memory A ring: two groups of
//               four warps, group g decoding every other stage (A slot g) in
//               full; its warp w covers lane quadrant w % 4 (the lanes a warp
//               may access)
//   warps 10-17 epilogue, two warps per lane quadrant splitting the columns:
//               tensor memory -> registers, SwiGLU (gate|up) or y (down).
// Every mbarrier wait is bounded: on a timeout the kernel records
// DEV_ERR_WAIT_TIMEOUT, stops issuing work, waits (bounded) for the copies and
// MMAs it has in flight, frees its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "mx_decode.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int N_DEC_WARPS = 8;
constexpr int N_DEC_GROUPS = N_DEC_WARPS / 4;  // groups of four warps, one per tensor-memory lane quadrant
constexpr int N_EPI_WARPS = 8;                 // two per tensor-memory lane quadrant, splitting the columns
constexpr int NUM_THREADS = (2 + N_DEC_WARPS + N_EPI_WARPS) * 32;
constexpr int WARP_BLOAD = 0, WARP_MMA = 1, WARP_DEC0 = 2, WARP_EPI0 = WARP_DEC0 + N_DEC_WARPS;
constexpr int NMAX = 192;                      // token columns of a work item
constexpr int NBUF = 2;                        // accumulators: one item's epilogue overlaps the next item's MMAs
constexpr int A_STAGES = 2;                    // A ring (tensor memory)
constexpr int B_STAGES = 4;                    // B ring (shared memory)
constexpr int TMEM_COLS = 512;                 // the whole tensor memory of the SM
constexpr int A_SLOT_COLS = 64;                // tensor-memory columns of a stage of A: 128 16-bit values per lane
constexpr int TMEM_A0 = NBUF * NMAX;           // first column of the A ring, after the accumulators
static_assert(TMEM_A0 + A_STAGES * A_SLOT_COLS <= TMEM_COLS, "tensor memory");
// Decoder group g fills A slot g only (stages g, g + A_STAGES, ...): it then
// waits on that slot's empty barrier for its own previous stage alone, never
// for a phase two behind (where the parity it waits for would already read as
// complete from an older phase).
static_assert(N_DEC_GROUPS == A_STAGES, "one decoder group per A slot");
constexpr int B_SLICE_BYTES = NMAX * HALF_K * 2;  // 24 KB: 192 token rows x 64 16-bit values (one swizzled tile)
constexpr int B_STAGE_BYTES = 2 * B_SLICE_BYTES;  // two slices: 128 K values of one plane, or 64 of two planes
static_assert(B_SLICE_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
// BF16 weights need no decode: their A tiles (128 rows x 64 values, one
// swizzled 16 KB tile per 64-wide half of a chunk of the TILE store) come by
// TMA into the same shared-memory stage as the token tiles, and the MMA reads A
// from there.  Stages are 64 values of K: a token slice (two for down, h hi and
// lo) plus the A tile, five stages (40 KB) for gate|up and three (64 KB) for down.
constexpr int A_SMEM_TILE = TILE_ROWS * HALF_K * 2;
constexpr int RING_MAX = 5;
constexpr int RING_BYTES_MAX = 5 * (B_SLICE_BYTES + A_SMEM_TILE);
static_assert(RING_BYTES_MAX >= B_STAGES * B_STAGE_BYTES && RING_BYTES_MAX >= 3 * (2 * B_SLICE_BYTES + A_SMEM_TILE),
              "ring room");
// B operand TMA boxes: 64 token rows (8 KB) each, so that a stage takes few
// TMA issues; 16 rows when a B tensor has fewer than 64 rows
constexpr int B_BOX_ROWS_BIG = 64, B_BOX_ROWS_SMALL = 16;
// the token loader also prefetches the weight chunks this many chunks ahead of
// the stage it loads into L2, where the decoders' own loads (issued one of
// their stages ahead) then find them
constexpr int PF_CHUNKS = 8;

struct TcArgs {
    const uint8_t *wbase;
    size_t group_bytes;
    int kchunks, chunk_bytes, row_tiles;
    const uint8_t *row_base;  // FP16 operands: largest E8M0 exponent of every row, [G][row_tiles * 128]
    const int *grp_start, *grp_count;
    int E, G, I, H;
    // gate|up output: BF16 operands h hi + lo planes; FP16 operands one FP16 plane h16
    uint16_t *h_out;
    long long h_plane;
    uint16_t *h16;
    const int *row_token;  // token of each position
    const int *xsp;        // FP16 operands: power of two of each position's FP16 token row
    // down output: BF16 operands FP32 y; FP16 operands FP16 y16 with a power of two per position
    float *y_out;
    uint16_t *y16;
    const int *ys;
    const int *hsp;        // FP16 operands: per-position power of two of the FP16 h rows (written by
                           // gate|up with it, read by down)
    int *err;
    int brows;  // token rows per TMA box of the B operand (16, or 64 when every B tensor has that many rows)
};

// operand paths: FP16 (MXFP4 decoded exactly), BF16, and FP16 hi + lo pairs of
// group-32 INT4 weights (two MMAs per K step on 64-value stages)
enum { OP_F16 = 0, OP_BF16 = 1, OP_I4 = 2 };

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// The four K=16 MMAs of one 64-wide stage with A in tensor memory: A advances
// by 8 columns (16 values per lane) and the B descriptor by 32 bytes (2 in the
// address field) per K step; the first MMA accumulates only when acc0 != 0,
// the other three always.
__device__ __forceinline__ void tc_mma4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t acc0)
{
    asm volatile(
        "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %4, 0;\n setp.eq.b32 p1, %4, %4;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, p1;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc0), "r"(a_tmem + 8), "l"(b_desc + 2), "r"(a_tmem + 16),
        "l"(b_desc + 4), "r"(a_tmem + 24), "l"(b_desc + 6)
        : "memory");
}

// 16 consecutive tensor-memory columns of this warp's 32 lanes from registers
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// 32 consecutive tensor-memory columns of this warp's 32 lanes, one wait
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr), "r"(taddr + 16)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// core groups 1024 bytes apart (SBO), leading offset unused for this layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor of kind::f16: FP16 (OP_F16) or BF16 A and B, FP32 D,
// both K-major, M = 128, N given.
template <int OP>
__device__ __forceinline__ uint32_t make_idesc(int n)
{
    const uint32_t ab = OP == OP_BF16 ? (1u << 7) | (1u << 10) : 0u;
    return (1u << 4) | ab | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TILE_ROWS >> 4) << 24);
}

// The four K=16 MMAs of one 64-wide stage with both operands in shared memory
// (128-byte-swizzled K-major tiles): both descriptors advance by 32 bytes (2 in
// the address field) per K step.
__device__ __forceinline__ void tc_mma4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t acc0)
{
    asm volatile(
        "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %4, 0;\n setp.eq.b32 p1, %4, %4;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, p1;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, p1;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc0), "l"(a_desc + 2), "l"(b_desc + 2), "l"(a_desc + 4),
        "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
        : "memory");
}

// One INT4 pair into FP16 hi and lo words: w holds the pair's codes in bits
// 0..3 and 16..19; 0x6400 | q is the FP16 value 1024 + q (ulp 1), so
// subtracting zz = {1024 + z, 1024 + z} leaves q - z exactly; hi = s2 (q - z)
// rounded to FP16, lo = s2 (q - z) - hi from one fused multiply-add (exact: the
// product has at most 15 significant bits, hi takes 11).
__device__ __forceinline__ void i4_pair_hilo(uint32_t w, uint32_t zz, uint32_t s2, uint32_t &hi, uint32_t &lo)
{
    const uint32_t v = (w & 0x000F000Fu) | 0x64006400u;
    uint32_t qz;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(qz) : "r"(v), "r"(zz));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(qz), "r"(s2));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(qz), "r"(s2), "r"(hi ^ 0x80008000u));
}

// {2^d, 2^d} in FP16 for d in [-24, 0] (below -14 a subnormal, exactly)
__device__ __forceinline__ uint32_t f16x2_pow2(int d)
{
    const uint32_t b = d >= -14 ? (uint32_t)(d + 15) << 10 : 1u << (d + 24);
    return b * 0x10001u;
}

// 8 E2M1 codes (4 bytes; element 2j in the low nibble of byte j) -> 4 FP16
// pairs times the power of two s2 (low element in the low half)
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t s2, uint32_t *out)
{
    uint32_t c[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[i]) : "r"(c[i]), "r"(s2));
}

// 2^k as a float for |k| <= 126
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((127 + k) << 23); }

struct Smem {
    static constexpr int BAR_OFF = RING_BYTES_MAX;
    static constexpr int N_BARS = 2 * RING_MAX + 2 * A_STAGES + 2 * NBUF;
    static constexpr int SCHED_OFF = BAR_OFF + N_BARS * 8;
    static constexpr int MISC_OFF = SCHED_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int COLSC_OFF = MISC_OFF + 32;    // epilogue: column scales of an item, one row per warp
    static constexpr int HSC_OFF = COLSC_OFF + N_EPI_WARPS * NMAX * 4;  // gate|up: h scales, one row per warp
    static constexpr int TOTAL = HSC_OFF + N_EPI_WARPS * NMAX * 4 + 1024;  // + alignment slack
};

// ------------------------------------------------------------------ kernel

template <bool GU, int OP, int WFMT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b2,
                   const __grid_constant__ CUtensorMap map_a)
{
    static_assert(OP == OP_BF16 || (OP == OP_F16 && WFMT == FMT_MXFP4) || (OP == OP_I4 && WFMT == FMT_INT4),
                  "FP16 operands decode MXFP4 weights, FP16 pairs INT4 weights");
    constexpr bool FT = OP != OP_BF16;                  // FP16 token operands (x16, h16) and scaled epilogues
    constexpr int NB = (!GU && OP == OP_BF16) ? 2 : 1;  // token planes: down with BF16 operands reads h hi + lo
    constexpr bool AS = WFMT == FMT_BF16;               // A by TMA into shared memory (BF16 weights)
    constexpr int KST = (AS || NB == 2 || OP == OP_I4) ? HALF_K : CHUNK_K;  // K values per stage
    constexpr int NSL = KST / HALF_K;                   // 64-wide K slices per stage
    constexpr int NSLB = NSL * NB;                      // swizzled B tiles per stage
    constexpr int NBLK = KST / 32;                      // 32-value blocks per stage
    using L = Smem;
    static_assert(L::TOTAL <= 232448, "shared memory");
    static_assert(NSLB == 2 || ((OP == OP_I4 || AS) && NSLB == 1), "a stage holds two swizzled B tiles (INT4: one)");
    // the stage ring: token tiles, and with AS the A tile after them
    constexpr int STAGE_BYTES = AS ? NSLB * B_SLICE_BYTES + A_SMEM_TILE : B_STAGE_BYTES;
    constexpr int RING = AS ? (NSLB == 1 ? 5 : 3) : B_STAGES;
    static_assert(RING <= RING_MAX && RING * STAGE_BYTES <= RING_BYTES_MAX && STAGE_BYTES % 1024 == 0, "ring");

    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *b_full = bars, *b_empty = b_full + RING_MAX;
    uint64_t *a_full = b_empty + RING_MAX, *a_empty = a_full + A_STAGES;
    uint64_t *acc_full = a_empty + A_STAGES, *acc_empty = acc_full + NBUF;
    int *prefix = reinterpret_cast<int *>(smem + L::SCHED_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rt_n = a.row_tiles;
    const int rb_stride = a.row_tiles * TILE_ROWS;

    if (tid == 0) {
        for (int i = 0; i < RING; ++i) {
            mbar_init(&b_full[i], 1);  // the token copies (expect-tx)
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < A_STAGES; ++i) {
            mbar_init(&a_full[i], 4);  // the four warps of the slot's decoder group
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < NBUF; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], N_EPI_WARPS);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == WARP_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == WARP_BLOAD)
        schedule_prefix(a.grp_count, a.G, rt_n, NMAX, prefix, lane);
    if (warp == WARP_BLOAD && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b2)) : "memory");
        if (AS)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = prefix[a.G];
    const int nstages = a.kchunks * (CHUNK_K / KST);
    // first weight chunk of row tile w.rt of group w.g
    auto tile_src = [&](const WorkItem &w) {
        return a.wbase + (size_t)w.g * a.group_bytes + (size_t)w.rt * a.kchunks * (size_t)a.chunk_bytes;
    };

    // Every role walks the same static schedule t = blockIdx.x, +gridDim.x, ...
    // (decompose() over row tiles: w.rt is the tile).  Single-thread roles keep
    // the whole warp in the loop (lane 0 issues).
    if (warp == WARP_BLOAD) {
        // ---------------------------------------------------------- token tiles (B) -> stage ring
        uint32_t sc = 0, armed = 0, armed_par = 0;
        bool ok = true;
        // L2 prefetch cursor over this CTA's (item, chunk) sequence, PF_CHUNKS chunks
        // ahead of the loads
        int pf_t = blockIdx.x, pf_c = 0;
        const uint8_t *pf_src = nullptr;
        auto pf_next = [&]() {  // prefetch one chunk and advance
            if (pf_t >= total)
                return;
            if (pf_c == 0)
                pf_src = tile_src(decompose(pf_t, prefix, a.grp_count, a.G, rt_n, NMAX));
            if (lane == 0)
                prefetch_l2(pf_src + (size_t)pf_c * a.chunk_bytes, (uint32_t)a.chunk_bytes);
            if (++pf_c == a.kchunks) {
                pf_c = 0;
                pf_t += gridDim.x;
            }
        };
        for (int i = 0; i < PF_CHUNKS; ++i)
            pf_next();
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, rt_n, NMAX);
            int row0;
            const CUtensorMap *m0 = &map_b;
            if (GU && w.g >= a.E) {  // shared groups read the token rows by token, routed groups gathered rows
                row0 = w.tok0;
                m0 = &map_b2;
            } else {
                row0 = a.grp_start[w.g] + w.tok0;
            }
            // whole boxes of brows rows (past the tile's tokens: rows the MMAs do not
            // read, or zero fill past the tensor's last row)
            const int nbox = (w.n_mma + a.brows - 1) / a.brows;
            const int box_bytes = a.brows * HALF_K * 2;
            const uint32_t bytes = (uint32_t)(nbox * box_bytes * NSLB) + (AS ? (uint32_t)A_SMEM_TILE : 0u);
            // AS: the item's A tiles, rows of the TILE store seen as [halves * 128][64]
            const int a_row0 = ((w.g * rt_n + w.rt) * a.kchunks) * 2 * TILE_ROWS;
            for (int st = 0; st < nstages; ++st, ++sc) {
                const int slot = sc % RING;
                const uint32_t ph = (sc / RING) & 1;
                if (!(ok = mbar_wait_sleep_warp(&b_empty[slot], ph ^ 1, abort_flag, a.err, lane)))
                    break;
                if (KST == CHUNK_K || (st & 1) == 0)
                    pf_next();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&b_full[slot], bytes);
                    uint8_t *bdst = smem + slot * STAGE_BYTES;
                    if (AS)
                        tma_2d(bdst + NSLB * B_SLICE_BYTES, &map_a, 0, a_row0 + st * TILE_ROWS, &b_full[slot]);
                    // the stage's two swizzled tiles: two 64-wide K slices of one plane,
                    // or one slice of the h hi and lo planes
                    for (int b = 0; b < nbox; ++b) {
                        if (NSLB == 1) {
                            tma_2d(bdst + b * box_bytes, m0, st * KST, row0 + b * a.brows, &b_full[slot]);
                        } else if (NB == 1) {
                            tma_2d(bdst + b * box_bytes, m0, st * KST, row0 + b * a.brows, &b_full[slot]);
                            tma_2d(bdst + B_SLICE_BYTES + b * box_bytes, m0, st * KST + HALF_K, row0 + b * a.brows,
                                   &b_full[slot]);
                        } else {
                            tma_2d(bdst + b * box_bytes, m0, st * KST, row0 + b * a.brows, &b_full[slot]);
                            tma_2d(bdst + B_SLICE_BYTES + b * box_bytes, &map_b2, st * KST, row0 + b * a.brows,
                                   &b_full[slot]);
                        }
                    }
                }
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (ph << slot);
            }
        }
        // drain: every armed stage's B tiles have landed (returns at once on the
        // normal path, where the MMA has consumed them; bounded after an abort)
        if (lane == 0)
            for (int s = 0; s < RING; ++s)
                if (armed & (1u << s))
                    mbar_drain(&b_full[s], (armed_par >> s) & 1);
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------- MMA issue
        // Lane 0 alone runs this role: its waits, fences and MMAs need no
        // warp-wide step between stages.
        if (lane == 0) {
            uint32_t sc = 0, tc = 0;
            const uint64_t desc0 = sw128_desc(smem_addr(smem));  // K-major SW128 descriptor of B stage 0
            bool ok = true, partial = false;  // partial: an aborted item has MMAs in flight
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const WorkItem w = decompose(t, prefix, a.grp_count, a.G, rt_n, NMAX);
                const int buf = tc % NBUF;
                if (!(ok = mbar_wait(&acc_empty[buf], ((tc / NBUF) & 1) ^ 1, abort_flag, a.err)))
                    break;
                tc_fence_after();
                const uint32_t idesc = make_idesc<OP == OP_BF16 ? OP_BF16 : OP_F16>(w.n_mma);
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * NMAX);
                for (int st = 0; st < nstages; ++st, ++sc) {
                    // a_full completes once the stage's A is in tensor memory and its B
                    // tiles have landed (the decoder group waits for the token copy
                    // before it arrives), so each stage costs the MMA thread one wait
                    const int bs = sc % RING, as = sc % A_STAGES;
                    // AS: the stage's A and B tiles come together on b_full
                    if (!(ok = AS ? mbar_wait(&b_full[bs], (sc / RING) & 1, abort_flag, a.err)
                                  : mbar_wait(&a_full[as], (sc / A_STAGES) & 1, abort_flag, a.err)))
                        break;
                    tc_fence_after();
                    // descriptors of this slot: base plus the slot's offset (address field = bytes >> 4)
                    const uint64_t bd = desc0 + (uint64_t)((bs * STAGE_BYTES) >> 4);
                    const uint32_t at = tmem_base + (uint32_t)(TMEM_A0 + as * A_SLOT_COLS);
                    if (AS) {
                        const uint64_t ad = bd + (uint64_t)((NSLB * B_SLICE_BYTES) >> 4);
                        tc_mma4_ss(d_tmem, ad, bd, idesc, st);
                        if (NB == 2)
                            tc_mma4_ss(d_tmem, ad, bd + (uint64_t)(B_SLICE_BYTES >> 4), idesc, 1u);
                    } else if (OP == OP_I4) {
                        // the stage's 64 values of K: the hi tile (columns 0..31), then the lo tile
                        tc_mma4(d_tmem, at, bd, idesc, st);
                        tc_mma4(d_tmem, at + 32, bd, idesc, 1u);
                    } else if (NB == 1) {
#pragma unroll
                        for (int sl = 0; sl < NSL; ++sl)
                            tc_mma4(d_tmem, at + 32 * sl, bd + (uint64_t)((sl * B_SLICE_BYTES) >> 4), idesc,
                                    st > 0 || sl > 0);
                    } else {
                        tc_mma4(d_tmem, at, bd, idesc, st);
                        tc_mma4(d_tmem, at, bd + (uint64_t)(B_SLICE_BYTES >> 4), idesc, 1u);
                    }
                    tc_commit(&b_empty[bs]);
                    if (!AS)
                        tc_commit(&a_empty[as]);
                    partial = true;
                }
                if (!ok)
                    break;
                tc_commit(&acc_full[buf]);
                partial = false;
            }
            // drain: every MMA issued has completed.  After an abort in the middle of
            // item tc, its MMAs are committed to its accumulator barrier first.
            if (partial) {
                tc_commit(&acc_full[tc % NBUF]);
                mbar_drain(&acc_full[tc % NBUF], (tc / NBUF) & 1);
            } else if (tc > 0) {
                mbar_drain(&acc_full[(tc - 1) % NBUF], ((tc - 1) / NBUF) & 1);
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ---------------------------------------------------------- decoders
        // Group gi decodes every N_DEC_GROUPS-th stage (gs = gi, gi + 2, ...: A
        // slot gi) in full; its warp of lane quadrant q = warp % 4 decodes rows
        // 32q..32q+31 (lane = row) of the item's row tile over the stage's KST
        // values of K into the slot's columns of the tensor-memory A ring, so each
        // warp pays the stage hand-off (wait, fences, arrive) once per two stages.  A lane
        // loads its next stage's raw codes and scales straight from global
        // memory (into registers) as soon as it has handed over the current one;
        // the token loader has prefetched them into L2.
        const int q = warp & 3;
        const int gi = (warp - WARP_DEC0) >> 2;
        const int r = 32 * q + lane;  // row inside the tile
        const uint32_t tlane = (uint32_t)(32 * q) << 16;
        const int n_items = total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
        const int total_st = AS ? 0 : n_items * nstages;  // AS: the A tiles come by TMA, no decoding
        uint4 rc[NBLK];   // MXFP4: 16 code bytes per 32-value block
        uint32_t re[NBLK], rb = 127;
        const uint8_t *src = nullptr;  // the stage's chunk
        int kh = 0;                    // 64-wide half of the chunk (stages of 64 values)
        int cached_ii = -1;
        const uint8_t *tile0 = nullptr;
        uint32_t base_c = 127;
        auto locate = [&](int gs) {
            const int ii = gs / nstages, st = gs - ii * nstages;
            if (ii != cached_ii) {
                cached_ii = ii;
                const WorkItem w = decompose(blockIdx.x + ii * gridDim.x, prefix, a.grp_count, a.G, rt_n, NMAX);
                tile0 = tile_src(w);
                if (FT)
                    base_c = __ldg(a.row_base + (size_t)w.g * rb_stride + w.rt * TILE_ROWS + r);
            }
            src = tile0 + (size_t)(st * KST / CHUNK_K) * a.chunk_bytes;
            kh = KST == CHUNK_K ? 0 : (st & 1);
        };
        auto fetch = [&](int gs) {  // MXFP4: the stage's codes and scales into registers
            if (WFMT == FMT_BF16)
                return;
            locate(gs);
            rb = base_c;
#pragma unroll
            for (int b = 0; b < NBLK; ++b) {
                const int blk = NBLK == 4 ? b : 2 * kh + b;  // 32-value block of the chunk
                if (OP == OP_I4) {
                    // TILE_I4: 16 code bytes of (block, row r); the FP16 scale and the zero point
                    rc[b] = __ldg(reinterpret_cast<const uint4 *>(src + (blk * TILE_ROWS + r) * 16));
                    re[b] = (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(src + CHUNK_MX_CODE_BYTES) +
                                            blk * TILE_ROWS + r) |
                            ((uint32_t)__ldg(src + CHUNK_MX_CODE_BYTES + CHUNK_I4_SCALE_BYTES + blk * TILE_ROWS + r)
                             << 16);
                } else if (OP == OP_F16) {
                    // TILE_F16: 16 code bytes of (block, row r), then the E8M0 bytes
                    rc[b] = __ldg(reinterpret_cast<const uint4 *>(src + (blk * TILE_ROWS + r) * 16));
                    re[b] = __ldg(src + CHUNK_MX_CODE_BYTES + blk * TILE_ROWS + r);
                } else {
                    // TILE: repacked words of (half blk / 2, block blk % 2) of row r, then the scales
                    rc[b] = __ldg(reinterpret_cast<const uint4 *>(src + (blk >> 1) * (CHUNK_MX_CODE_BYTES / 2) +
                                                                  r * 32 + (blk & 1) * 16));
                    re[b] = __ldg(src + CHUNK_MX_CODE_BYTES + r * 4 + blk);
                }
            }
        };
        bool ok = true;
        int gs = gi;
        if (gs < total_st)
            fetch(gs);
        for (; gs < total_st && ok; gs += N_DEC_GROUPS) {
            const int slot = gi;  // = gs % A_STAGES
            if (!(ok = mbar_wait_warp(&a_empty[slot], ((gs / A_STAGES) & 1) ^ 1, abort_flag, a.err, lane)))
                break;
            tc_fence_after();
            if (WFMT == FMT_BF16)
                locate(gs);
#pragma unroll
            for (int b = 0; b < NBLK; ++b) {
                uint32_t o[16];
                if (WFMT == FMT_BF16) {
                    // BF16 TILE: 64 values of half (k / 64) of row r
                    const int k0 = (NBLK == 4 ? 0 : kh * HALF_K) + 32 * b;
                    const uint4 *p = reinterpret_cast<const uint4 *>(src + (k0 >> 6) * (CHUNK_BF16_BYTES / 2) + r * 128 +
                                                                     (k0 & 63) * 2);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 x4 = __ldg(p + v);
                        o[4 * v] = x4.x;
                        o[4 * v + 1] = x4.y;
                        o[4 * v + 2] = x4.z;
                        o[4 * v + 3] = x4.w;
                    }
                } else if (OP == OP_I4) {
                    // w = s (q - z) relative to the row base: s' = s * 2^-b_row (below 2^12),
                    // hi = fp16(s' (q - z)), lo = s' (q - z) - hi (exact in FP16: at most
                    // four significant bits left), into two tensor-memory tiles
                    const float sf = __half2float(__ushort_as_half((unsigned short)(re[b] & 0xFFFFu))) *
                                     __int_as_float((254 - (int)rb) << 23);
                    const uint32_t sh = (uint32_t)__half_as_ushort(__float2half_rn(sf));
                    const uint32_t s2 = sh | (sh << 16);
                    const uint32_t zz = (0x6400u + (re[b] >> 16)) * 0x10001u;
                    uint32_t lo[16];
                    const uint32_t words[4] = {rc[b].x, rc[b].y, rc[b].z, rc[b].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            i4_pair_hilo(words[c] >> (4 * p), zz, s2, o[4 * c + p], lo[4 * c + p]);
                    tmem_st16(tmem_base + tlane + (uint32_t)(TMEM_A0 + slot * A_SLOT_COLS + 32 + b * 16), lo);
                } else if (OP == OP_F16) {
                    int d = (int)re[b] - (int)rb;
                    d = d < -24 ? -24 : (d > 0 ? 0 : d);  // only blocks past K (code 0) fall outside [-23, 0]
                    const uint32_t s2 = f16x2_pow2(d);
                    e2m1x8_f16(rc[b].x, s2, o);
                    e2m1x8_f16(rc[b].y, s2, o + 4);
                    e2m1x8_f16(rc[b].z, s2, o + 8);
                    e2m1x8_f16(rc[b].w, s2, o + 12);
                } else {
                    const uint32_t s2 = e8m0_to_bf16x2(re[b]);
                    decode_word(rc[b].x, s2, o);
                    decode_word(rc[b].y, s2, o + 4);
                    decode_word(rc[b].z, s2, o + 8);
                    decode_word(rc[b].w, s2, o + 12);
                }
                tmem_st16(tmem_base + tlane + (uint32_t)(TMEM_A0 + slot * A_SLOT_COLS + b * 16), o);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            // the stage's token tiles must have landed too: the MMA thread waits on
            // a_full alone (this group waited on this B slot four stages ago, so the
            // parity below is never two phases ahead)
            if (!(ok = mbar_wait_warp(&b_full[gs % RING], (gs / RING) & 1, abort_flag, a.err, lane)))
                break;
            if (lane == 0)
                mbar_arrive(&a_full[slot]);
            if (gs + N_DEC_GROUPS < total_st)
                fetch(gs + N_DEC_GROUPS);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                   // tensor-memory lane quadrant of this warp
        const int eh = (warp - WARP_EPI0) >> 2;   // which column chunks of the quadrant it takes
        // this warp's column scales (FP16 token operands), indexed by column
        float *csc = reinterpret_cast<float *>(smem + L::COLSC_OFF) + (warp - WARP_EPI0) * NMAX;
        float *hsc = reinterpret_cast<float *>(smem + L::HSC_OFF) + (warp - WARP_EPI0) * NMAX;  // gate|up, FP16
        // columns per tensor-memory wait: gate|up 32, down 16
        constexpr int EC = GU ? 32 : 16;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, rt_n, NMAX);
            const int pos0 = a.grp_start[w.g] + w.tok0;
            // FP16 operands: the power of two of each of this warp's columns' token row
            // (gate|up) or h row (down), staged in shared memory while the item's MMAs
            // still run
            if (FT) {
#pragma unroll 1
                for (int i = 0; i < NMAX / (2 * EC); ++i)
                    for (int c = EC * eh + 2 * EC * i + lane; c < EC * eh + 2 * EC * i + EC && c < w.nvalid; c += 32) {
                        if (GU) {
                            csc[c] = pow2i(__ldg(a.xsp + pos0 + c));
                            hsc[c] = pow2i(-__ldg(a.hsp + pos0 + c));
                        } else {
                            // the h row's power of two over the y row's
                            csc[c] = pow2i(__ldg(a.hsp + pos0 + c) - __ldg(a.ys + pos0 + c));
                        }
                    }
                __syncwarp();
            }
            const int buf = tc % NBUF;
            if (!mbar_wait_sleep_warp(&acc_full[buf], (tc / NBUF) & 1, abort_flag, a.err, lane))
                break;
            tc_fence_after();
            const int rt = w.rt;
            const int row = 32 * q + lane;
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * NMAX);
            // FP16 operands: this row's weight scale 2^(b - 127) (exact; a subnormal for b = 0)
            const float wsc = FT
                                  ? ldexpf(1.0f, (int)__ldg(a.row_base + (size_t)w.g * rb_stride + rt * TILE_ROWS + row) - 127)
                                  : 1.0f;
            // column groups of this warp: EC columns at c0 = EC * eh + 2 * EC * i
            constexpr int NG = NMAX / (2 * EC);
#pragma unroll 1
            for (int i = 0; i < NG; ++i) {
                const int c0 = EC * eh + 2 * EC * i;
                if (c0 >= w.n_mma)
                    break;
                // EC columns per wait (a second load may lie past n_mma, inside the
                // accumulator, and is then ignored)
                float v2[EC];
                if constexpr (EC == 32)
                    tmem_ld32(taddr + c0, v2);
                else
                    tmem_ld16(taddr + c0, v2);
#pragma unroll
                for (int half = 0; half < EC / 16; ++half) {
                    const int c1 = c0 + 16 * half;
                    if (c1 >= w.n_mma)
                        break;
                    const float *v = v2 + 16 * half;
                    if (GU) {
                        // rows 16*gr + i: gate of feature 8*gr + i%8 when i < 8, up when i >= 8;
                        // the gate lane finishes tokens c1..c1+7, its up partner (lane ^ 8) c1+8..c1+15
                        const int n = gu_row_feature(rt, row);
                        const bool up_lane = gu_row_is_up(lane);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const float send = (up_lane ? v[jj] : v[8 + jj]) * wsc;
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
                            float gv = up_lane ? recv : v[jj] * wsc;
                            float uv = up_lane ? v[8 + jj] * wsc : recv;
                            const int tok = c1 + (up_lane ? 8 : 0) + jj;
                            const bool valid = tok < w.nvalid && n < a.I;
                            if (FT) {
                                // undo the token row's power of two; h leaves in FP16 times
                                // the position's power of two
                                if (valid) {
                                    gv *= csc[tok];
                                    uv *= csc[tok];
                                    const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                                    a.h16[(size_t)(pos0 + tok) * a.I + n] = __half_as_ushort(__float2half_rn(hv * hsc[tok]));
                                }
                            } else if (valid) {
                                const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                                const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                                const __nv_bfloat16 lb = __float2bfloat16_rn(hv - __bfloat162float(hb));
                                const size_t o = (size_t)(pos0 + tok) * a.I + n;
                                a.h_out[o] = __bfloat16_as_ushort(hb);
                                a.h_out[o + a.h_plane] = __bfloat16_as_ushort(lb);
                            }
                        }
                    } else {
                        const int m = rt * TILE_ROWS + row;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            if (m < a.H && c1 + jj < w.nvalid) {
                                const size_t o = (size_t)(pos0 + c1 + jj) * a.H + m;
                                if (FT)
                                    a.y16[o] = __half_as_ushort(__float2half_rn(v[jj] * wsc * csc[c1 + jj]));
                                else
                                    a.y_out[o] = v[jj];
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

template <bool GU, int OP, int WFMT>
cudaError_t launch_cfg(const TcArgs &a, const CUtensorMap &m1, const CUtensorMap &m2, const CUtensorMap &ma,
                       cudaStream_t st)
{
    constexpr int SMEM = Smem::TOTAL;
    auto kern = gemm_tc_kernel<GU, OP, WFMT>;
    static std::atomic<int> attr_set[MAX_DEVICES];
    cudaError_t e = smem_limit_once(attr_set, (const void *)kern, SMEM);
    if (e != cudaSuccess)
        return e;
    kern<<<sm_count(), NUM_THREADS, SMEM, st>>>(a, m1, m2, ma);
    return cudaGetLastError();
}

// The A tensor map of a BF16 TILE store: its 64-wide halves of 128 rows as a
// [G * row_tiles * kchunks * 2 * 128][64] BF16 tensor, 128-row boxes.
cudaError_t make_a_map(CUtensorMap *m, const WeightStore &w, int G)
{
    const long long rows = (long long)G * w.row_tiles * w.kchunks * 2 * TILE_ROWS;
    return make_map(m, w.base, rows, HALF_K, TILE_ROWS);
}

template <bool GU>
cudaError_t launch_any(const TcArgs &a, const WeightStore &w, int fmt, bool f16, const CUtensorMap &m1,
                       const CUtensorMap &m2, cudaStream_t st)
{
    if (f16)
        return fmt == FMT_MXFP4  ? launch_cfg<GU, OP_F16, FMT_MXFP4>(a, m1, m2, m1, st)
               : fmt == FMT_INT4 ? launch_cfg<GU, OP_I4, FMT_INT4>(a, m1, m2, m1, st)
                                 : cudaErrorInvalidValue;
    if (fmt == FMT_MXFP4)
        return launch_cfg<GU, OP_BF16, FMT_MXFP4>(a, m1, m2, m1, st);
    CUtensorMap ma;
    cudaError_t e = make_a_map(&ma, w, a.G);
    if (e != cudaSuccess)
        return e;
    return launch_cfg<GU, OP_BF16, FMT_BF16>(a, m1, m2, ma, st);
}

TcArgs base_args(const Plan &p, const WeightStore &w)
{
    TcArgs a{};
    a.wbase = w.base;
    a.group_bytes = w.group_bytes;
    a.kchunks = w.kchunks;
    a.chunk_bytes = w.chunk_bytes;
    a.row_tiles = w.row_tiles;
    a.row_base = w.row_base;
    a.grp_start = p.grp_start;
    a.grp_count = p.grp_count;
    a.E = p.E;
    a.G = p.G;
    a.I = p.I;
    a.H = p.H;
    a.row_token = p.row_token;
    a.err = p.err;
    return a;
}

}  // namespace

// x_perm[p] = x[row_token[p]] for the routed positions p < T*k (16-byte copies)
__global__ void gather_rows_kernel(const uint4 *__restrict__ x, const int *__restrict__ row_token, int n_rows,
                                   int row_vecs, uint4 *__restrict__ out)
{
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    long long total = (long long)n_rows * row_vecs;
    for (; i < total; i += (long long)gridDim.x * blockDim.x) {
        const long long p = i / row_vecs, c = i % row_vecs;
        out[i] = x[(long long)row_token[p] * row_vecs + c];
    }
}

cudaError_t launch_gather_rows(const Plan &p, const uint16_t *x, cudaStream_t st)
{
    const int n = p.T * p.k;
    if (n == 0)
        return cudaSuccess;
    const int row_vecs = p.H / 8;
    long long total = (long long)n * row_vecs;
    long long blocks = (total + 255) / 256;
    if (blocks > 4 * 152 * 8)
        blocks = 4 * 152 * 8;
    gather_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4 *>(x), p.row_token, n, row_vecs,
                                                         reinterpret_cast<uint4 *>(p.x_perm));
    return cudaGetLastError();
}

// FP16 token rows, and the power of two of each position's h.  One CTA per
// token t.
//  - xs[t] = floor(log2 max|x_t|) - 14 (0 for an all-zero row, clamped to
//    [-100, 100]) and x16 = x_t * 2^-xs[t] in FP16, natural K order: the
//    largest |x| of a token lands in [2^14, 2^15); a BF16 value has 8
//    significant bits, so the conversion is exact for every element within
//    2^31 of the token's largest.  The row goes to x16[t] (read by the shared
//    groups and dense slices) and to x_perm[p] for each routed position p of
//    the token (slot_pos), so that no separate gather pass reads it back.
//  - hsp[p]: h = SiLU(g) * u obeys |h| <= |g| |u| (|SiLU(z)| <= |z|) and, by
//    Cauchy-Schwarz, |g_n| |u_n| <= |x|^2 |w_g,n| |w_u,n|.  With
//    L_e = max_n log2(|w_g,n| |w_u,n|) over the features of the position's
//    group (computed at load, see gu_norm_kernel) and log2 |x_t|^2 from the
//    FP16 row, hsp[p] = ceil(log2 bound + 0.01) - 15 keeps |h| * 2^-hsp below
//    2^15, inside FP16, before h exists; FP16 keeps 11 significant bits of
//    every value above 2^-14 in those units.
//  - ys[p]: the power of two of the position's FP16 y row (y_scale_of), from
//    the same h bound and the load-time row norms of the down matrix.
//  - xsp[p] = xs[t] for every position of the token.
__device__ __forceinline__ float ordered_key_to_float(int key)
{
    const uint32_t k = (uint32_t)key;
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ int h_scale_of(float lx, float lw)
{
    const float l = lx + lw;
    int hs = l > -1000.f ? (int)ceilf(l + 0.01f) - 15 : -100;
    return hs < -100 ? -100 : (hs > 100 ? 100 : hs);
}

// Power of two of a position's FP16 y row: |y_m| <= |h| |w_d,m| <= sqrt(I) *
// max|h| * max_m |w_d,m|, and max|h| <= 2^(hs + 15), so ys = hs + ceil(log2
// sqrt(I) + ld + 0.01) keeps |y| * 2^-ys below 2^15 (ld = max_m log2 |w_d,m| of
// the group), clamped so that 2^ys and 2^(hs - ys) stay normal FP32 numbers.
__device__ __forceinline__ int y_scale_of(int hs, int I, float ld)
{
    const float l = 0.5f * __log2f((float)I) + ld;
    int ys = l > -1000.f ? hs + (int)ceilf(l + 0.01f) : hs - 126;
    ys = ys < hs - 126 ? hs - 126 : (ys > hs + 126 ? hs + 126 : ys);
    return ys < -126 ? -126 : (ys > 126 ? 126 : ys);
}

__global__ void token_prep_f16_kernel(const uint16_t *__restrict__ x, int H, uint16_t *__restrict__ x16,
                                      uint16_t *__restrict__ x_perm, int *__restrict__ xs, int *__restrict__ xsp,
                                      int *__restrict__ hsp, const int *__restrict__ slot_pos,
                                      const int *__restrict__ topk_ids, const int *__restrict__ gkey,
                                      const int *__restrict__ dkey, int *__restrict__ ys, int I, int k, int E, int T,
                                      int S)
{
    __shared__ uint32_t red[32];
    __shared__ float fred[32];
    __shared__ int pos[32];  // routed positions of this token (k <= 32)
    const int t = blockIdx.x;
    const int n_routed = T * k;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    const int nv = H / 8;
    if ((int)threadIdx.x < k)
        pos[threadIdx.x] = slot_pos[(size_t)t * k + threadIdx.x];
    uint32_t mx = 0;  // max |x| as BF16 bits without sign (monotonic for finite values)
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    }
    for (int o = 16; o > 0; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        mx = max(mx, red[i]);
    int sc = mx == 0 ? 0 : (int)(mx >> 7) - 127 - 14;
    sc = sc < -100 ? -100 : (sc > 100 ? 100 : sc);
    const float mul = __int_as_float((127 - sc) << 23);
    uint4 *dst = reinterpret_cast<uint4 *>(x16 + (size_t)t * H);
    float ss = 0.f;  // sum of squares of the FP16 row (each below 2^30: no overflow at any H here)
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half lo = __float2half_rn(__uint_as_float(w[j] << 16) * mul);
            const __half hi = __float2half_rn(__uint_as_float(w[j] & 0xFFFF0000u) * mul);
            const float fl = __half2float(lo), fh = __half2float(hi);
            ss = fmaf(fl, fl, fmaf(fh, fh, ss));
            o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        dst[i] = ov;
        for (int j = 0; j < k; ++j)
            if (pos[j] >= 0)  // (an empty slot of caller routing has no position)
                reinterpret_cast<uint4 *>(x_perm + (size_t)pos[j] * H)[i] = ov;
    }
    for (int o = 16; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0)
        fred[threadIdx.x >> 5] = ss;
    __syncthreads();
    ss = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        ss += fred[i];
    // log2 |x_t|^2 (the row's FP16 values times 2^xs), rounded up a little for the
    // FP32 sum's own rounding
    const float lx = ss > 0.f ? 2.f * (float)sc + __log2f(ss) + 0.01f : -2000.f;
    if (threadIdx.x == 0)
        xs[t] = sc;
    if ((int)threadIdx.x < k && pos[threadIdx.x] >= 0) {
        const int p = pos[threadIdx.x];
        const int e = topk_ids[(size_t)t * k + threadIdx.x];
        const int hs = h_scale_of(lx, ordered_key_to_float(gkey[e]));
        xsp[p] = sc;
        hsp[p] = hs;
        ys[p] = y_scale_of(hs, I, ordered_key_to_float(dkey[e]));
    }
    for (int s = threadIdx.x; s < S; s += blockDim.x) {  // shared groups / dense slices: position n + s*T + t
        const size_t p = (size_t)n_routed + (size_t)s * T + t;
        const int hs = h_scale_of(lx, ordered_key_to_float(gkey[E + s]));
        xsp[p] = sc;
        hsp[p] = hs;
        ys[p] = y_scale_of(hs, I, ordered_key_to_float(dkey[E + s]));
    }
}

cudaError_t launch_token_prep_f16(const Plan &p, const uint16_t *x, const int *gu_norm_key, const int *dn_norm_key,
                                  cudaStream_t st)
{
    if (p.T == 0)
        return cudaSuccess;
    if (p.k > 32)
        return cudaErrorInvalidValue;
    token_prep_f16_kernel<<<p.T, 256, 0, st>>>(x, p.H, p.x16, p.x_perm, p.xs, p.xsp, p.hsp, p.slot_pos, p.topk_ids,
                                               gu_norm_key, dn_norm_key, p.ys, p.I, p.k, p.E, p.T, p.S);
    return cudaGetLastError();
}

cudaError_t launch_gemm_gate_up_tc(const Plan &p, const WeightStore &w, int fmt, bool f16, const uint16_t *x_rows,
                                   cudaStream_t st)
{
    TcArgs a = base_args(p, w);
    a.h_out = p.h;
    a.h_plane = (long long)p.P * p.I;
    a.h16 = p.h16;
    a.hsp = p.hsp;
    a.xsp = p.xsp;
    a.brows = p.T >= B_BOX_ROWS_BIG && (p.T * p.k == 0 || p.T * p.k >= B_BOX_ROWS_BIG) ? B_BOX_ROWS_BIG
                                                                                       : B_BOX_ROWS_SMALL;
    CUtensorMap m1, m2;
    cudaError_t e = make_map(&m2, x_rows, p.T, p.H, a.brows);
    if (e != cudaSuccess)
        return e;
    if (p.T * p.k > 0) {
        if ((e = make_map(&m1, p.x_perm, (long long)p.T * p.k, p.H, a.brows)) != cudaSuccess)
            return e;
    } else {
        m1 = m2;
    }
    return launch_any<true>(a, w, fmt, f16, m1, m2, st);
}

cudaError_t launch_gemm_down_tc(const Plan &p, const WeightStore &w, int fmt, bool f16, cudaStream_t st)
{
    TcArgs a = base_args(p, w);
    a.y_out = p.y;
    a.y16 = reinterpret_cast<uint16_t *>(p.y);
    a.ys = p.ys;
    a.hsp = p.hsp;
    a.brows = p.P >= B_BOX_ROWS_BIG ? B_BOX_ROWS_BIG : B_BOX_ROWS_SMALL;
    CUtensorMap m1, m2;
    cudaError_t e;
    if (f16) {
        if ((e = make_map(&m1, p.h16, p.P, p.I, a.brows)) != cudaSuccess)
            return e;
        m2 = m1;
    } else {
        if ((e = make_map(&m1, p.h, p.P, p.I, a.brows)) != cudaSuccess)
            return e;
        if ((e = make_map(&m2, p.h + (size_t)p.P * p.I, p.P, p.I, a.brows)) != cudaSuccess)
            return e;
    }
    return launch_any<false>(a, w, fmt, f16, m1, m2, st);
}

}  // namespace moe
