// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a): gate|up with fused SwiGLU, and down.
//
// Operation (per expert group g and token position p of the group):
//   gate|up:  g_n = x_p . W_g[n],  u_n = x_p . W_u[n],  h_pn = SiLU(g_n) * u_n
//   down:     y_pm = h_p . W_d[m]
// with the SwiGLU expert of "Cascadia: Resident 975B MoE Inference on Eleven
// AI PCs" §3.1 and MXFP4 weights decoded inside the reduction as in
// "DeepSeek-V4-Flash on a four-GPU Ampere workstation", section "MXFP4 is not
// NVFP4, and the difference matters on Ampere" (scale loaded once per 32-value
// block, FP32 accumulation, no decoded copy of an expert in device memory).
//
// Mapping to the hardware ("swap-AB": weights are the M side):
//   D[128 weight rows, N tokens] (FP32, TMEM)  +=  A[128 rows, K] . B[N tokens, K]^T
//   A = 128 weight rows decoded to BF16 in shared memory by CUDA-core warps,
//       straight from the MXFP4 chunks in global memory (each decoder thread
//       keeps its next stages' raw bytes in flight in registers);
//   B = token rows (BF16; for down the hi and lo BF16 planes of h, two MMAs per
//       K step), loaded by TMA into the 128-byte-swizzled K-major layout;
//   MMA = tcgen05.mma kind::f16, M=128, N = 16..NMAX, K=16, issued by one thread.
// A work item is (group, pair of 128-row tiles, token tile): both row tiles
// share every staged token tile, so a 64 KB stage feeds 2 x 128 x N x 64
// multiply-adds -- twice as many per staged byte as one row tile.
// One CTA per SM walks a static schedule of work items.  Warp roles:
//   warp 0      TMA-loads token tiles (B) into the stage ring
//   warp 1      allocates TMEM, issues the MMAs, commits to mbarriers
//   warps 2-17  decode MXFP4 (or copy BF16) into the swizzled A stages
//   warps 18-25 epilogue, two warps per TMEM lane quadrant splitting the
//               columns: TMEM -> registers, SwiGLU (gate|up) or FP32 y (down)
// Two TMEM accumulator sets (when N allows) let the epilogue of one work item
// overlap the MMAs of the next.  Every mbarrier wait is bounded: on a timeout
// the kernel records DEV_ERR_WAIT_TIMEOUT, stops issuing work, waits (bounded)
// for the copies and MMAs it has in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "mx_decode.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int N_DEC_WARPS = 16;
constexpr int N_EPI_WARPS = 8;  // two per TMEM lane quadrant, splitting the columns
constexpr int NUM_THREADS = (2 + N_DEC_WARPS + N_EPI_WARPS) * 32;
constexpr int WARP_BLOAD = 0, WARP_MMA = 1, WARP_DEC0 = 2, WARP_EPI0 = WARP_DEC0 + N_DEC_WARPS;
constexpr int A_STAGE_BYTES = TILE_ROWS * HALF_K * 2;  // 16 KB: 128 rows x 64 BF16
// B operand TMA boxes: 64 token rows (8 KB) each, so that a stage takes few
// TMA issues; 16 rows when a B tensor has fewer than 64 rows
constexpr int B_BOX_ROWS_BIG = 64, B_BOX_ROWS_SMALL = 16;

using TcArgs = GemmArgs;

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// The four K=16 MMAs of one 64-wide stage: descriptors advance by 32 bytes
// (2 in the address field) per K step; the first MMA accumulates only when
// acc0 != 0, the other three always.
__device__ __forceinline__ void tc_mma4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
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

// 32 consecutive TMEM columns of this warp's 32 lanes, one wait
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

// Instruction descriptor of kind::f16: BF16 A and B, FP32 D, both K-major,
// M = 128, N given.
__device__ __forceinline__ uint32_t idesc_bf16(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TILE_ROWS >> 4) << 24);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled
// K-major tile whose rows are 128 bytes: 8-row groups are 1024 bytes apart
// and the chunk index is XORed with the row's position in its group.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c)
{
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Work item: (expert group, pair of 128-row weight tiles, token tile).  The two
// row tiles share every token (B) stage, which halves the token bytes staged
// per multiply-add against one row tile per item.
__device__ __forceinline__ int tile_pairs(int row_tiles) { return (row_tiles + 1) / 2; }

template <int NMAX, int NB, int S>
struct Smem {
    static constexpr int A_STAGE = 2 * A_STAGE_BYTES;        // two row tiles x 128 rows x 64 BF16
    static constexpr int B_STAGE = NMAX * HALF_K * 2 * NB;   // NB token planes
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int BAR_OFF = S * STAGE;
    static constexpr int N_BARS = 2 * S + 4;
    static constexpr int SCHED_OFF = BAR_OFF + N_BARS * 8;
    static constexpr int MISC_OFF = SCHED_OFF + (MAX_GROUPS + 1) * 4;
    static constexpr int TOTAL = MISC_OFF + 32 + 1024;  // + alignment slack
};

// Stages of raw weights a decoder thread keeps in flight in registers (its own
// global loads, so no shared-memory staging of the raw chunks is needed).
template <int WFMT>
struct DecPipe {
    static constexpr int PD = WFMT == FMT_MXFP4 ? 4 : 2;
    static constexpr int V = WFMT == FMT_MXFP4 ? 1 : 2;  // vectors per thread, tile and stage (MXFP4: 8 bytes)
};

// ------------------------------------------------------------------ kernel

template <bool GU, int WFMT, int NMAX, int S>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b2)
{
    constexpr int NB = GU ? 1 : 2;
    using L = Smem<NMAX, NB, S>;
    constexpr int NBUF = 4 * NMAX <= 512 ? 2 : 1;      // accumulator sets (two row tiles each)
    constexpr int TMEM_COLS_RAW = 2 * NMAX * NBUF;
    constexpr int TMEM_COLS = TMEM_COLS_RAW < 32 ? 32 : TMEM_COLS_RAW;
    static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
    static_assert(L::TOTAL <= 232448, "shared memory");
    using DP = DecPipe<WFMT>;
    constexpr int PD = DP::PD, V = DP::V;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *ab_full = bars, *ab_empty = bars + S;
    uint64_t *acc_full = bars + 2 * S, *acc_empty = acc_full + 2;
    int *prefix = reinterpret_cast<int *>(smem + L::SCHED_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pairs = tile_pairs(a.row_tiles);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&ab_full[i], 1 + N_DEC_WARPS);
            mbar_init(&ab_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
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
        schedule_prefix(a.grp_count, a.G, pairs, NMAX, prefix, lane);
    if (warp == WARP_BLOAD && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b2)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = prefix[a.G];
    const int nstages = 2 * a.kchunks;

    // Every role walks the same static schedule t = blockIdx.x, +gridDim.x, ...
    // (decompose() over row-tile pairs: w.rt is the pair index).  Single-thread
    // roles keep the whole warp in the loop (lane 0 issues).
    if (warp == WARP_BLOAD) {
        // ---------------------------------------------------------- token tiles (B) -> stage ring
        uint32_t sc = 0, armed = 0, armed_par = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, pairs, NMAX);
            int row0;
            const CUtensorMap *m0 = &map_b;
            if (GU && w.g >= a.E) {  // shared groups read x by token, routed groups gathered rows
                row0 = w.tok0;
                m0 = &map_b2;
            } else {
                row0 = a.grp_start[w.g] + w.tok0;
            }
            // whole boxes of brows rows (past the tile's tokens: rows the MMAs do not
            // read, or zero fill past the tensor's last row)
            const int nbox = (w.n_mma + a.brows - 1) / a.brows;
            const int box_bytes = a.brows * HALF_K * 2;
            const uint32_t bytes = (uint32_t)(nbox * box_bytes * NB);
            for (int st = 0; st < nstages; ++st, ++sc) {
                const int slot = sc % S;
                const uint32_t ph = (sc / S) & 1;
                if (!(ok = mbar_wait_sleep_warp(&ab_empty[slot], ph ^ 1, abort_flag, a.err, lane)))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&ab_full[slot], bytes);
                    uint8_t *bdst = smem + slot * L::STAGE + L::A_STAGE;
                    for (int b = 0; b < nbox; ++b) {
                        tma_2d(bdst + b * box_bytes, m0, st * HALF_K, row0 + b * a.brows, &ab_full[slot]);
                        if (!GU)
                            tma_2d(bdst + NMAX * HALF_K * 2 + b * box_bytes, &map_b2, st * HALF_K,
                                   row0 + b * a.brows, &ab_full[slot]);
                    }
                }
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (ph << slot);
            }
        }
        // drain: every armed stage's B tiles have landed (returns at once on the
        // normal path, where the MMA has consumed them; bounded after an abort)
        if (lane == 0)
            for (int s = 0; s < S; ++s)
                if (armed & (1u << s))
                    mbar_drain(&ab_full[s], (armed_par >> s) & 1);
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------- MMA issue (lane 0)
        uint32_t sc = 0, tc = 0, last_acc = 0, last_par = 0;
        const uint64_t desc0 = sw128_desc(smem_addr(smem));  // K-major SW128 descriptor of stage 0
        bool issued = false, ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, pairs, NMAX);
            const bool two = 2 * w.rt + 1 < a.row_tiles;
            const int buf = NBUF == 2 ? (tc & 1) : 0;
            const uint32_t aph = (NBUF == 2 ? (tc >> 1) : tc) & 1;
            if (!(ok = mbar_wait_sleep_warp(&acc_empty[buf], aph ^ 1, abort_flag, a.err, lane)))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * 2 * NMAX);
            const uint32_t idesc = idesc_bf16(w.n_mma);
            for (int st = 0; st < nstages; ++st, ++sc) {
                const int slot = sc % S;
                if (!(ok = mbar_wait_sleep_warp(&ab_full[slot], (sc / S) & 1, abort_flag, a.err, lane)))
                    break;
                tc_fence_after();
                if (lane == 0) {
                    // descriptors of this slot: base plus the slot's offset (address field = bytes >> 4)
                    const uint64_t ad0 = desc0 + (uint64_t)((slot * L::STAGE) >> 4);
                    const uint64_t bd0 = ad0 + (uint64_t)(L::A_STAGE >> 4);
                    tc_mma4(d_tmem, ad0, bd0, idesc, st);
                    if (!GU)
                        tc_mma4(d_tmem, ad0, bd0 + (uint64_t)((NMAX * HALF_K * 2) >> 4), idesc, 1u);
                    if (two) {
                        const uint64_t ad1 = ad0 + (uint64_t)(A_STAGE_BYTES >> 4);
                        tc_mma4(d_tmem + NMAX, ad1, bd0, idesc, st);
                        if (!GU)
                            tc_mma4(d_tmem + NMAX, ad1, bd0 + (uint64_t)((NMAX * HALF_K * 2) >> 4), idesc, 1u);
                    }
                    tc_commit(&ab_empty[slot]);
                }
                __syncwarp();
                issued = true;
            }
            if (!ok)
                break;
            if (lane == 0)
                tc_commit(&acc_full[buf]);
            __syncwarp();
            last_acc = buf;
            last_par = aph;
        }
        // drain: the MMAs of the last committed item have completed
        if (lane == 0 && issued)
            mbar_drain(&acc_full[last_acc], last_par);
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ---------------------------------------------------------- decoders
        // Thread (r, blk, hf) owns row r of both row tiles and the 16 elements
        // hf of the 32-wide block blk of every 64-wide stage.  It loads its raw
        // codes and scale straight from global memory PD stages ahead (into
        // registers), decodes the current stage into the swizzled A stage and
        // arrives on ab_full once per warp.
        const int dt = tid - WARP_DEC0 * 32;                     // 0..511
        const int r = dt >> 2, blk = (dt >> 1) & 1, hf = dt & 1;  // tile row, block, half of the block
        uint32_t soff[2];                                         // swizzled offsets of this thread's 2 x 16 bytes
#pragma unroll
        for (int c = 0; c < 2; ++c)
            soff[c] = sw128_offset(r, blk * 4 + hf * 2 + c);
        uint2 qc[PD][2][V];                    // raw codes (MXFP4: 8 bytes; BF16: 2 x 8... see V) per tile
        uint4 qb[PD][2][V];                    // BF16 weights: 2 x 16 bytes per tile
        uint32_t qs[PD][2];                    // E8M0 scale bytes (MXFP4)
        (void)qc;
        (void)qb;
        // raw source of the stage PD ahead of the one being decoded; walked with
        // counters (item, stage in item, chunk pointers) so that no division or
        // schedule search runs per stage
        int f_ii = 0, f_st = 0;                // next stage to fetch: item index, stage in item
        const uint8_t *f_src[2] = {nullptr, nullptr};
        const int n_items = total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
        auto set_item = [&](int ii) {
            const WorkItem w = decompose(blockIdx.x + ii * gridDim.x, prefix, a.grp_count, a.G, pairs, NMAX);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int rt = 2 * w.rt + j;
                f_src[j] = rt < a.row_tiles
                               ? a.wbase + (size_t)w.g * a.group_bytes + (size_t)rt * a.kchunks * (size_t)a.chunk_bytes
                               : nullptr;
            }
        };
        if (n_items > 0)
            set_item(0);
        auto fetch = [&](int k) {
            if (f_ii >= n_items)
                return;
            const int h = f_st & 1;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (!f_src[j])
                    continue;
                const uint8_t *ch = f_src[j];
                if (WFMT == FMT_MXFP4) {
                    qc[k][j][0] = __ldg(reinterpret_cast<const uint2 *>(ch + h * (CHUNK_MX_CODE_BYTES / 2) + r * 32 +
                                                                        blk * 16 + hf * 8));
                    qs[k][j] = __ldg(ch + CHUNK_MX_CODE_BYTES + r * 4 + h * 2 + blk);
                } else {
                    const uint4 *src =
                        reinterpret_cast<const uint4 *>(ch + h * (CHUNK_BF16_BYTES / 2) + r * 128 + blk * 64 + hf * 32);
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        qb[k][j][v] = __ldg(src + v);
                }
            }
            // advance: next half of the chunk, next chunk, or the next item
            if (h == 1) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (f_src[j])
                        f_src[j] += a.chunk_bytes;
            }
            if (++f_st == nstages) {
                f_st = 0;
                if (++f_ii < n_items)
                    set_item(f_ii);
            }
        };
        const int total_st = n_items * nstages;
#pragma unroll
        for (int k = 0; k < PD; ++k)
            fetch(k);
        bool ok = true;
        int c_st = 0, c_ii = 0;   // stage being decoded: stage in item, item
        bool two = false;
        if (n_items > 0) {
            const WorkItem w = decompose(blockIdx.x, prefix, a.grp_count, a.G, pairs, NMAX);
            two = 2 * w.rt + 1 < a.row_tiles;
        }
        for (int gs0 = 0; gs0 < total_st && ok; gs0 += PD) {
#pragma unroll
            for (int k = 0; k < PD; ++k) {
                const int gs = gs0 + k;
                if (gs >= total_st)
                    break;
                const int slot = gs % S;
                if (!(ok = mbar_wait_sleep_warp(&ab_empty[slot], ((gs / S) & 1) ^ 1, abort_flag, a.err, lane)))
                    break;
                uint8_t *adst = smem + slot * L::STAGE;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (j == 1 && !two)
                        break;
                    uint8_t *aj = adst + j * A_STAGE_BYTES;
                    if (WFMT == FMT_MXFP4) {
                        const uint32_t s2 = e8m0_to_bf16x2(qs[k][j]);
                        const uint32_t words[2] = {qc[k][j][0].x, qc[k][j][0].y};
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t o[4];
                            decode_word(words[c], s2, o);
                            *reinterpret_cast<uint4 *>(aj + soff[c]) = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            *reinterpret_cast<uint4 *>(aj + soff[c]) = qb[k][j][c];
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ab_full[slot]);
                fetch(k);
                if (++c_st == nstages) {
                    c_st = 0;
                    if (++c_ii < n_items) {
                        const WorkItem w =
                            decompose(blockIdx.x + c_ii * gridDim.x, prefix, a.grp_count, a.G, pairs, NMAX);
                        two = 2 * w.rt + 1 < a.row_tiles;
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const int eh = (warp - WARP_EPI0) >> 2;         // which column chunks of the quadrant it takes
        // columns per TMEM wait: gate|up (whose epilogue the MMAs wait for) 32, down 16
        constexpr int EC = GU ? 32 : 16;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const WorkItem w = decompose(t, prefix, a.grp_count, a.G, pairs, NMAX);
            const int buf = NBUF == 2 ? (tc & 1) : 0;
            const uint32_t aph = (NBUF == 2 ? (tc >> 1) : tc) & 1;
            if (!mbar_wait_sleep_warp(&acc_full[buf], aph, abort_flag, a.err, lane))
                break;
            tc_fence_after();
            const int pos0 = a.grp_start[w.g] + w.tok0;
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                const int rt = 2 * w.rt + j;
                if (rt >= a.row_tiles)
                    break;
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * 2 * NMAX + j * NMAX);
                for (int c0 = EC * eh; c0 < w.n_mma; c0 += 2 * EC) {
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
                        // the gate lane finishes tokens c0..c0+7, its up partner (lane ^ 8) c0+8..c0+15
                        const int n = gu_row_feature(rt, 32 * q + lane);
                        const bool up_lane = gu_row_is_up(lane);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const float send = up_lane ? v[jj] : v[8 + jj];
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
                            const float gv = up_lane ? recv : v[jj];
                            const float uv = up_lane ? v[8 + jj] : recv;
                            const int tok = c1 + (up_lane ? 8 : 0) + jj;
                            if (tok < w.nvalid && n < a.I) {
                                const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                                const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                                const __nv_bfloat16 lb = __float2bfloat16_rn(hv - __bfloat162float(hb));
                                const size_t o = (size_t)(pos0 + tok) * a.I + n;
                                a.h_out[o] = __bfloat16_as_ushort(hb);
                                a.h_out[o + a.h_plane] = __bfloat16_as_ushort(lb);
                            }
                        }
                    } else {
                        const int m = rt * TILE_ROWS + 32 * q + lane;
                        if (m < a.H) {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                if (c1 + jj < w.nvalid)
                                    a.y_out[(size_t)(pos0 + c1 + jj) * a.H + m] = v[jj];
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

template <bool GU, int WFMT, int NMAX, int S>
cudaError_t launch_cfg(const TcArgs &a, const CUtensorMap &m1, const CUtensorMap &m2, cudaStream_t st)
{
    constexpr int NB = GU ? 1 : 2;
    constexpr int SMEM = Smem<NMAX, NB, S>::TOTAL;
    auto kern = gemm_tc_kernel<GU, WFMT, NMAX, S>;
    static std::atomic<int> attr_set[MAX_DEVICES];
    cudaError_t e = smem_limit_once(attr_set, (const void *)kern, SMEM);
    if (e != cudaSuccess)
        return e;
    kern<<<sm_count(), NUM_THREADS, SMEM, st>>>(a, m1, m2);
    return cudaGetLastError();
}

// token tile sizes: small batches use a small tile (more stages in flight),
// larger batches the full tile.
constexpr int SMALL_T = 64;

template <bool GU>
cudaError_t launch_any(const TcArgs &a, int fmt, int T, const CUtensorMap &m1, const CUtensorMap &m2,
                       cudaStream_t st)
{
    const bool small = T <= SMALL_T;
    if constexpr (GU) {
        if (fmt == FMT_MXFP4)
            return small ? launch_cfg<true, FMT_MXFP4, 64, 4>(a, m1, m2, st)
                         : launch_cfg<true, FMT_MXFP4, 256, 3>(a, m1, m2, st);
        return small ? launch_cfg<true, FMT_BF16, 64, 4>(a, m1, m2, st)
                     : launch_cfg<true, FMT_BF16, 256, 3>(a, m1, m2, st);
    } else {
        if (fmt == FMT_MXFP4)
            return small ? launch_cfg<false, FMT_MXFP4, 64, 4>(a, m1, m2, st)
                         : launch_cfg<false, FMT_MXFP4, 128, 3>(a, m1, m2, st);
        return small ? launch_cfg<false, FMT_BF16, 64, 4>(a, m1, m2, st)
                     : launch_cfg<false, FMT_BF16, 128, 3>(a, m1, m2, st);
    }
}

}  // namespace

// x_perm[p] = x[row_token[p]] for the routed positions p < T*k (16-byte copies).
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

cudaError_t launch_gemm_gate_up_tc(const Plan &p, const WeightStore &w, int fmt, const uint16_t *x, cudaStream_t st)
{
    TcArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.row_tiles, p.grp_start, p.grp_count, p.E, p.G,
             p.I, p.H, p.h, (long long)p.P * p.I, nullptr, p.err};
    a.brows = p.T >= B_BOX_ROWS_BIG && (p.T * p.k == 0 || p.T * p.k >= B_BOX_ROWS_BIG) ? B_BOX_ROWS_BIG
                                                                                       : B_BOX_ROWS_SMALL;
    CUtensorMap m1, m2;
    cudaError_t e = make_map(&m2, x, p.T, p.H, a.brows);
    if (e != cudaSuccess)
        return e;
    if (p.T * p.k > 0) {
        if ((e = make_map(&m1, p.x_perm, (long long)p.T * p.k, p.H, a.brows)) != cudaSuccess)
            return e;
    } else {
        m1 = m2;
    }
    return launch_any<true>(a, fmt, p.T, m1, m2, st);
}

cudaError_t launch_gemm_down_tc(const Plan &p, const WeightStore &w, int fmt, cudaStream_t st)
{
    TcArgs a{w.base, w.group_bytes, w.kchunks, w.chunk_bytes, w.row_tiles, p.grp_start, p.grp_count, p.E, p.G,
             p.I, p.H, nullptr, 0, p.y, p.err};
    a.brows = p.P >= B_BOX_ROWS_BIG ? B_BOX_ROWS_BIG : B_BOX_ROWS_SMALL;
    CUtensorMap m1, m2;
    cudaError_t e = make_map(&m1, p.h, p.P, p.I, a.brows);
    if (e != cudaSuccess)
        return e;
    if ((e = make_map(&m2, p.h + (size_t)p.P * p.I, p.P, p.I, a.brows)) != cudaSuccess)
        return e;
    return launch_any<false>(a, fmt, p.T, m1, m2, st);
}

}  // namespace moe
