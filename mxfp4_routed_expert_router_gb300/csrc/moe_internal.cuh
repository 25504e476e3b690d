// moe_internal.cuh -- internal layout constants, structures and kernel
// launchers of libmoe_gb300.so.  Not part of the public C ABI (include/moe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- weight store
//
// Every weight matrix of every expert group is repacked at load time into
// "chunks": a chunk holds TILE_ROWS weight rows x CHUNK_K contraction
// elements and is contiguous in device memory, so that the GEMM kernels can
// stream a whole chunk with one bulk copy.  Chunks of one row tile are
// consecutive along K; row tiles of one group are consecutive; groups are
// consecutive.
//
// Two chunk layouts are kept (two copies of every matrix; each kernel reads
// only its own, so HBM traffic per call is that of one copy):
//
// TILE layout (tcgen05 kernel), K = 128 split into two halves of 64:
//   MXFP4: [h*4096 + r*32, +32)  half h of row r: two 16-byte blocks of 32
//                                elements, each 4 repacked words (mx_decode.cuh)
//          [8192 + r*4, +4)      E8M0 scales of row r, one per 32 elements
//   BF16:  [h*16384 + r*128, +128)  64 BF16 values of half h of row r
//
// FRAG layout (register-streaming kernel): rows grouped by 16 (group w =
// r / 16), K by 16 (step j = 0..7).  Thread t (g = t / 4, q = t % 4) of the
// warp owning group w needs, per step j, the elements of the warp-level MMA
// A fragment: (row g, k 2q..2q+1), (row g+8, k 2q..2q+1), (row g, k 2q+8..9),
// (row g+8, k 2q+8..9) with k relative to 16j.
//   MXFP4: word ((w*2 + j/4)*32 + t)*4 + j%4 holds those 8 elements in that
//          order (repacked word format, mx_decode.cuh);
//          [8192 + (w*8 + g)*8, +8)  scales: row 16w+g blocks 0..3, then row
//                                    16w+g+8 blocks 0..3
//   BF16:  [((w*8 + j)*32 + t)*16, +16)  the 8 BF16 values in that order
//   INT4 (group-32 INT4, FRAG_F16 only): see FRAG_F16 below
//
// Row order inside a row tile (both layouts): r = 16*w + i.
//   gate|up matrices: feature n = 64*tile + 8*w + (i % 8), of W_g when i < 8
//     and of W_u when i >= 8, so that gate and up of one feature are rows g
//     and g+8 of the same 16-row group.  A tile covers 64 intermediate features.
//   down matrices: tile row r holds output feature 128*tile + r.
// Rows past the logical end, and K past the logical end, are zero codes.
constexpr int TILE_ROWS = 128;
constexpr int CHUNK_K = 128;
constexpr int GU_FEATURES_PER_TILE = 64;
constexpr int CHUNK_MX_CODE_BYTES = TILE_ROWS * CHUNK_K / 2;        // 8192
constexpr int CHUNK_MX_SCALE_BYTES = TILE_ROWS * CHUNK_K / 32;      // 512
constexpr int CHUNK_MX_BYTES = CHUNK_MX_CODE_BYTES + CHUNK_MX_SCALE_BYTES;  // 8704
constexpr int CHUNK_BF16_BYTES = TILE_ROWS * CHUNK_K * 2;           // 32768
constexpr int CHUNK_I4_SCALE_BYTES = TILE_ROWS * CHUNK_K / 32 * 2;  // 1024: FP16 group scales
constexpr int CHUNK_I4_ZERO_BYTES = TILE_ROWS * CHUNK_K / 32;       // 512: zero points
constexpr int CHUNK_I4_BYTES = CHUNK_MX_CODE_BYTES + CHUNK_I4_SCALE_BYTES + CHUNK_I4_ZERO_BYTES;  // 9728
constexpr int HALF_K = CHUNK_K / 2;                                 // K of one pipeline stage

enum ChunkLayout { LAYOUT_TILE = 0, LAYOUT_FRAG = 1, LAYOUT_FRAG_F16 = 2, LAYOUT_TILE_F16 = 3, LAYOUT_TILE_I4 = 4 };

// TILE_I4 layout (tcgen05 kernel, group-32 INT4): the 128-K chunk is four
// 32-value blocks b; row r's 32 codes of block b are 16 bytes at
// [(b*128 + r)*16, +16): word c holds values 8c..8c+7 of the block, the pair
// (8c + 2p, 8c + 2p + 1) in nibbles p and p + 4, so that one shift and one mask
// put a pair into the two halves of a 32-bit word.  The FP16 scale of (block b,
// row r) is at [8192 + (b*128 + r)*2], its zero point at [9216 + b*128 + r]
// (9,728 bytes, as CHUNK_I4_BYTES).  The row base kept beside the chunks is
// b_row + 127 with b_row = floor(log2 max|s|) - 11 over the row's scales, so
// that s * 2^-b_row lies below 2^12 and every weight below 15 * 2^12 in FP16.
constexpr int TILE_I4_BASE_SHIFT = 11;

// TILE_F16 layout (tcgen05 kernel with FP16 operands, MXFP4 only): the 128-K
// chunk is four 32-value blocks b; row r's codes of block b are 16 plain pack4
// bytes (element 2j in the low nibble of byte j) at [(b*128 + r)*16, +16), so
// that 32 lanes holding 32 consecutive rows read 512 contiguous bytes; the
// E8M0 byte of (block b, row r) is at [8192 + b*128 + r].  The largest
// exponent of every row over its whole K (the row base b_row) is kept beside
// the chunks (WeightStore::row_base); a weight decodes to FP16
// v(c) * 2^(e - b_row), exact when the row's exponents span at most
// TILE_F16_MAX_SPREAD.
constexpr int TILE_F16_MAX_SPREAD = 23;

// FRAG_F16 layout (streaming layer with FP16 operands): the same fragment
// order as FRAG, but each word holds the 8 codes as 4 plain OCP E2M1 byte
// pairs (first element in the low nibble) so that the hardware e2m1x2 -> f16x2
// conversion decodes a byte per instruction:
//   byte 0: (row g, k 2q, 2q+1), byte 1: (row g+8, k 2q, 2q+1),
//   byte 2: (row g, k 2q+8, 2q+9), byte 3: (row g+8, k 2q+8, 2q+9).
// The codes decode to FP16 unscaled (exactly: |v| <= 6); the raw E8M0 bytes
// (same positions as in FRAG) scale each 32-wide block's MMA partial sum in
// FP32, where every power of two 2^(e-127), e in [0, 254], is exact.
// Group-32 INT4 weights use the same word positions, with the fragment's
// element pair p (byte p above) in nibbles p (first element) and p + 4
// (second), so that one shift and one mask put a pair in the two halves of a
// word; the codes decode exactly to FP16 q - z, and each block's MMA partial
// sum takes the group's FP16 scale in FP32.  After the codes:
//   [8192 + (w*8 + g)*16, +16)         FP16 scales: row 16w+g blocks 0..3, then
//                                      row 16w+g+8 blocks 0..3
//   [9216 + (w*8 + g)*8, +8)           zero points (bytes), same order
// FP16 token rows (x16 and its gathered copies) store K in a permuted order
// inside every 16-element group so that a lane's two MMA B registers are
// adjacent: physical element 4q + c (q, c in 0..3) holds logical element
// 2q + (c & 1) + 8 * (c >> 1).
__host__ __device__ constexpr int x16_logical_k(int phys) { return 2 * (phys / 4) + (phys & 1) + 8 * ((phys & 3) >> 1); }
__host__ __device__ constexpr int x16_phys_k(int k) { return 4 * ((k & 7) >> 1) + (k & 1) + 2 * (k >> 3); }

// gate|up row order (see above)
__host__ __device__ constexpr int gu_row_feature(int tile, int r) { return tile * 64 + 8 * (r >> 4) + (r & 7); }
__host__ __device__ constexpr bool gu_row_is_up(int r) { return (r & 8) != 0; }

enum WeightFormat { FMT_MXFP4 = 0, FMT_BF16 = 1, FMT_INT4 = 2 };

struct WeightStore {
    uint8_t *base = nullptr;  // device
    int rows = 0;             // logical rows (2I for gate|up, H for down)
    int cols = 0;             // logical K
    int row_tiles = 0;
    int kchunks = 0;
    int chunk_bytes = 0;
    size_t group_bytes = 0;   // bytes of one expert group's matrix
    uint8_t *row_base = nullptr;  // TILE_F16: largest E8M0 exponent of each row, [G][row_tiles * 128] (device)
};

// A caller-side source matrix for the repack: row r starts at
// codes + r * code_stride (bytes); its scales are elements
// r * scale_stride .. of `scales` (bytes for MXFP4, FP16 for INT4) and its
// INT4 zero points bytes r * scale_stride .. of `zeros` (NULL: all 8).
struct SrcMat {
    const uint8_t *codes;
    const uint8_t *scales;
    long long code_stride;
    long long scale_stride;
    const uint8_t *zeros;
};

// ---------------------------------------------------------------- forward plan
//
// Expert groups g in [0, G): g < E routed, g >= E shared (a dense layer is
// E = 0 routed and G = n_slices shared groups).  Rows of h and y ("positions")
// are ordered: routed positions 0..T*k-1 in expert-major sorted order, then
// shared group s at T*k + s*T + t.
struct Plan {
    int T, k, E, S, G, H, I;
    int P;                    // T*k + S*T positions
    int ebase, etotal;        // caller routing: the routed groups are expert ids [ebase, ebase + E) of etotal
    // workspace arrays
    int *topk_ids;            // [T*k]
    float *topk_w;            // [T*k]
    int *counts;              // [max(E,1)]
    int *chunk_cnt;           // [ceil(T*k/1024)][E+1] per-chunk expert (and empty-slot) counts of the permutation (NULL: the
                              // one-CTA-per-expert permutation kernel, which needs no such scratch)
    int *expert_offsets;      // [E+1]
    int *sorted_slot;         // [T*k]
    int *slot_pos;            // [T*k]
    int *grp_start;           // [G]
    int *grp_count;           // [G]
    int *row_token;           // [P] token index of each position
    uint16_t *x_perm;         // [T*k][H] rows of x gathered in routed position order (BF16, or FP16 for
                              // the FP16 streaming path)
    uint16_t *x16;            // [T][H] token rows of the streaming path in x16 K order: FP16
                              // x_t * 2^-xs[t] for MXFP4 and INT4 weights, BF16 x_t for BF16 weights;
                              // on the tcgen05 FP16 path FP16 x_t * 2^-xs[t] in natural K order
    int *xs;                  // [T] per-token power-of-two scale exponent of x16
    int *xsp;                 // [P] tcgen05 FP16 path: xs of each position's token
    uint16_t *h;              // [2][P][I] h = hi plane + lo plane: BF16 (lo = bf16(h - hi)); on the FP16
                              // streaming path the first plane only, FP16 h * 2^-hs; x16 K order on the
                              // streaming path.
    uint16_t *h16;            // [P][I] tcgen05 FP16 path: FP16 h * 2^-hsp[p]
    int *hsp;                 // [P] tcgen05 FP16 path: power of two of each position's h16 row
    int *hs;                  // [P][hs_pitch] FP16 streaming path: power-of-two scale of each position's
                              // 64-feature block of h
    int hs_pitch;             // ceil(I/64) rounded up to a multiple of 4 (16-byte rows)
    float *y;                 // [P][H] FP32; the tcgen05 FP16 path keeps FP16 y * 2^-ys[p] here instead
    int *ys;                  // [P] tcgen05 FP16 path: power of two of each position's FP16 y row
    int *sync;                // streaming path: grid-wide counters, zeroed before each launch
    int *err;                 // device-visible error flag (mapped host memory)
};

// error codes written into *err by kernels (first error wins)
enum DeviceError {
    DEV_ERR_NONE = 0,
    DEV_ERR_PERMUTE_COUNT = 1,
    DEV_ERR_BOUNDS = 2,
    DEV_ERR_WAIT_TIMEOUT = 3,
};

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.

cudaError_t launch_repack(int fmt, int layout, bool gate_up, const SrcMat &gate, const SrcMat &up,
                          const WeightStore &ws, int group, int I, int H, int *bad_scale, cudaStream_t st);

cudaError_t launch_router(const float *logits, int T, int E, int k, int *ids, float *w, int *counts, int n_counts,
                          cudaStream_t st);

// caller-given routing (ids, weights) copied into the call's routing arrays;
// an id outside [0, E) records DEV_ERR_BOUNDS and becomes expert 0, weight 0;
// counts[0 .. n_counts) are cleared for the histogram
cudaError_t launch_routing_copy(const int *ids_in, const float *w_in, int n, int E, int ebase, int etotal, int *ids,
                                float *w, int *counts,
                                int n_counts, int *err, cudaStream_t st);

// sigmoid scores, bias-adjusted top-k, weights normalised over the selection
// times scale (bias may be NULL)
cudaError_t launch_router_sigmoid(const float *logits, const float *bias, int T, int E, int k, float scale, int *ids,
                                  float *w, cudaStream_t st);

cudaError_t launch_permute(const Plan &p, cudaStream_t st);

cudaError_t launch_dense_plan(const Plan &p, cudaStream_t st);

cudaError_t launch_combine(const Plan &p, float *out, int accumulate, cudaStream_t st);
// the same over the FP16 rows y16 * 2^ys[p] of the tcgen05 FP16 path (in p.y)
cudaError_t launch_combine_f16(const Plan &p, float *out, int accumulate, cudaStream_t st);

// x_perm[p] = x[row_token[p]] for the routed positions (BF16 operands)
cudaError_t launch_gather_rows(const Plan &p, const uint16_t *x, cudaStream_t st);

// row bases of a TILE_F16 store for one group: for every tile row, the
// largest E8M0 exponent over the row's K; a row whose exponents span more than
// TILE_F16_MAX_SPREAD sets *wide.  With fmt FMT_INT4, the TILE_I4 row base
// (see above; wide is not used)
cudaError_t launch_row_base(int fmt, bool gate_up, const SrcMat &gate, const SrcMat &up, const WeightStore &ws,
                            int group, int I, int H, int *wide, cudaStream_t st);

// For the h scales of the tcgen05 path with FP16 operands: out[group] = an
// order-preserving integer key of max_n log2(|w_g,n| |w_u,n|) over the
// features n of one group (Euclidean norms of the decoded gate and up rows of
// an MXFP4 matrix, rounded up; unsigned order of the key bits); out[group]
// must start at 0
cudaError_t launch_gu_norm(int fmt, const SrcMat &gate, const SrcMat &up, int group, int I, int H, int *out,
                           cudaStream_t st);
// the same for the rows of a down matrix (H rows of I values): a key of
// max_m log2 |w_d,m|.  fmt: FMT_MXFP4 or FMT_INT4 (group-32 INT4 sources)
cudaError_t launch_dn_norm(int fmt, const SrcMat &dn, int group, int I, int H, int *out, cudaStream_t st);

// tcgen05 path with FP16 operands (after the permutation): FP16 token rows x16,
// their copies in routed position order (x_perm), the powers of two xs / xsp,
// and the per-position h scales hsp from gu_norm_key (one key per group)
cudaError_t launch_token_prep_f16(const Plan &p, const uint16_t *x, const int *gu_norm_key, const int *dn_norm_key,
                                  cudaStream_t st);

// f16: FP16 operands (TILE_F16 MXFP4 store, token rows x_rows = x16 and the
// gathered FP16 rows in x_perm); otherwise BF16 operands (x_rows = the caller's x)
cudaError_t launch_gemm_gate_up_tc(const Plan &p, const WeightStore &w, int fmt, bool f16, const uint16_t *x_rows,
                                   cudaStream_t st);

cudaError_t launch_gemm_down_tc(const Plan &p, const WeightStore &w, int fmt, bool f16, cudaStream_t st);

// The whole layer in one persistent kernel for decode-sized batches
// (layer_stream.cu): token tiles of at most STREAM_MAX_T tokens; larger
// groups are split into several items.
constexpr int STREAM_MAX_T = 64;
constexpr int LS_MAX_EXPERTS = 512;
constexpr int LS_MAX_SLOTS = 4096;  // T * k

// bytes of the grid-wide counters the streaming layer needs (Plan::sync)
size_t layer_stream_sync_bytes(int G);

// true when the streaming layer kernel can run this plan (sizes within its
// shared-memory and scheduling limits)
bool layer_stream_fits(const Plan &p, int fmt);

// zeroes p.sync, then launches the layer kernel cooperatively (one CTA per SM).
// expire_wait_us > 0 (tests of the device-side wait limit only): the kernel's
// grid-wide completion wait before the combine gets a target no launch reaches
// and a limit of that many microseconds, so it expires, records
// DEV_ERR_WAIT_TIMEOUT and the kernel leaves without combining.
cudaError_t launch_layer_stream(const Plan &p, const WeightStore &gu, const WeightStore &dn, int fmt,
                                const uint16_t *x, const float *logits, const int *ids_in, const float *w_in,
                                float *out, int accumulate, cudaStream_t st, int expire_wait_us = 0);

// Record msg as the calling thread's moe_last_error() text; returns status.
int set_last_error(int status, const char *msg);

}  // namespace moe
