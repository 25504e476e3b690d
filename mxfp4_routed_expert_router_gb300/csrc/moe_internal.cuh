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
// MXFP4 chunk (CHUNK_MX_BYTES), K = 128 elements split into two halves of 64:
//   [h*4096 + r*32, +32)  half h (h = 0, 1) of row r: two 16-byte blocks of 32
//                         elements, each block 4 repacked words (mx_decode.cuh)
//   [8192 + r*4, +4)      E8M0 scales of row r, one per 32 elements
// BF16 chunk (CHUNK_BF16_BYTES): [h*16384 + r*128, +128) = 64 BF16 values of
//   half h of row r.
//
// Row order inside a row tile:
//   gate|up matrices: tile row r = 32*q + l (q = r / 32, l = r % 32) holds
//     feature n = 64*tile + 16*q + (l % 16) of W_g when l < 16 and of W_u
//     when l >= 16, so that gate and up of one feature sit 16 lanes apart in
//     the same warp of the epilogue.  A tile covers 64 intermediate features.
//   down matrices: tile row r holds output feature 128*tile + r.
// Rows past the logical end, and K past the logical end, are zero codes.
constexpr int TILE_ROWS = 128;
constexpr int CHUNK_K = 128;
constexpr int GU_FEATURES_PER_TILE = 64;
constexpr int CHUNK_MX_CODE_BYTES = TILE_ROWS * CHUNK_K / 2;        // 8192
constexpr int CHUNK_MX_SCALE_BYTES = TILE_ROWS * CHUNK_K / 32;      // 512
constexpr int CHUNK_MX_BYTES = CHUNK_MX_CODE_BYTES + CHUNK_MX_SCALE_BYTES;  // 8704
constexpr int CHUNK_BF16_BYTES = TILE_ROWS * CHUNK_K * 2;           // 32768
constexpr int HALF_K = CHUNK_K / 2;                                 // K of one pipeline stage

enum WeightFormat { FMT_MXFP4 = 0, FMT_BF16 = 1 };

struct WeightStore {
    uint8_t *base = nullptr;  // device
    int rows = 0;             // logical rows (2I for gate|up, H for down)
    int cols = 0;             // logical K
    int row_tiles = 0;
    int kchunks = 0;
    int chunk_bytes = 0;
    size_t group_bytes = 0;   // bytes of one expert group's matrix
};

// A caller-side source matrix for the repack: row r starts at
// codes + r * code_stride (bytes), its scales at scales + r * scale_stride.
struct SrcMat {
    const uint8_t *codes;
    const uint8_t *scales;
    long long code_stride;
    long long scale_stride;
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
    // workspace arrays
    int *topk_ids;            // [T*k]
    float *topk_w;            // [T*k]
    int *counts;              // [max(E,1)]
    int *expert_offsets;      // [E+1]
    int *sorted_slot;         // [T*k]
    int *slot_pos;            // [T*k]
    int *grp_start;           // [G]
    int *grp_count;           // [G]
    int *row_token;           // [P] token index of each position
    uint16_t *x_perm;         // [T*k][H] BF16 rows of x gathered in routed position order
    uint16_t *h;              // [2][P][I] BF16: h = hi plane + lo plane (lo = bf16(h - hi))
    float *y;                 // [P][H] FP32
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

cudaError_t launch_repack(int fmt, bool gate_up, const SrcMat &gate, const SrcMat &up, const WeightStore &ws,
                          int group, int I, int H, int *bad_scale, cudaStream_t st);

cudaError_t launch_router(const float *logits, int T, int E, int k, int *ids, float *w, int *counts, int n_counts,
                          cudaStream_t st);

cudaError_t launch_permute(const Plan &p, cudaStream_t st);

cudaError_t launch_dense_plan(const Plan &p, cudaStream_t st);

cudaError_t launch_gemm_gate_up(const Plan &p, const WeightStore &w, int fmt, const uint16_t *x, cudaStream_t st);

cudaError_t launch_gemm_down(const Plan &p, const WeightStore &w, int fmt, cudaStream_t st);

cudaError_t launch_combine(const Plan &p, float *out, int accumulate, cudaStream_t st);

cudaError_t launch_gather_rows(const Plan &p, const uint16_t *x, cudaStream_t st);

cudaError_t launch_gemm_gate_up_tc(const Plan &p, const WeightStore &w, int fmt, const uint16_t *x, cudaStream_t st);

cudaError_t launch_gemm_down_tc(const Plan &p, const WeightStore &w, int fmt, cudaStream_t st);

}  // namespace moe
