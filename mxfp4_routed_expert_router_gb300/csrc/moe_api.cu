// moe_api.cu -- the C ABI of libmoe_gb300.so (declared in include/moe.h):
// argument checks, the library's weight copy, workspace layout and the launch
// sequence of one forward pass.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/moe.h"
#include "moe_internal.cuh"

using namespace moe;

struct MoeHandle {
    MoeConfig cfg;
    int E = 0, S = 0, G = 0;   // routed groups, shared groups (a dense layer: E = 0, S = n_slices)
    int H = 0, I = 0;          // hidden, per-group intermediate
    int fmt = 0;
    int k_max = 0;
    int ebase = 0, etotal = 0;  // the experts held are ids [ebase, ebase + E) of etotal (moe_set_expert_range)
    int device = 0;
    WeightStore gu, dn;        // TILE or TILE_F16 layout (tensor-memory GEMMs, large batches)
    bool tc_f16 = false;       // the tensor-memory GEMMs run FP16 operands (TILE_F16 store with row bases)
    int *gu_norm_key = nullptr;  // FP16 operands: per group, key of max_n log2(|w_g,n| |w_u,n|) (device)
    int *dn_norm_key = nullptr;  // FP16 operands: per group, key of max_m log2 |w_d,m| (device)
    WeightStore gu_f, dn_f;    // FRAG layout (register-streaming GEMMs, decode-sized batches)
    int *err_host = nullptr;   // mapped pinned host memory, written by kernels on device-side errors
    int *err_dev = nullptr;    // device alias of err_host
    int expire_wait_us = 0;    // moe_debug_expire_next_wait: armed for the next single-kernel launch
    bool profile = false;      // record stage events (moe_profile_enable)
    bool profiled = false;     // a call has recorded its events
    cudaEvent_t ev[7] = {};
};

constexpr int N_STAGES = 6;

namespace {

thread_local char g_msg[512] = "no error";

MoeStatus fail(MoeStatus s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

MoeStatus cuda_fail(cudaError_t e, const char *what)
{
    return fail(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void init_store(WeightStore &w, int rows_per_group_tiles_basis, bool gate_up, int K, int fmt)
{
    // gate|up: a row tile covers 64 intermediate features (128 rows); down: 128 output features.
    w.rows = rows_per_group_tiles_basis;
    w.cols = K;
    w.row_tiles = gate_up ? (rows_per_group_tiles_basis + GU_FEATURES_PER_TILE - 1) / GU_FEATURES_PER_TILE
                          : (rows_per_group_tiles_basis + TILE_ROWS - 1) / TILE_ROWS;
    w.kchunks = (K + CHUNK_K - 1) / CHUNK_K;
    w.chunk_bytes = fmt == FMT_MXFP4 ? CHUNK_MX_BYTES : fmt == FMT_INT4 ? CHUNK_I4_BYTES : CHUNK_BF16_BYTES;
    w.group_bytes = (size_t)w.row_tiles * w.kchunks * w.chunk_bytes;
}

// Workspace carve-up for T tokens and top-k (see Plan in moe_internal.cuh).
size_t plan_layout(const MoeHandle *h, int T, int k, char *base, Plan *p)
{
    const int E = h->E, S = h->S, G = h->G, H = h->H, I = h->I;
    const long long n = (long long)T * k;
    const long long P = n + (long long)S * T;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *ptr = base ? base + off : nullptr;
        off = align_up(off + bytes, 256);
        return ptr;
    };
    Plan q{};
    q.T = T;
    q.k = k;
    q.E = E;
    q.S = S;
    q.G = G;
    q.H = H;
    q.I = I;
    q.P = (int)P;
    q.ebase = h->ebase;
    q.etotal = h->etotal;
    q.topk_ids = (int *)take(sizeof(int) * (n > 0 ? n : 1));
    q.topk_w = (float *)take(sizeof(float) * (n > 0 ? n : 1));
    q.counts = (int *)take(sizeof(int) * (E > 0 ? E : 1));
    q.chunk_cnt = (int *)take(sizeof(int) * (size_t)((n + 1023) / 1024 + 1) * (E + 1));
    q.expert_offsets = (int *)take(sizeof(int) * (E + 1));
    q.sorted_slot = (int *)take(sizeof(int) * (n > 0 ? n : 1));
    q.slot_pos = (int *)take(sizeof(int) * (n > 0 ? n : 1));
    q.grp_start = (int *)take(sizeof(int) * G);
    q.grp_count = (int *)take(sizeof(int) * G);
    q.row_token = (int *)take(sizeof(int) * P);
    q.x_perm = (uint16_t *)take(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * H);
    q.x16 = (uint16_t *)take(sizeof(uint16_t) * (size_t)T * H);
    q.xs = (int *)take(sizeof(int) * (size_t)T);
    q.hs_pitch = ((I + 63) / 64 + 3) & ~3;
    q.hs = (int *)take(sizeof(int) * (size_t)P * q.hs_pitch);
    q.h = (uint16_t *)take(2 * sizeof(uint16_t) * (size_t)P * I);
    q.h16 = (uint16_t *)take(sizeof(uint16_t) * (size_t)P * I);
    q.hsp = (int *)take(sizeof(int) * (size_t)P);
    q.xsp = (int *)take(sizeof(int) * (size_t)P);
    q.y = (float *)take(sizeof(float) * (size_t)P * H);
    q.ys = (int *)take(sizeof(int) * (size_t)P);
    q.sync = (int *)take(layer_stream_sync_bytes(G));
    q.err = h->err_dev;
    if (p)
        *p = q;
    return off;
}

MoeStatus check_pending(const MoeHandle *h)
{
    int e = *(volatile int *)h->err_host;
    if (e != DEV_ERR_NONE)
        return fail(MOE_EDEVICE, "a kernel of an earlier call reported device error %d", e);
    return MOE_OK;
}

// One forward call.  Routing comes from the logits (softmax top-k), or, when
// ids_in is given, from the caller's ids and weights.
MoeStatus run_layer(MoeHandle *h, const void *x, const float *logits, const int *ids_in, const float *w_in, int T,
                    int k, float *out, int accumulate, void *ws, size_t ws_bytes, const MoeRoutingOut *routing,
                    cudaStream_t st)
{
    Plan p;
    size_t need = plan_layout(h, T, k, (char *)ws, &p);
    if (ws_bytes < need)
        return fail(MOE_EWORKSPACE, "workspace has %zu bytes, this call needs %zu", ws_bytes, need);
    if (routing) {
        if (routing->topk_ids) p.topk_ids = routing->topk_ids;
        if (routing->topk_w) p.topk_w = routing->topk_w;
        if (routing->expert_offsets) p.expert_offsets = routing->expert_offsets;
        if (routing->sorted_slot) p.sorted_slot = routing->sorted_slot;
        if (routing->slot_pos) p.slot_pos = routing->slot_pos;
    }
    cudaError_t e;
    auto mark = [&](int i) {
        if (h->profile)
            cudaEventRecord(h->ev[i], st);
    };
    // Decode-sized batches (few tokens per expert) run the whole layer in one
    // persistent weight-streaming kernel; larger batches use the tensor-memory
    // GEMMs between the routing, permutation and combine kernels.
    const bool stream = h->E > 0 ? (long long)T * k <= 16LL * h->E : T <= STREAM_MAX_T;
    if (stream && layer_stream_fits(p, h->fmt)) {
        for (int i = 0; i <= 5; ++i)
            mark(i);
        const int expire = h->expire_wait_us;
        h->expire_wait_us = 0;
        if ((e = launch_layer_stream(p, h->gu_f, h->dn_f, h->fmt, (const uint16_t *)x, logits, ids_in, w_in, out,
                                     accumulate, st, expire)) != cudaSuccess)
            return cuda_fail(e, "layer launch");
        mark(6);
        if (h->profile)
            h->profiled = true;
        return MOE_OK;
    }
    mark(0);
    if (h->E > 0) {
        if (ids_in) {
            if ((e = launch_routing_copy(ids_in, w_in, T * k, h->E, h->ebase, h->etotal, p.topk_ids, p.topk_w,
                                         p.counts, h->E, p.err, st)) != cudaSuccess)
                return cuda_fail(e, "routing copy launch");
        } else if ((e = launch_router(logits, T, h->E, k, p.topk_ids, p.topk_w, p.counts, h->E, st)) !=
                   cudaSuccess) {
            return cuda_fail(e, "router launch");
        }
        mark(1);
        if ((e = launch_permute(p, st)) != cudaSuccess)
            return cuda_fail(e, "permute launch");
    } else {
        mark(1);
        if ((e = launch_dense_plan(p, st)) != cudaSuccess)
            return cuda_fail(e, "dense plan launch");
    }
    const uint16_t *xb = (const uint16_t *)x;
    if (h->tc_f16) {
        // FP16 operands: FP16 token rows with a power of two per token, written
        // in token and in position order by one pass, with the power of two of
        // each position's h (from a bound on |h|); gate|up writes one FP16 plane
        // of h, which down reads
        if ((e = launch_token_prep_f16(p, xb, h->gu_norm_key, h->dn_norm_key, st)) != cudaSuccess)
            return cuda_fail(e, "token prep launch");
        mark(2);
        if ((e = launch_gemm_gate_up_tc(p, h->gu, h->fmt, true, p.x16, st)) != cudaSuccess)
            return cuda_fail(e, "gate/up launch");
        mark(3);
        if ((e = launch_gemm_down_tc(p, h->dn, h->fmt, true, st)) != cudaSuccess)
            return cuda_fail(e, "down launch");
    } else {
        if ((e = launch_gather_rows(p, xb, st)) != cudaSuccess)
            return cuda_fail(e, "gather launch");
        mark(2);
        if ((e = launch_gemm_gate_up_tc(p, h->gu, h->fmt, false, xb, st)) != cudaSuccess)
            return cuda_fail(e, "gate/up launch");
        mark(3);
        if ((e = launch_gemm_down_tc(p, h->dn, h->fmt, false, st)) != cudaSuccess)
            return cuda_fail(e, "down launch");
    }
    mark(4);
    if ((e = h->tc_f16 ? launch_combine_f16(p, out, accumulate, st) : launch_combine(p, out, accumulate, st)) !=
        cudaSuccess)
        return cuda_fail(e, "combine launch");
    mark(5);
    mark(6);
    if (h->profile)
        h->profiled = true;
    return MOE_OK;
}

void destroy(MoeHandle *h)
{
    if (!h)
        return;
    if (h->gu.base)
        cudaFree(h->gu.base);
    if (h->dn.base)
        cudaFree(h->dn.base);
    if (h->gu_norm_key)
        cudaFree(h->gu_norm_key);
    if (h->dn_norm_key)
        cudaFree(h->dn_norm_key);
    if (h->gu.row_base)
        cudaFree(h->gu.row_base);
    if (h->dn.row_base)
        cudaFree(h->dn.row_base);
    if (h->gu_f.base)
        cudaFree(h->gu_f.base);
    if (h->dn_f.base)
        cudaFree(h->dn_f.base);
    if (h->err_host)
        cudaFreeHost(h->err_host);
    for (cudaEvent_t &ev : h->ev)
        if (ev)
            cudaEventDestroy(ev);
    delete h;
}

}  // namespace

// Lets entry points defined in other files report through moe_last_error().
int moe::set_last_error(int status, const char *msg)
{
    return (int)fail((MoeStatus)status, "%s", msg);
}

extern "C" {

MoeStatus moe_load_weights(const MoeConfig *cfg, const MoeMx *gate_up, const MoeMx *down, void *cuda_stream,
                           MoeHandle **out)
{
    if (!cfg || !gate_up || !down || !out)
        return fail(MOE_EINVAL, "moe_load_weights: NULL argument");
    const MoeConfig c = *cfg;
    if (c.fmt != MOE_W_MXFP4 && c.fmt != MOE_W_BF16 && c.fmt != MOE_W_INT4G32)
        return fail(MOE_EINVAL, "unknown weight format %d", (int)c.fmt);
    if (c.hidden <= 0 || c.inter <= 0 || c.hidden % 32 || c.inter % 32 || c.hidden > 65536 || c.inter > 262144)
        return fail(MOE_EDIMS, "hidden (%d) and inter (%d) must be positive multiples of 32 (hidden <= 65536)",
                    c.hidden, c.inter);
    const bool dense = c.n_slices > 0;
    int E, S, I, G, k_max;
    if (dense) {
        if (c.n_experts != c.n_slices || c.n_shared != 0)
            return fail(MOE_EINVAL, "dense layer: n_experts must equal n_slices and n_shared must be 0");
        if (c.n_slices > 1024 || c.inter % c.n_slices || (c.inter / c.n_slices) % 32)
            return fail(MOE_EDIMS, "dense layer: inter %d cannot be cut into %d slices of a multiple of 32",
                        c.inter, c.n_slices);
        E = 0;
        S = c.n_slices;
        I = c.inter / c.n_slices;
        k_max = 0;
    } else {
        if (c.n_slices < 0)
            return fail(MOE_EINVAL, "n_slices must be >= 0");
        if (c.n_experts < 1 || c.n_experts > 1024 || c.n_shared < 0 || c.n_shared > 64)
            return fail(MOE_EINVAL, "n_experts must be in [1, 1024] and n_shared in [0, 64]");
        if (c.k_max < 1 || c.k_max > 32)
            return fail(MOE_EINVAL, "k_max must be in [1, 32]");
        E = c.n_experts;
        S = c.n_shared;
        I = c.inter;
        k_max = c.k_max;
    }
    G = E + S;
    const int fmt = c.fmt == MOE_W_MXFP4 ? FMT_MXFP4 : c.fmt == MOE_W_INT4G32 ? FMT_INT4 : FMT_BF16;
    const bool nib = fmt != FMT_BF16;               // 4-bit codes
    const long long ssz = fmt == FMT_INT4 ? 2 : 1;  // bytes per scale
    const int n_gu = dense ? 2 : G, n_dn = dense ? 1 : G;
    for (int i = 0; i < n_gu; ++i)
        if (!gate_up[i].codes || (nib && !gate_up[i].scales))
            return fail(MOE_EINVAL, "gate_up[%d] has a NULL pointer", i);
    for (int i = 0; i < n_dn; ++i)
        if (!down[i].codes || (nib && !down[i].scales))
            return fail(MOE_EINVAL, "down[%d] has a NULL pointer", i);
    if (fmt == FMT_INT4) {
        for (int i = 0; i < n_gu; ++i)
            if (!aligned(gate_up[i].scales, 2))
                return fail(MOE_EINVAL, "gate_up[%d].scales (FP16) is not 2-byte aligned", i);
        for (int i = 0; i < n_dn; ++i)
            if (!aligned(down[i].scales, 2))
                return fail(MOE_EINVAL, "down[%d].scales (FP16) is not 2-byte aligned", i);
    }

    MoeHandle *h = new (std::nothrow) MoeHandle();
    if (!h)
        return fail(MOE_ENOMEM, "host allocation failed");
    h->cfg = c;
    h->E = E;
    h->S = S;
    h->G = G;
    h->H = c.hidden;
    h->I = I;
    h->fmt = fmt;
    h->k_max = k_max;
    h->ebase = 0;
    h->etotal = E;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        destroy(h);
        return cuda_fail(e, "cudaGetDevice");
    }
    init_store(h->gu, I, true, c.hidden, fmt);
    init_store(h->dn, c.hidden, false, I, fmt);
    h->gu_f = h->gu;
    h->dn_f = h->dn;
    const int f_layout = nib ? LAYOUT_FRAG_F16 : LAYOUT_FRAG;
    // [0] device error flag, [1] a rejected scale at load, [2] an MXFP4 row whose
    // exponents span too widely for FP16 operands
    if ((e = cudaHostAlloc((void **)&h->err_host, 4 * sizeof(int), cudaHostAllocMapped)) != cudaSuccess) {
        destroy(h);
        return cuda_fail(e, "cudaHostAlloc");
    }
    for (int i = 0; i < 4; ++i)
        h->err_host[i] = 0;
    if ((e = cudaHostGetDevicePointer((void **)&h->err_dev, h->err_host, 0)) != cudaSuccess) {
        destroy(h);
        return cuda_fail(e, "cudaHostGetDevicePointer");
    }
    // two copies of every weight: a TILE-family one for the tensor-memory GEMMs and
    // a FRAG one for the single-kernel layer
    if (cudaMalloc(&h->gu.base, h->gu.group_bytes * G) != cudaSuccess ||
        cudaMalloc(&h->dn.base, h->dn.group_bytes * G) != cudaSuccess ||
        cudaMalloc(&h->gu_f.base, h->gu_f.group_bytes * G) != cudaSuccess ||
        cudaMalloc(&h->dn_f.base, h->dn_f.group_bytes * G) != cudaSuccess) {
        cudaGetLastError();
        destroy(h);
        return fail(MOE_ENOMEM, "device allocation of %zu bytes of weights failed",
                    2 * (h->gu.group_bytes + h->dn.group_bytes) * (size_t)G);
    }
    int *bad_scale = &h->err_dev[1];
    // scale (and INT4 zero point) arrays advanced by a number of elements; NULL
    // (BF16 scales, absent zero points) stays NULL
    auto sc_at = [&](const void *p, long long elems) -> const uint8_t * {
        return nib && p ? (const uint8_t *)p + elems * ssz : nullptr;
    };
    auto zp_at = [&](const void *p, long long elems) -> const uint8_t * {
        return fmt == FMT_INT4 && p ? (const uint8_t *)p + elems : nullptr;
    };
    // source matrices of group g: gate and up rows of gate|up, and down
    auto sources = [&](int g, SrcMat &gate, SrcMat &up, SrcMat &dn) {
        const long long gs = nib ? c.hidden / 2 : (long long)c.hidden * 2;  // code bytes of a gate|up row
        const long long ss = c.hidden / 32;                                  // scales of a gate|up row
        if (dense) {
            // slice g: gate/up rows [g*I, (g+1)*I) of the unsliced W_g / W_u; down columns likewise
            const long long r0 = (long long)g * I;
            gate = {(const uint8_t *)gate_up[0].codes + r0 * gs, sc_at(gate_up[0].scales, r0 * ss), gs, ss,
                    zp_at(gate_up[0].zeros, r0 * ss)};
            up = {(const uint8_t *)gate_up[1].codes + r0 * gs, sc_at(gate_up[1].scales, r0 * ss), gs, ss,
                  zp_at(gate_up[1].zeros, r0 * ss)};
            const long long dstride = nib ? c.inter / 2 : (long long)c.inter * 2;
            const long long dss = c.inter / 32;
            const long long col_off = nib ? (long long)g * I / 2 : (long long)g * I * 2;
            dn = {(const uint8_t *)down[0].codes + col_off, sc_at(down[0].scales, (long long)g * I / 32), dstride,
                  dss, zp_at(down[0].zeros, (long long)g * I / 32)};
        } else {
            gate = {(const uint8_t *)gate_up[g].codes, sc_at(gate_up[g].scales, 0), gs, ss,
                    zp_at(gate_up[g].zeros, 0)};
            up = {(const uint8_t *)gate_up[g].codes + (long long)I * gs, sc_at(gate_up[g].scales, (long long)I * ss),
                  gs, ss, zp_at(gate_up[g].zeros, (long long)I * ss)};
            const long long dstride = nib ? I / 2 : (long long)I * 2;
            dn = {(const uint8_t *)down[g].codes, sc_at(down[g].scales, 0), dstride, I / 32,
                  zp_at(down[g].zeros, 0)};
        }
    };
    // MXFP4 on the tensor-memory GEMMs: FP16 operands when every row's block
    // exponents span at most TILE_F16_MAX_SPREAD (checked on the device, one
    // pass over the scales), else BF16 operands.  Group-32 INT4: FP16 hi + lo
    // operands against a per-row base (TILE_I4), always.
    int tile_layout = LAYOUT_TILE;
    if (fmt == FMT_MXFP4 || fmt == FMT_INT4) {
        const size_t gu_rb = (size_t)h->gu.row_tiles * TILE_ROWS * G, dn_rb = (size_t)h->dn.row_tiles * TILE_ROWS * G;
        if (cudaMalloc(&h->gu.row_base, gu_rb) != cudaSuccess || cudaMalloc(&h->dn.row_base, dn_rb) != cudaSuccess ||
            cudaMalloc(&h->gu_norm_key, sizeof(int) * (size_t)G) != cudaSuccess ||
            cudaMalloc(&h->dn_norm_key, sizeof(int) * (size_t)G) != cudaSuccess) {
            cudaGetLastError();
            destroy(h);
            return fail(MOE_ENOMEM, "device allocation of %zu bytes of row bases failed", gu_rb + dn_rb);
        }
        if ((e = cudaMemsetAsync(h->gu_norm_key, 0, sizeof(int) * (size_t)G, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(h->dn_norm_key, 0, sizeof(int) * (size_t)G, st)) != cudaSuccess) {
            destroy(h);
            return cuda_fail(e, "norm key clear");
        }
        int *wide = &h->err_dev[2];
        for (int g = 0; g < G; ++g) {
            SrcMat gate{}, up{}, dn{};
            sources(g, gate, up, dn);
            if ((e = launch_row_base(fmt, true, gate, up, h->gu, g, I, c.hidden, wide, st)) != cudaSuccess ||
                (e = launch_row_base(fmt, false, dn, dn, h->dn, g, I, c.hidden, wide, st)) != cudaSuccess ||
                (e = launch_gu_norm(fmt, gate, up, g, I, c.hidden, h->gu_norm_key, st)) != cudaSuccess ||
                (e = launch_dn_norm(fmt, dn, g, I, c.hidden, h->dn_norm_key, st)) != cudaSuccess) {
                destroy(h);
                return cuda_fail(e, "row base launch");
            }
        }
        if ((e = cudaStreamSynchronize(st)) != cudaSuccess) {
            destroy(h);
            return cuda_fail(e, "row bases");
        }
        if (fmt == FMT_INT4) {
            tile_layout = LAYOUT_TILE_I4;
            h->tc_f16 = true;
        } else if (*(volatile int *)wide == 0) {
            tile_layout = LAYOUT_TILE_F16;
            h->tc_f16 = true;
        } else {
            cudaFree(h->gu.row_base);
            cudaFree(h->dn.row_base);
            cudaFree(h->gu_norm_key);
            cudaFree(h->dn_norm_key);
            h->gu.row_base = h->dn.row_base = nullptr;
            h->gu_norm_key = h->dn_norm_key = nullptr;
        }
    }
    for (int g = 0; g < G; ++g) {
        SrcMat gate{}, up{}, dn{};
        sources(g, gate, up, dn);
        if ((e = launch_repack(fmt, tile_layout, true, gate, up, h->gu, g, I, c.hidden, bad_scale, st)) !=
                cudaSuccess ||
            (e = launch_repack(fmt, tile_layout, false, dn, dn, h->dn, g, I, c.hidden, bad_scale, st)) !=
                cudaSuccess ||
            (e = launch_repack(fmt, f_layout, true, gate, up, h->gu_f, g, I, c.hidden, bad_scale, st)) !=
                cudaSuccess ||
            (e = launch_repack(fmt, f_layout, false, dn, dn, h->dn_f, g, I, c.hidden, bad_scale, st)) !=
                cudaSuccess) {
            destroy(h);
            return cuda_fail(e, "repack launch");
        }
    }
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) {
        destroy(h);
        return cuda_fail(e, "repack");
    }
    if (*(volatile int *)bad_scale) {
        destroy(h);
        return fail(MOE_ESCALE, fmt == FMT_INT4 ? "an INT4 FP16 scale is Inf or NaN, or a zero point is above 15"
                                                : "an E8M0 scale byte is 255 (NaN)");
    }
    *out = h;
    return MOE_OK;
}

size_t moe_workspace_bytes(const MoeHandle *h, int T, int k)
{
    if (!h || T <= 0 || k < 0)
        return 0;
    return plan_layout(h, T, h->E > 0 ? k : 0, nullptr, nullptr);
}

MoeStatus moe_forward(MoeHandle *h, const void *x_bf16, const float *router_logits, int T, int k, float *out_fp32,
                      int accumulate, void *workspace, size_t ws_bytes, const MoeRoutingOut *routing,
                      void *cuda_stream)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_forward: NULL handle");
    if (h->E == 0)
        return fail(MOE_EINVAL, "moe_forward on a dense handle; use moe_dense_sliced_forward");
    if (T < 0 || T > (1 << 24))
        return fail(MOE_EINVAL, "T = %d out of range [0, 2^24]", T);
    if (k < 1 || k > h->k_max || k > h->E)
        return fail(MOE_EINVAL, "k = %d out of range [1, %d]", k, h->k_max < h->E ? h->k_max : h->E);
    if (h->ebase != 0 || h->etotal != h->E)
        return fail(MOE_EINVAL, "moe_forward on a handle holding experts [%d, %d) of %d: route first "
                                "(moe_route_static, moe_route_sigmoid) and call moe_forward_routed",
                    h->ebase, h->ebase + h->E, h->etotal);
    if (T == 0)
        return check_pending(h);
    if (!x_bf16 || !router_logits || !out_fp32 || !workspace)
        return fail(MOE_EINVAL, "moe_forward: NULL pointer");
    if (!aligned(x_bf16, 16) || !aligned(out_fp32, 16) || !aligned(router_logits, 4))
        return fail(MOE_EINVAL, "x and out must be 16-byte aligned, logits 4-byte aligned");
    if (!aligned(workspace, 256))
        return fail(MOE_EWORKSPACE, "workspace must be 256-byte aligned");
    MoeStatus s = check_pending(h);
    if (s != MOE_OK)
        return s;
    return run_layer(h, x_bf16, router_logits, nullptr, nullptr, T, k, out_fp32, accumulate, workspace, ws_bytes,
                     routing, (cudaStream_t)cuda_stream);
}

MoeStatus moe_forward_routed(MoeHandle *h, const void *x_bf16, const int32_t *topk_ids, const float *topk_w, int T,
                             int k, float *out_fp32, int accumulate, void *workspace, size_t ws_bytes,
                             const MoeRoutingOut *routing, void *cuda_stream)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_forward_routed: NULL handle");
    if (h->E == 0)
        return fail(MOE_EINVAL, "moe_forward_routed on a dense handle; use moe_dense_sliced_forward");
    if (T < 0 || T > (1 << 24))
        return fail(MOE_EINVAL, "T = %d out of range [0, 2^24]", T);
    if (k < 1 || k > h->k_max)
        return fail(MOE_EINVAL, "k = %d out of range [1, %d]", k, h->k_max);
    if (T == 0)
        return check_pending(h);
    if (!x_bf16 || !topk_ids || !topk_w || !out_fp32 || !workspace)
        return fail(MOE_EINVAL, "moe_forward_routed: NULL pointer");
    if (!aligned(x_bf16, 16) || !aligned(out_fp32, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(MOE_EINVAL, "x and out must be 16-byte aligned, ids and weights 4-byte aligned");
    if (!aligned(workspace, 256))
        return fail(MOE_EWORKSPACE, "workspace must be 256-byte aligned");
    MoeStatus s = check_pending(h);
    if (s != MOE_OK)
        return s;
    return run_layer(h, x_bf16, nullptr, topk_ids, topk_w, T, k, out_fp32, accumulate, workspace, ws_bytes, routing,
                     (cudaStream_t)cuda_stream);
}

MoeStatus moe_set_expert_range(MoeHandle *h, int expert_base, int n_experts_total)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_set_expert_range: NULL handle");
    if (h->E == 0)
        return fail(MOE_EINVAL, "moe_set_expert_range on a dense handle");
    if (expert_base < 0 || n_experts_total < 1 || n_experts_total > (1 << 20) ||
        (long long)expert_base + h->E > n_experts_total)
        return fail(MOE_EINVAL, "experts [%d, %d) are not a part of [0, %d) (at most 2^20 experts)", expert_base,
                    expert_base + h->E, n_experts_total);
    h->ebase = expert_base;
    h->etotal = n_experts_total;
    return MOE_OK;
}

MoeStatus moe_route_sigmoid(const float *router_logits, const float *bias, int T, int E, int k, float routed_scale,
                            int32_t *topk_ids, float *topk_w, void *cuda_stream)
{
    if (T < 0 || T > (1 << 24))
        return fail(MOE_EINVAL, "T = %d out of range [0, 2^24]", T);
    if (E < 1 || E > MOE_ROUTE_SIGMOID_MAX_EXPERTS)
        return fail(MOE_EINVAL, "E = %d out of range [1, %d]", E, MOE_ROUTE_SIGMOID_MAX_EXPERTS);
    if (k < 1 || k > E || k > 32)
        return fail(MOE_EINVAL, "k = %d out of range [1, min(E, 32)]", k);
    if (T == 0)
        return MOE_OK;
    if (!router_logits || !topk_ids || !topk_w)
        return fail(MOE_EINVAL, "moe_route_sigmoid: NULL pointer");
    if (!aligned(router_logits, 4) || !aligned(bias, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(MOE_EINVAL, "moe_route_sigmoid: arrays must be 4-byte aligned");
    cudaError_t e = launch_router_sigmoid(router_logits, bias, T, E, k, routed_scale, topk_ids, topk_w,
                                          (cudaStream_t)cuda_stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "sigmoid router launch");
    return MOE_OK;
}

MoeStatus moe_dense_sliced_forward(MoeHandle *h, const void *x_bf16, int T, float *out_fp32, int accumulate,
                                   void *workspace, size_t ws_bytes, void *cuda_stream)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_dense_sliced_forward: NULL handle");
    if (h->E != 0)
        return fail(MOE_EINVAL, "moe_dense_sliced_forward on a routed handle; use moe_forward");
    if (T < 0 || T > (1 << 24))
        return fail(MOE_EINVAL, "T = %d out of range [0, 2^24]", T);
    if (T == 0)
        return check_pending(h);
    if (!x_bf16 || !out_fp32 || !workspace)
        return fail(MOE_EINVAL, "moe_dense_sliced_forward: NULL pointer");
    if (!aligned(x_bf16, 16) || !aligned(out_fp32, 16))
        return fail(MOE_EINVAL, "x and out must be 16-byte aligned");
    if (!aligned(workspace, 256))
        return fail(MOE_EWORKSPACE, "workspace must be 256-byte aligned");
    MoeStatus s = check_pending(h);
    if (s != MOE_OK)
        return s;
    return run_layer(h, x_bf16, nullptr, nullptr, nullptr, T, 0, out_fp32, accumulate, workspace, ws_bytes, nullptr,
                     (cudaStream_t)cuda_stream);
}

MoeStatus moe_sync_status(MoeHandle *h, void *cuda_stream)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_sync_status: NULL handle");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)cuda_stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    MoeStatus s = check_pending(h);
    if (s != MOE_OK)
        return s;
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "CUDA runtime");
    return MOE_OK;
}

// ---------------------------------------------------------------- CUDA graphs

struct MoeGraph {
    MoeHandle *h = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

MoeStatus moe_graph_create(MoeHandle *h, const void *x_bf16, const float *router_logits, const int32_t *topk_ids,
                           const float *topk_w, int T, int k, float *out_fp32, int accumulate, void *workspace,
                           size_t ws_bytes, const MoeHostIO *host, MoeGraph **graph)
{
    if (!graph)
        return fail(MOE_EINVAL, "moe_graph_create: NULL graph pointer");
    *graph = nullptr;
    if (!h)
        return fail(MOE_EINVAL, "moe_graph_create: NULL handle");
    if (T < 1)
        return fail(MOE_EINVAL, "moe_graph_create: T = %d, a graph needs at least one token", T);
    if (h->E > 0 && !router_logits == !topk_ids)
        return fail(MOE_EINVAL, "moe_graph_create: give either router logits or ids + weights");
    // capture the call on a private stream, in this thread's capture mode only
    cudaStream_t cs;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamCreateWithFlags");
    if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return cuda_fail(e, "cudaStreamBeginCapture");
    }
    // optional copies of the step's inputs from pinned host memory, before the call
    auto h2d = [&](void *dst, const void *src, size_t bytes) {
        return dst && src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, cs) : cudaSuccess;
    };
    const size_t tk = (size_t)T * (size_t)(k > 0 ? k : 0);
    if (host && (e = h2d((void *)x_bf16, host->x_host, (size_t)T * h->H * 2)) == cudaSuccess &&
        (e = h2d((void *)router_logits, host->logits_host, (size_t)T * h->E * sizeof(float))) == cudaSuccess &&
        (e = h2d((void *)topk_ids, host->ids_host, tk * sizeof(int32_t))) == cudaSuccess)
        e = h2d((void *)topk_w, host->w_host, tk * sizeof(float));
    if (e != cudaSuccess) {
        cudaGraph_t g0 = nullptr;
        cudaStreamEndCapture(cs, &g0);
        if (g0)
            cudaGraphDestroy(g0);
        cudaStreamDestroy(cs);
        return cuda_fail(e, "moe_graph_create: input copy");
    }
    MoeStatus st;
    if (h->E == 0)
        st = moe_dense_sliced_forward(h, x_bf16, T, out_fp32, accumulate, workspace, ws_bytes, cs);
    else if (router_logits)
        st = moe_forward(h, x_bf16, router_logits, T, k, out_fp32, accumulate, workspace, ws_bytes, nullptr, cs);
    else
        st = moe_forward_routed(h, x_bf16, topk_ids, topk_w, T, k, out_fp32, accumulate, workspace, ws_bytes,
                                nullptr, cs);
    // optional copy of the result to pinned host memory, after the call
    if (st == MOE_OK && host && host->out_host &&
        (e = cudaMemcpyAsync(host->out_host, out_fp32, (size_t)T * h->H * sizeof(float), cudaMemcpyDeviceToHost,
                             cs)) != cudaSuccess)
        st = cuda_fail(e, "moe_graph_create: output copy");
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (st != MOE_OK) {
        if (g)
            cudaGraphDestroy(g);
        return st;  // the failing call has set the message
    }
    if (e != cudaSuccess || !g) {
        if (g)
            cudaGraphDestroy(g);
        return cuda_fail(e != cudaSuccess ? e : cudaErrorStreamCaptureInvalidated, "cudaStreamEndCapture");
    }
    cudaGraphExec_t ex = nullptr;
    if ((e = cudaGraphInstantiate(&ex, g, 0)) != cudaSuccess) {
        cudaGraphDestroy(g);
        return cuda_fail(e, "cudaGraphInstantiate");
    }
    MoeGraph *mg = new (std::nothrow) MoeGraph;
    if (!mg) {
        cudaGraphExecDestroy(ex);
        cudaGraphDestroy(g);
        return fail(MOE_ENOMEM, "moe_graph_create: out of host memory");
    }
    mg->h = h;
    mg->graph = g;
    mg->exec = ex;
    *graph = mg;
    return MOE_OK;
}

MoeStatus moe_graph_launch(MoeGraph *g, void *cuda_stream)
{
    if (!g)
        return fail(MOE_EINVAL, "moe_graph_launch: NULL graph");
    MoeStatus s = check_pending(g->h);
    if (s != MOE_OK)
        return s;
    cudaError_t e = cudaGraphLaunch(g->exec, (cudaStream_t)cuda_stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGraphLaunch");
    return MOE_OK;
}

void moe_graph_free(MoeGraph *g)
{
    if (!g)
        return;
    if (g->exec)
        cudaGraphExecDestroy(g->exec);
    if (g->graph)
        cudaGraphDestroy(g->graph);
    delete g;
}

MoeStatus moe_profile_enable(MoeHandle *h, int enable)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_profile_enable: NULL handle");
    if (enable && !h->ev[0]) {
        for (cudaEvent_t &ev : h->ev) {
            cudaError_t e = cudaEventCreate(&ev);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaEventCreate");
        }
    }
    h->profile = enable != 0;
    h->profiled = false;
    return MOE_OK;
}

int moe_profile_read(MoeHandle *h, float *ms, int n)
{
    if (!h || !ms || !h->profile || !h->profiled)
        return -1;
    if (cudaEventSynchronize(h->ev[N_STAGES]) != cudaSuccess)
        return -1;
    int m = n < N_STAGES ? n : N_STAGES;
    for (int i = 0; i < m; ++i) {
        float t = 0.f;
        cudaEventElapsedTime(&t, h->ev[i], h->ev[i + 1]);
        ms[i] = t;
    }
    return m;
}

MoeStatus moe_debug_expire_next_wait(MoeHandle *h, int limit_us)
{
    if (!h)
        return fail(MOE_EINVAL, "moe_debug_expire_next_wait: NULL handle");
    if (limit_us < 1 || limit_us > 1000000)
        return fail(MOE_EINVAL, "moe_debug_expire_next_wait: limit %d us outside [1, 1000000]", limit_us);
    h->expire_wait_us = limit_us;
    return MOE_OK;
}

const char *moe_last_error(void) { return g_msg; }

void moe_free(MoeHandle *h)
{
    if (!h)
        return;
    cudaDeviceSynchronize();
    destroy(h);
}

}  // extern "C"
