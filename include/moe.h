/*
 * moe.h -- C ABI of libmoe_gb300.so, a GB300 (sm_103a) Mixture-of-Experts
 * feed-forward layer with MXFP4 expert weights.
 *
 * What one forward call computes, step by step (sources are named by page
 * title and section):
 *
 *  1. Routing.  For each token t, softmax over the E router logits, keep the
 *     k largest and renormalise over them, so that w_tj = exp(l_tj - l_max) /
 *     sum_{j' < k} exp(l_tj' - l_max).  Larger logits come first; equal logits
 *     (+0 equals -0) go to the lower expert index; NaN ranks below every
 *     number.  The expert computation sees the routing only as one expert id
 *     and one weight per selection ("Cascadia: Resident 975B MoE Inference on
 *     Eleven AI PCs" §3.1).
 *  2. Grouping.  Slots s = t*k + j are grouped by expert with a stable counting
 *     sort (ascending slot order within an expert) -- the expert-major
 *     arrangement of the same paper's §3.1.
 *  3. Experts.  Every routed expert, and every shared expert (always included,
 *     weight 1.0, same paper §3.1), is a SwiGLU FFN
 *        h = SiLU(x W_g^T) * (x W_u^T),   y = h W_d^T,   SiLU(z) = z / (1 + e^-z)
 *     whose weights are OCP MXFP4: 4-bit E2M1 codes c with one unsigned E8M0
 *     exponent e per 32 consecutive values of a row, decoding to
 *     v(c) * 2^(e-127), v over {0, 0.5, 1, 1.5, 2, 3, 4, 6} plus a sign bit
 *     (4.25 bits per weight) -- "DeepSeek-V4-Flash on a four-GPU Ampere
 *     workstation", section "MXFP4 is not NVFP4, and the difference matters on
 *     Ampere".  Weights are decoded on chip inside the reduction; no BF16 copy
 *     of an expert is ever written to device memory.  Products accumulate in
 *     FP32; h is kept between the two projections in FP16 with a power-of-two
 *     scale (per token on the tensor-core path, per token and 64 features on
 *     the decode path), or as a BF16 hi + lo pair when the weights are BF16.
 *     Weights may also be BF16, or group-32 INT4 with an FP16 scale and a zero
 *     point per 32 values (the format of "Cascadia" §3.1; MoeWeightFormat).
 *  4. Combine.  out_t = sum_{j<k} w_tj y_{e_tj}(x_t) + sum_shared y_s(x_t) in
 *     FP32 ("Cascadia" §3.3, Eq. 1), written to (or, with accumulate, added
 *     to) the caller's FP32 buffer.
 *
 *  A dense SwiGLU FFN is run as n_slices all-active slices of its intermediate
 *  dimension, each with unit weight ("Cascadia" §3.4, Eq. 2).
 *
 *  Other entry points: moe_forward_routed runs steps 2-4 on expert ids and
 *  weights the caller computed (the interface of "Cascadia" §3.1, whose router
 *  runs elsewhere); moe_route_sigmoid is that paper's routing variant (sigmoid
 *  scores, bias-adjusted selection); moe_graph_create / moe_graph_launch
 *  replay a captured forward call as one CUDA graph; moe_route_static routes
 *  and groups without a workspace.
 *
 * Layouts (all row-major, C order):
 *  - pack4 (MXFP4 codes): byte j of a row holds element 2j in its low nibble
 *    and element 2j+1 in its high nibble.  Code bit 3 is the sign; bits 0..2
 *    index the magnitude list above in the printed order.
 *  - scales: one E8M0 byte per 32 consecutive elements of a row (INT4: one
 *    FP16 bit pattern, and one zero-point byte, per 32 elements).
 *  - BF16 tensors are 16-bit BF16 bit patterns.
 *
 * Conventions:
 *  - Tensor pointers are DEVICE pointers owned by the caller unless a comment
 *    says otherwise.  The library owns only the handle and its own repacked
 *    copy of the weights (made at load; the caller's weight buffers can be
 *    freed as soon as moe_load_weights returns).
 *  - The forward calls (moe_forward, moe_forward_routed,
 *    moe_dense_sliced_forward) enqueue work on `cuda_stream` (a cudaStream_t,
 *    NULL = legacy default stream) and return without waiting for it.  They
 *    allocate nothing and never synchronise.
 *  - Every argument is checked on the host before anything is enqueued; a bad
 *    argument returns a status, never aborts, and leaves the outputs untouched.
 *    moe_last_error() then describes the problem.
 *  - A device-side failure of an earlier call (a kernel's own bounds or wait
 *    check) is reported as MOE_EDEVICE by the next call on the same handle,
 *    or by moe_sync_status().
 *  - One handle may be used from several host threads only if the caller
 *    serialises the calls; separate handles are independent.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct MoeHandle MoeHandle;

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,     /* a NULL or misaligned pointer, a negative size, k out of range, wrong handle kind */
    MOE_EDIMS = 2,      /* hidden / inter / slice width not a multiple of 32, or too large */
    MOE_ESCALE = 3,     /* a scale the format rejects: an E8M0 byte of 255 (NaN in the OCP format); for
                           group-32 INT4 an FP16 scale that is Inf or NaN, or a zero point above 15 */
    MOE_ENOMEM = 4,     /* the library could not allocate its weight copy */
    MOE_ECUDA = 5,      /* a CUDA runtime call failed (message in moe_last_error) */
    MOE_EWORKSPACE = 6, /* workspace smaller than moe_workspace_bytes() or not 256-byte aligned */
    MOE_EDEVICE = 7     /* a kernel of an earlier call reported a device-side error */
} MoeStatus;

/* Weight formats.  MXFP4 and BF16 as in "DeepSeek-V4-Flash on a four-GPU
 * Ampere workstation" (section "MXFP4 is not NVFP4, and the difference matters
 * on Ampere").  MOE_W_INT4G32 is the group-32 INT4 format of "Cascadia:
 * Resident 975B MoE Inference on Eleven AI PCs" (§3.1: packed 4-bit nibbles
 * with one FP16 scale per 32-value group; §3.5: zero points): the weight is
 * s * (q - z) for the unsigned code q and its group's FP16 scale s and zero
 * point z in 0..15.  INT4 layers run both paths: the single kernel decodes
 * s * (q - z) exactly (FP16 q - z, the scale applied in FP32 to each 32-value
 * block); the tensor-core GEMMs of larger batches split each weight, relative
 * to a power of two per row, into an FP16 pair hi + lo and run two MMAs per K
 * step (exact for every group whose scale is within 2^-24 of its row's
 * largest; smaller groups round at about 2^-35 of the row's largest weight). */
typedef enum { MOE_W_MXFP4 = 0, MOE_W_BF16 = 1, MOE_W_INT4G32 = 2 } MoeWeightFormat;

typedef struct {
    int hidden;            /* H, multiple of 32, 32 .. 65536 */
    int inter;             /* I per expert, or the dense FFN's total I; multiple of 32 */
    int n_experts;         /* E routed experts (1 .. 1024); for a dense layer: n_slices */
    int n_shared;          /* S always-on shared experts (0 .. 64); 0 for a dense layer */
    int k_max;             /* largest k a forward call may ask for, 1 .. 32 (moe_forward also needs
                              k <= E; moe_forward_routed does not); ignored when dense */
    int n_slices;          /* 0: routed MoE layer.  > 0: dense FFN cut into this many slices */
    MoeWeightFormat fmt;   /* MXFP4, BF16 or group-32 INT4 weights */
} MoeConfig;

/* One weight matrix.  MXFP4: codes = pack4 bytes [rows][cols/2] (element 2j
 * in the low nibble of byte j), scales = E8M0 bytes [rows][cols/32].
 * BF16: codes = BF16 [rows][cols], scales NULL.  INT4G32: codes as for MXFP4
 * (unsigned 4-bit codes), scales = FP16 bits [rows][cols/32] (2-byte
 * aligned), zeros = zero point bytes [rows][cols/32] or NULL (every zero
 * point 8: the symmetric grid -8..7).  zeros is ignored by the other formats.
 * Device pointers; any alignment except the INT4 scales'. */
typedef struct {
    const void *codes;
    const void *scales;
    const void *zeros;
} MoeMx;

/* Copy the weights into the library's own storage and return a handle.
 *
 * Routed layer (n_slices == 0): gate_up[g] and down[g] for g in [0, E+S);
 *   g < E are the routed experts, g >= E the shared ones.
 *   gate_up[g] is the [2I][H] matrix whose rows 0..I-1 are W_g and rows
 *   I..2I-1 are W_u; down[g] is W_d [H][I].
 * Dense layer (n_slices > 0, n_experts == n_slices, n_shared == 0):
 *   gate_up[0] = W_g [I][H], gate_up[1] = W_u [I][H], down[0] = W_d [H][I],
 *   all unsliced.  The library cuts I into n_slices equal slices; each width
 *   must be a multiple of 32 so that no MX block is cut (a requested split
 *   that would cut a 32-value block is rejected, as the loader rule in
 *   "DeepSeek-V4-Flash on a four-GPU Ampere workstation", section "Why it
 *   would not run", requires; weights and their scales are sliced together).
 *
 * The library repacks into its own buffers (a copy, never a view of the
 * caller's memory, per the same section's note on narrow() views).  The call
 * is synchronous: it waits for `cuda_stream` before returning.
 * Errors: MOE_EINVAL (NULL pointers, bad counts, INT4 scales not 2-byte
 * aligned), MOE_EDIMS, MOE_ESCALE, MOE_ENOMEM, MOE_ECUDA.  *out is set only
 * on MOE_OK. */
MoeStatus moe_load_weights(const MoeConfig *cfg, const MoeMx *gate_up, const MoeMx *down, void *cuda_stream,
                           MoeHandle **out);

/* Bytes of device workspace a forward call with T tokens and top-k needs
 * (for a dense handle pass k = 0).  0 for a NULL handle or T <= 0. */
size_t moe_workspace_bytes(const MoeHandle *h, int T, int k);

/* Optional routing outputs of moe_forward; each pointer may be NULL.
 *  topk_ids [T][k] int32, topk_w [T][k] float (j = 0 has the largest weight),
 *  expert_offsets [E+1] int32 (first sorted position of each expert,
 *  expert_offsets[E] = T*k), sorted_slot [T*k] int32 (slot s = t*k + j at
 *  sorted position p), slot_pos [T*k] int32 (inverse of sorted_slot). */
typedef struct {
    int *topk_ids;
    float *topk_w;
    int *expert_offsets;
    int *sorted_slot;
    int *slot_pos;
} MoeRoutingOut;

/* One routed MoE layer on T tokens.
 *  x_bf16        [T][H] BF16, 16-byte aligned
 *  router_logits [T][E] float, 4-byte aligned
 *  out_fp32      [T][H] float, 16-byte aligned; overwritten, or added to when
 *                accumulate != 0 (e.g. a residual stream)
 *  workspace     >= moe_workspace_bytes(h, T, k) bytes, 256-byte aligned;
 *                contents on entry do not matter
 *  routing       NULL or device pointers that receive the routing
 * T == 0 enqueues nothing and returns MOE_OK.
 * Errors: MOE_EINVAL (NULL/misaligned pointers, T < 0, k outside
 * [1, min(k_max, E)], a dense handle, a handle given an expert range other
 * than [0, E) of E), MOE_EWORKSPACE, MOE_EDEVICE, MOE_ECUDA. */
MoeStatus moe_forward(MoeHandle *h, const void *x_bf16, const float *router_logits, int T, int k, float *out_fp32,
                      int accumulate, void *workspace, size_t ws_bytes, const MoeRoutingOut *routing,
                      void *cuda_stream);

/* One routed MoE layer on T tokens for routing given by the caller: the
 * interface of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1,
 * whose expert computation receives one expert id and one weight per
 * selection from a router that runs elsewhere (the shared experts are added
 * with weight 1, as in moe_forward).
 *  topk_ids [T][k] int32 in [0, E) or -1, 4-byte aligned (an expert may
 *           appear more than once for a token; each occurrence is its own
 *           slot).  -1 is an empty slot: it adds nothing and its weight is
 *           not read.  On a handle given an expert range (moe_set_expert_range)
 *           the ids are global ids in [0, n_experts_total) or -1, and a slot
 *           of an expert outside the handle's range is an empty slot too.
 *  topk_w   [T][k] float, 4-byte aligned, used as given
 *  other arguments as for moe_forward; `routing` receives the copy of the
 *  ids (the handle's own expert indices 0..E-1) and weights the layer ran
 *  with (an empty slot: id -1, weight 0) and the grouping: expert_offsets[E]
 *  is then the number of non-empty slots, slot_pos is -1 for an empty slot
 *  and sorted_slot is -1 at the positions from expert_offsets[E] to T*k.
 * Any other id cannot be checked on the host: the device records it, runs
 * that slot as expert 0 with weight 0 so that every access stays in bounds,
 * and moe_sync_status() then reports MOE_EDEVICE.
 * Errors: MOE_EINVAL (NULL/misaligned pointers, T < 0, k outside [1, k_max],
 * a dense handle), MOE_EWORKSPACE, MOE_EDEVICE, MOE_ECUDA. */
MoeStatus moe_forward_routed(MoeHandle *h, const void *x_bf16, const int32_t *topk_ids, const float *topk_w, int T,
                             int k, float *out_fp32, int accumulate, void *workspace, size_t ws_bytes,
                             const MoeRoutingOut *routing, void *cuda_stream);

/* Expert parallelism: the handle's E routed experts are experts
 * [expert_base, expert_base + E) of a layer of n_experts_total, held in order
 * (its expert i is the layer's expert expert_base + i).  moe_forward_routed
 * then takes the layer's global expert ids and runs only the slots of the
 * experts held, as empty slots otherwise, so that the outputs of holders of
 * disjoint ranges (the shared experts loaded on one of them) add up to the
 * whole layer: Eq. (1) of "Cascadia: Resident 975B MoE Inference on Eleven AI
 * PCs" §3.3 is a sum over experts.  The token rows and routing are given to
 * every holder whole, and the caller adds the FP32 outputs (an all-reduce or
 * reduce-scatter across devices).  moe_forward, which routes over the
 * handle's own experts, is refused on a handle with a range other than
 * [0, E) of E.  Host-side only: no device work; applies to later calls.
 * Errors: MOE_EINVAL (NULL or dense handle, expert_base < 0,
 * expert_base + E > n_experts_total, n_experts_total > 2^20). */
MoeStatus moe_set_expert_range(MoeHandle *h, int expert_base, int n_experts_total);

/* Largest E moe_route_sigmoid takes (one warp per token, 32 experts a lane). */
#define MOE_ROUTE_SIGMOID_MAX_EXPERTS 1024

/* The routing variant of "Cascadia" §3.1: sigmoid scores, a bias-adjusted
 * top-k selection, and weights normalised over the selected experts times a
 * model scale factor.  For token t: s_e = 1 / (1 + exp(-l_te)); the k
 * largest keys s_e + bias_e are kept (larger first, equal keys by the lower
 * index, a NaN after every number); w_j = routed_scale * s_j / sum of the
 * kept s.  The bias decides only the selection.  Scores and keys are FP64,
 * weights are stored as float.  The outputs feed moe_forward_routed.
 *  router_logits [T][E] float, bias [E] float or NULL (zeros), topk_ids and
 *  topk_w [T][k]: device pointers, 4-byte aligned, enqueued on cuda_stream.
 * No handle and no workspace.  T == 0 enqueues nothing.
 * Errors: MOE_EINVAL (T < 0, E outside [1, MOE_ROUTE_SIGMOID_MAX_EXPERTS], k
 * outside [1, min(E, 32)], NULL or misaligned pointers), MOE_ECUDA. */
MoeStatus moe_route_sigmoid(const float *router_logits, const float *bias, int T, int E, int k, float routed_scale,
                            int32_t *topk_ids, float *topk_w, void *cuda_stream);

/* ---- CUDA graphs: one forward call captured with fixed buffers ----
 *
 * A captured call replays with one launch: the counter clear, the layer's
 * kernels and their dependencies become one graph.  For a routed handle give
 * either router_logits (moe_forward) or topk_ids + topk_w (moe_forward_routed);
 * for a dense handle neither (moe_dense_sliced_forward).  The other arguments
 * are those of the captured call.  The graph keeps every pointer it was
 * created with: write each step's inputs into the same x / logits / ids /
 * weights buffers before moe_graph_launch, read out afterwards, and keep the
 * buffers and the workspace alive and unused by other calls while a launch is
 * in flight.  T is fixed per graph.  To serve a varying number of tokens,
 * create one graph per bucket of T and pad: with ids + weights, give padded
 * rows an id some real row uses and weight 0, so that they add no expert
 * (their own out rows are to be ignored; real rows agree with an unpadded call
 * within the layer's error bound, as the grouping, and with it the order of
 * some sums, can differ).
 * host (may be NULL; each member may be NULL) adds copies to the graph: the
 * step's x, logits or ids and weights from PINNED host memory into the
 * captured device buffers before the call, and out back to pinned host
 * memory after it, so that one launch runs a whole serving step.
 * Capture runs on a private stream in this thread's capture mode; nothing is
 * enqueued by moe_graph_create.  Argument errors are those of the captured
 * call.
 * Errors: MOE_EINVAL (NULL graph pointer or handle, T < 1, both or neither of
 * logits and ids for a routed handle, or any error of the captured call),
 * MOE_EWORKSPACE, MOE_EDEVICE, MOE_ENOMEM, MOE_ECUDA.  *graph is set only on
 * MOE_OK. */
typedef struct MoeGraph MoeGraph;
typedef struct {
    const void *x_host;         /* [T][H] BF16, copied into x_bf16 */
    const float *logits_host;   /* [T][E], copied into router_logits */
    const int32_t *ids_host;    /* [T][k], copied into topk_ids */
    const float *w_host;        /* [T][k], copied into topk_w */
    float *out_host;            /* [T][H], receives out_fp32 */
} MoeHostIO;
MoeStatus moe_graph_create(MoeHandle *h, const void *x_bf16, const float *router_logits, const int32_t *topk_ids,
                           const float *topk_w, int T, int k, float *out_fp32, int accumulate, void *workspace,
                           size_t ws_bytes, const MoeHostIO *host, MoeGraph **graph);

/* Replays a captured call on cuda_stream.  Errors: MOE_EINVAL (NULL graph),
 * MOE_EDEVICE (an earlier call reported a device error), MOE_ECUDA. */
MoeStatus moe_graph_launch(MoeGraph *graph, void *cuda_stream);

/* Frees a graph (NULL is a no-op).  No launch of it may be in flight. */
void moe_graph_free(MoeGraph *graph);

/* The dense FFN of a dense handle on T tokens, as the sum of its all-active
 * slices ("Cascadia" §3.4, Eq. 2).  Arguments as for moe_forward; the
 * workspace size is moe_workspace_bytes(h, T, 0).
 * Errors: MOE_EINVAL (also for a routed handle), MOE_EWORKSPACE, MOE_EDEVICE,
 * MOE_ECUDA. */
MoeStatus moe_dense_sliced_forward(MoeHandle *h, const void *x_bf16, int T, float *out_fp32, int accumulate,
                                   void *workspace, size_t ws_bytes, void *cuda_stream);

/* Wait for `cuda_stream`, then report MOE_EDEVICE if any kernel of this handle
 * has flagged a device-side error, MOE_ECUDA if the CUDA runtime reports an
 * error, else MOE_OK.  The flag is sticky until moe_free. */
MoeStatus moe_sync_status(MoeHandle *h, void *cuda_stream);

/* Per-stage timing for benchmarking.  While enabled, every forward call on
 * this handle records CUDA events on its stream around its stages.  Stages:
 * [0] routing (router kernel, or the copy of caller routing), [1] grouping and
 * token rows (histogram + permutation, or the dense plan; then, with FP16
 * operands, the per-token FP16 conversion, and the gather of token rows into
 * position order), [2] gate|up GEMM with SwiGLU (with FP16 operands also the
 * clear of the per-position maxima and the conversion of h to one FP16 plane),
 * [3] down GEMM, [4] combine, [5] the single-kernel layer that decode-sized
 * batches run instead of [0]..[4].  A stage a call does not run reads 0.
 * Errors: MOE_EINVAL (NULL handle), MOE_ECUDA (event creation failed). */
MoeStatus moe_profile_enable(MoeHandle *h, int enable);

/* Wait for the events of the most recent profiled call and write up to n
 * stage durations in milliseconds to the HOST array ms.  Returns the number of
 * stages written (at most 6), or -1 if profiling is off or no call was profiled. */
int moe_profile_read(MoeHandle *h, float *ms, int n);

/* Limits of moe_route_static's fixed scratch. */
#define MOE_ROUTE_STATIC_MAX_EXPERTS 1024
#define MOE_ROUTE_STATIC_MAX_SLOTS 65536 /* T * k */

/* Routing and grouping without any device allocation.  No counterpart in the
 * paper: this is a deployment variant of the routing step of moe_forward.
 *
 * It is for callers that cannot allocate device memory or hand the library a
 * workspace: for example code that runs while another allocator owns all
 * free device memory, or a latency-bound loop where cudaMalloc/cudaFree
 * would synchronise the device and stall other streams.  The call runs the
 * same router, histogram and permutation kernels as moe_forward and writes
 * the same routing results.  Their scratch (expert counts, group table,
 * position -> token map; 274,436 bytes) is a fixed array in the library's
 * device memory, one per device, that exists from module load to process
 * exit.  No cudaMalloc, cudaFree or other allocating routine is called.
 *
 *  router_logits  [T][E] float, device
 *  topk_ids       [T][k] int32, device; j = 0 has the largest weight
 *  topk_w         [T][k] float, device; softmax over the k kept logits
 *  expert_offsets [E+1] int32, device
 *  sorted_slot    [T*k] int32, device (slot s = t*k + j at sorted position p)
 *  slot_pos       [T*k] int32, device (inverse of sorted_slot)
 *  cuda_stream    cudaStream_t or NULL; all work is enqueued on it
 * Outputs are as in MoeRoutingOut.  T == 0 enqueues nothing.
 *
 * Set-up: the first call made with a given device current looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it for later calls
 * on that device.  Make that first call before any stream capture starts.
 *
 * Shared scratch: every call on a device uses the same array.  The expert
 * counts in it must start at zero; the router kernel of each call zeroes
 * them itself, so the caller clears nothing.  Two calls whose work overlaps
 * on the GPU (on different streams, or from several threads without an
 * ordering between their streams) race on the array and give wrong results:
 * order them on one stream, or with events.
 *
 * Device-side checks: the kernels record a failure in a flag of the same
 * scratch, which this call clears on its stream before its kernels run; read
 * it with moe_route_static_status().
 *
 * Errors: MOE_EINVAL (E outside [1, MOE_ROUTE_STATIC_MAX_EXPERTS], k outside
 * [1, min(E, 32)], T < 0, T * k > MOE_ROUTE_STATIC_MAX_SLOTS, NULL pointer),
 * MOE_EDEVICE (device ordinal >= 64), MOE_ECUDA (symbol lookup or launch
 * failed).  The message is available from moe_last_error(). */
MoeStatus moe_route_static(const float *router_logits, int T, int E, int k, int *topk_ids, float *topk_w,
                           int *expert_offsets, int *sorted_slot, int *slot_pos, void *cuda_stream);

/* Device-side status of moe_route_static on the current device.  Waits for
 * cuda_stream, then reads the error flag that the routing and grouping kernels
 * set in the fixed scratch (a permutation whose counts disagree with the
 * histogram).  Each moe_route_static call clears the flag on its stream before
 * its kernels run, so the status covers the most recent call on this device
 * (and any call that overlapped it).  Allocates nothing; a 4-byte synchronous
 * device-to-host copy reads the flag.
 * Returns MOE_OK (also when no call has run on this device), MOE_EDEVICE (the
 * flag is set, or the device ordinal is >= 64) or MOE_ECUDA. */
MoeStatus moe_route_static_status(void *cuda_stream);

/* Test hook for the device-side wait limit.  No counterpart in the paper.
 * Every wait in the kernels is bounded in time; this arms the next forward
 * call on this handle that runs the single-kernel path (a decode-sized batch)
 * so that its grid-wide completion wait before the combine has a target no
 * launch reaches and a limit of limit_us microseconds.  The wait then expires
 * in every CTA, which records a timeout and leaves without combining (out is
 * not written).  That wait runs after all of the kernel's copies and MMAs
 * have finished.  The handle's sticky device error is then reported as
 * MOE_EDEVICE by moe_sync_status and later calls; use a fresh handle
 * afterwards.  Not for production use.
 * Errors: MOE_EINVAL (NULL handle, limit_us outside [1, 1000000]). */
MoeStatus moe_debug_expire_next_wait(MoeHandle *h, int limit_us);

/* Human-readable description of the last non-OK status returned on the
 * calling thread (thread-local, never NULL). */
const char *moe_last_error(void);

/* Release the handle and the library's weight copy (waits for the device). */
void moe_free(MoeHandle *h);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
