/*
 * moe_oracle.c -- plain, slow CPU oracle of the MXFP4 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; it is written from the pages' definitions alone.
 *
 * Precision: MXFP4 (and BF16) weights are decoded exactly to float32, then all
 * arithmetic (routing weights, dot products, SiLU, combine) is done in double.
 *
 * Sources (page title, section / equation):
 *  [MX]  "DeepSeek-V4-Flash on a four-GPU Ampere workstation", section "MXFP4 is
 *        not NVFP4, and the difference matters on Ampere": a decoded weight is
 *        v(c) * 2^(e-127) for the 4-bit E2M1 code c of a 32-value block with
 *        unsigned E8M0 exponent e; the E2M1 magnitudes are
 *        {0, 0.5, 1, 1.5, 2, 3, 4, 6} plus one sign bit; a block costs
 *        4 + 8/32 = 4.25 bits per weight.
 *  [C31] "Cascadia: Resident 975B MoE Inference on Eleven AI PCs" §3.1: each
 *        expert is a SwiGLU FFN (gate/up projections, SwiGLU, down projection),
 *        expert outputs are combined by a weighted reduction with the routing
 *        weights, the experts see the routing only as ids and weights, and shared experts
 *        are always included.
 *  [C33] same paper §3.3, Eq. (1): y_i = sum_e w_ie E_e(x_i).
 *  [C34] same paper §3.4, Eq. (2): the dense FFN equals the sum of its
 *        intermediate-dimension slices, every slice active with unit weight.
 *  [I4]  same paper §3.1 (the exporter keeps the experts' group-32 INT4
 *        packed nibbles and stores each group's scale as FP16) and §3.5 (the
 *        expert bytes it counts include scale and zero-point overhead).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Router: softmax over all experts, keep the k largest, renormalise over
 *    the k kept (the full softmax denominator cancels).  Order: larger logit
 *    first; equal logits (+0 and -0 are equal) by lower expert index; NaN
 *    ranks below every number.
 *  - Nibble order: element 2j is the low nibble of byte j, 2j+1 the high one.
 *    Code bit 3 is the sign, bits 0..2 index the magnitude list in the order
 *    the page prints it.
 *  - E8M0 = 255 is NaN in the OCP format and is rejected.
 *  - Shared experts have weight 1.0 and are added outside the renormalisation.
 *  - Slots of one expert are kept in ascending slot order s = t*k + j.
 *  - Group-32 INT4 [I4]: a weight is s * (q - z) for its unsigned 4-bit code q,
 *    and the FP16 scale s and zero point z (0..15, one byte) of its group of
 *    32 consecutive values along a row.  Element 2j is the low nibble of byte
 *    j, as for MXFP4.  Without stored zero points every z is 8, which is the
 *    symmetric signed grid -8..7.  A scale that is Inf or NaN, or a zero point
 *    above 15, is rejected.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decode */

/* The E2M1 magnitudes as printed in [MX], indexed by the 3 low code bits. */
static const double E2M1_MAGNITUDES[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* v(c): value of a 4-bit E2M1 code, bit 3 being the sign bit [MX]. */
double oracle_e2m1_value(int code)
{
    double m = E2M1_MAGNITUDES[code & 7];
    return (code & 8) ? -m : m;
}

/* Decoded weight v(c) * 2^(e-127) of [MX], computed in double then rounded to
 * float (exact whenever the value is representable in float). */
float oracle_mx_value(int code, int e8m0)
{
    return (float)ldexp(oracle_e2m1_value(code), e8m0 - 127);
}

/* Storage of an MXFP4 matrix [rows, cols]: cols/2 code bytes plus cols/32
 * scale bytes per row, i.e. 4 + 8/32 = 4.25 bits per weight [MX]. */
int64_t oracle_mx_bytes(int64_t rows, int64_t cols)
{
    return rows * (cols / 2) + rows * (cols / 32);
}

/* Decode an MXFP4 matrix [rows, cols] (codes [rows, cols/2], scales
 * [rows, cols/32]) to float.  Element i of a row takes scale floor(i/32) [MX].
 * Returns 0, or -1 if a scale byte is 255 (NaN in E8M0). */
int oracle_mx_decode(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t cols, float *out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t *cr = codes + r * (cols / 2);
        const uint8_t *sr = scales + r * (cols / 32);
        for (int64_t i = 0; i < cols; ++i) {
            int e = sr[i / 32];
            if (e == 255)
                return -1;
            uint8_t byte = cr[i / 2];
            int code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[r * cols + i] = oracle_mx_value(code, e);
        }
    }
    return 0;
}

/* BF16 bit patterns to float (exact). */
void oracle_bf16_decode(const uint16_t *bits, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)bits[i] << 16;
        memcpy(&out[i], &u, 4);
    }
}

/* IEEE binary16 bits to double: sign bit 15, exponent bits 10..14 (bias 15),
 * fraction bits 0..9.  Exponent 0 is zero or subnormal (fraction * 2^-24);
 * exponent 31 is Inf (fraction 0) or NaN. */
double oracle_fp16_value(int bits)
{
    int sign = (bits >> 15) & 1, ex = (bits >> 10) & 31, fr = bits & 1023;
    double v;
    if (ex == 31)
        v = fr ? NAN : INFINITY;
    else if (ex == 0)
        v = ldexp((double)fr, -24);
    else
        v = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -v : v;
}

/* Decoded group-32 INT4 weight s * (q - z) [I4], computed in double and
 * rounded to float.  The rounding is exact: |q - z| <= 15 has 4 significant
 * bits and s has at most 11. */
float oracle_i4_value(int q, int z, int scale_bits)
{
    return (float)((double)(q - z) * oracle_fp16_value(scale_bits));
}

/* Storage of a group-32 INT4 matrix [rows, cols]: cols/2 code bytes, then
 * per 32 values a 2-byte FP16 scale and (when stored) a 1-byte zero point:
 * 4 + 16/32 (+ 8/32) bits per weight. */
int64_t oracle_i4_bytes(int64_t rows, int64_t cols, int with_zeros)
{
    return rows * (cols / 2) + rows * (cols / 32) * (with_zeros ? 3 : 2);
}

/* Decode a group-32 INT4 matrix [rows, cols] to float: codes [rows, cols/2],
 * FP16 scale bits [rows, cols/32], zero points [rows, cols/32] or NULL (all
 * 8).  Element i of a row takes group floor(i/32) [I4].  Returns 0, or -1 if a
 * scale is Inf / NaN or a zero point is above 15. */
int oracle_i4_decode(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros, int64_t rows, int64_t cols,
                     float *out)
{
    const int64_t ng = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < cols; ++i) {
            const int64_t grp = r * ng + i / 32;
            const int sb = scales[grp];
            const int z = zeros ? zeros[grp] : 8;
            if (((sb >> 10) & 31) == 31 || z > 15)
                return -1;
            const uint8_t byte = codes[r * (cols / 2) + i / 2];
            const int q = (i & 1) ? (byte >> 4) : (byte & 0xF);
            out[r * cols + i] = oracle_i4_value(q, z, sb);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- router */

typedef struct {
    float v;
    int idx;
} ScoredExpert;

/* Total order of the router: a number before NaN, larger before smaller,
 * equal values (including +0 / -0, or two NaNs) by lower index. */
static int router_order(const void *pa, const void *pb)
{
    const ScoredExpert *a = (const ScoredExpert *)pa, *b = (const ScoredExpert *)pb;
    int na = isnan(a->v), nb = isnan(b->v);
    if (na != nb)
        return na ? 1 : -1;
    if (!na && a->v != b->v)
        return a->v > b->v ? -1 : 1;
    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);
}

/* Softmax top-k with renormalisation.  For token t: sort the E logits in the
 * router order, keep the first k ids, and give them weights
 * w_j = exp(l_j - l_max) / sum_{j' < k} exp(l_j' - l_max)  (double). */
void oracle_route(const float *logits, int64_t T, int E, int k, int32_t *ids, double *w)
{
    ScoredExpert *s = (ScoredExpert *)malloc(sizeof(ScoredExpert) * (size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            s[e].v = logits[t * E + e];
            s[e].idx = e;
        }
        qsort(s, (size_t)E, sizeof(ScoredExpert), router_order);
        double lmax = (double)s[0].v;
        double denom = 0.0;
        for (int j = 0; j < k; ++j)
            denom += exp((double)s[j].v - lmax);
        for (int j = 0; j < k; ++j) {
            ids[t * k + j] = s[j].idx;
            w[t * k + j] = exp((double)s[j].v - lmax) / denom;
        }
    }
    free(s);
}

/* The routing of "Cascadia: Resident 975B MoE Inference on Eleven AI PCs"
 * §3.1: sigmoid scores, a bias-adjusted top-k selection, and weights
 * normalised over the selected experts, times a model scale factor.  For
 * token t and expert e: s_e = 1 / (1 + exp(-l_e)) in double; the selection
 * key is s_e + b_e (the bias decides only which experts are kept); the k
 * largest keys are kept in the router order (larger first, equal keys by the
 * lower index, a NaN key after every number); their weights are
 * w_j = scale * s_{e_j} / sum_{j' < k} s_{e_j'}.  bias may be NULL (zeros). */
typedef struct {
    double v;
    int idx;
} KeyedExpert;

static int keyed_order(const void *pa, const void *pb)
{
    const KeyedExpert *a = (const KeyedExpert *)pa, *b = (const KeyedExpert *)pb;
    int na = isnan(a->v), nb = isnan(b->v);
    if (na != nb)
        return na ? 1 : -1;
    if (!na && a->v != b->v)
        return a->v > b->v ? -1 : 1;
    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);
}

void oracle_route_sigmoid(const float *logits, const float *bias, int64_t T, int E, int k, double scale, int32_t *ids,
                          double *w)
{
    KeyedExpert *s = (KeyedExpert *)malloc(sizeof(KeyedExpert) * (size_t)E);
    double *score = (double *)malloc(sizeof(double) * (size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            score[e] = 1.0 / (1.0 + exp(-(double)logits[t * E + e]));
            s[e].v = score[e] + (bias ? (double)bias[e] : 0.0);
            s[e].idx = e;
        }
        qsort(s, (size_t)E, sizeof(KeyedExpert), keyed_order);
        double denom = 0.0;
        for (int j = 0; j < k; ++j)
            denom += score[s[j].idx];
        for (int j = 0; j < k; ++j) {
            ids[t * k + j] = s[j].idx;
            w[t * k + j] = scale * score[s[j].idx] / denom;
        }
    }
    free(score);
    free(s);
}

/* Group slots by expert: a stable counting sort of the flattened slots
 * s = t*k + j by their expert id.  off[e] is the first sorted position of
 * expert e (off[E] = the number of slots placed), sorted_slot[p] the slot at
 * position p, and slot_pos[s] its inverse.  A slot with id -1 (empty) is not
 * placed: its slot_pos is -1, and sorted_slot holds -1 at the positions from
 * off[E] to T*k that no slot takes. */
void oracle_permute(const int32_t *ids, int64_t T, int k, int E, int32_t *off, int32_t *sorted_slot,
                    int32_t *slot_pos)
{
    int64_t n = T * k;
    int32_t *next = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    for (int e = 0; e <= E; ++e)
        off[e] = 0;
    for (int64_t s = 0; s < n; ++s)
        if (ids[s] != -1)
            off[ids[s] + 1] += 1;
    for (int e = 0; e < E; ++e)
        off[e + 1] += off[e];
    for (int e = 0; e < E; ++e)
        next[e] = off[e];
    for (int64_t p = off[E]; p < n; ++p)
        sorted_slot[p] = -1;
    for (int64_t s = 0; s < n; ++s) {
        int32_t p = ids[s] == -1 ? -1 : next[ids[s]]++;
        slot_pos[s] = p;
        if (p >= 0)
            sorted_slot[p] = (int32_t)s;
    }
    free(next);
}

/* ---------------------------------------------------------------- expert */

/* One SwiGLU FFN [C31] in double:
 *   g_n = sum_k x_k Wg[n,k],  u_n = sum_k x_k Wu[n,k],
 *   h_n = g_n / (1 + exp(-g_n)) * u_n,
 *   y_m = sum_n h_n Wd[m,n].
 * Wg/Wu rows are ld_gu floats apart, Wd rows ld_d floats apart, so that a
 * slice of a larger matrix can be passed directly [C34]. */
void oracle_swiglu_ffn(const float *Wg, const float *Wu, int64_t ld_gu, const float *Wd, int64_t ld_d, int H, int I,
                       const double *x, double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        const float *wg = Wg + (int64_t)n * ld_gu;
        const float *wu = Wu + (int64_t)n * ld_gu;
        for (int kk = 0; kk < H; ++kk) {
            g += x[kk] * (double)wg[kk];
            u += x[kk] * (double)wu[kk];
        }
        h[n] = g / (1.0 + exp(-g)) * u;
    }
    for (int m = 0; m < H; ++m) {
        double acc = 0.0;
        const float *wd = Wd + (int64_t)m * ld_d;
        for (int n = 0; n < I; ++n)
            acc += h[n] * (double)wd[n];
        y[m] = acc;
    }
    free(h);
}

/* ---------------------------------------------------------------- layer */

/* Weights of one layer.  Expert e in [0, E) is routed, [E, E+S) shared.
 * MXFP4 (weight_format 0): gu_codes[e] [2I, H/2], gu_scales[e] uint8
 * [2I, H/32] (gate rows 0..I-1, up rows I..2I-1), d_codes[e] [H, I/2],
 * d_scales[e] uint8 [H, I/32].
 * BF16 (weight_format 1): gu_codes[e] is uint16 [2I, H], d_codes[e] uint16
 * [H, I], scales unused.
 * Group-32 INT4 (weight_format 2): codes as for MXFP4, scales uint16 FP16
 * bits of the same shape, zero points uint8 of the same shape (the arrays, or
 * an entry, may be NULL: all 8).
 * An entry may be NULL when no token uses it. */
typedef struct {
    int hidden, inter, n_experts, n_shared, weight_format;
    const void *const *gu_codes;
    const void *const *gu_scales;
    const void *const *d_codes;
    const void *const *d_scales;
    const uint8_t *const *gu_zeros;
    const uint8_t *const *d_zeros;
} OracleLayer;

typedef struct {
    const float *Wgu, *Wd;
    int H, I;
    const double *x;   /* [n_tok, H] */
    double *y;         /* [n_tok, nsel, H] */
    int nsel;
    const int64_t *work; /* pairs (t, j) */
    int64_t begin, end;
} FfnJob;

static void *ffn_job_run(void *p)
{
    FfnJob *job = (FfnJob *)p;
    for (int64_t i = job->begin; i < job->end; ++i) {
        int64_t t = job->work[2 * i], j = job->work[2 * i + 1];
        oracle_swiglu_ffn(job->Wgu, job->Wgu + (int64_t)job->I * job->H, job->H, job->Wd, job->I, job->H, job->I,
                          job->x + t * job->H, job->y + (t * job->nsel + j) * job->H);
    }
    return NULL;
}

static void run_ffn_jobs(const float *Wgu, const float *Wd, int H, int I, const double *x, double *y, int nsel,
                         const int64_t *work, int64_t nwork, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nwork)
        nthreads = (int)(nwork > 0 ? nwork : 1);
    FfnJob jobs[256];
    pthread_t th[256];
    if (nthreads > 256)
        nthreads = 256;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (FfnJob){Wgu, Wd, H, I, x, y, nsel, work, nwork * i / nthreads, nwork * (i + 1) / nthreads};
    }
    if (nthreads == 1) {
        ffn_job_run(&jobs[0]);
        return;
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_create(&th[i], NULL, ffn_job_run, &jobs[i]);
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
}

static int decode_matrix(int fmt, const void *codes, const void *scales, const uint8_t *zeros, int64_t rows,
                         int64_t cols, float *out)
{
    if (codes == NULL)
        return -2;
    if (fmt == 1) {
        oracle_bf16_decode((const uint16_t *)codes, rows * cols, out);
        return 0;
    }
    if (scales == NULL)
        return -2;
    if (fmt == 2)
        return oracle_i4_decode((const uint8_t *)codes, (const uint16_t *)scales, zeros, rows, cols, out);
    return oracle_mx_decode((const uint8_t *)codes, (const uint8_t *)scales, rows, cols, out);
}

/* The layer for given routing (ids [n_tok, k] in [0, E) or -1, weights w):
 * every selected and every shared expert on its tokens, then the weighted
 * reduction
 *   out_t = sum_{j<k} w_tj * y_{e_tj}(x_t) + sum_{shared s} y_s(x_t)   [C33, C31].
 * An id of -1 is an empty slot whose term is left out of the sum (its weight
 * is not read): Eq. (1)'s sum over experts split between holders of disjoint
 * expert subsets, each summing the terms of its own experts.
 * A token's result depends only on its own x row and routing row.
 * x_bf16 [n_tok, H] BF16 bits, out [n_tok, H] double.  Returns 0, -1 (a scale
 * the format rejects), -2 (weights of a used expert missing), -3 (bad args or
 * an id out of range). */
int oracle_moe_layer_routed(const OracleLayer *L, const uint16_t *x_bf16, const int32_t *ids, const double *w,
                            int64_t n_tok, int k, int nthreads, double *out)
{
    const int H = L->hidden, I = L->inter, E = L->n_experts, S = L->n_shared;
    if (k < 1 || H % 32 || I % 32)
        return -3;
    for (int64_t i = 0; i < n_tok * k; ++i)
        if (ids[i] != -1 && (ids[i] < 0 || ids[i] >= E))
            return -3;
    const int nsel = k + S;
    int rc = 0;
    double *x = (double *)malloc(sizeof(double) * (size_t)(n_tok * H + 1));
    double *y = (double *)calloc((size_t)(n_tok * nsel * H + 1), sizeof(double));
    int64_t *work = (int64_t *)malloc(sizeof(int64_t) * (size_t)(2 * n_tok * nsel + 2));
    float *Wgu = (float *)malloc(sizeof(float) * (size_t)2 * I * H);
    float *Wd = (float *)malloc(sizeof(float) * (size_t)H * I);

    for (int64_t i = 0; i < n_tok * H; ++i) {
        uint32_t u = (uint32_t)x_bf16[i] << 16;
        float f;
        memcpy(&f, &u, 4);
        x[i] = (double)f;
    }

    for (int e = 0; e < E + S && rc == 0; ++e) {
        int64_t nwork = 0;
        for (int64_t t = 0; t < n_tok; ++t) {
            if (e >= E) {
                work[2 * nwork] = t;
                work[2 * nwork + 1] = k + (e - E);
                ++nwork;
                continue;
            }
            for (int j = 0; j < k; ++j)
                if (ids[t * k + j] == e) {
                    work[2 * nwork] = t;
                    work[2 * nwork + 1] = j;
                    ++nwork;
                }
        }
        if (nwork == 0)
            continue;
        rc = decode_matrix(L->weight_format, L->gu_codes[e], L->gu_scales ? L->gu_scales[e] : NULL,
                           L->gu_zeros ? L->gu_zeros[e] : NULL, 2 * (int64_t)I, H, Wgu);
        if (rc == 0)
            rc = decode_matrix(L->weight_format, L->d_codes[e], L->d_scales ? L->d_scales[e] : NULL,
                               L->d_zeros ? L->d_zeros[e] : NULL, H, I, Wd);
        if (rc == 0)
            run_ffn_jobs(Wgu, Wd, H, I, x, y, nsel, work, nwork, nthreads);
    }

    if (rc == 0) {
        for (int64_t t = 0; t < n_tok; ++t) {
            for (int m = 0; m < H; ++m) {
                double acc = 0.0;
                for (int j = 0; j < k; ++j)
                    if (ids[t * k + j] != -1)
                        acc += w[t * k + j] * y[(t * nsel + j) * H + m];
                for (int s = 0; s < S; ++s)
                    acc += y[(t * nsel + k + s) * H + m];
                out[t * H + m] = acc;
            }
        }
    }
    free(x);
    free(y);
    free(work);
    free(Wgu);
    free(Wd);
    return rc;
}

/* The routed MoE layer for n_tok tokens: softmax top-k routing of the logits
 * (renormalised over the k kept), then the layer for that routing.  logits
 * [n_tok, E]; the routing goes to ids_out / w_out ([n_tok, k]) when given. */
int oracle_moe_layer(const OracleLayer *L, const uint16_t *x_bf16, const float *logits, int64_t n_tok, int k,
                     int nthreads, double *out, int32_t *ids_out, double *w_out)
{
    const int E = L->n_experts;
    if (k < 1 || k > E)
        return -3;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_tok * k + 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(n_tok * k + 1));
    oracle_route(logits, n_tok, E, k, ids, w);
    int rc = oracle_moe_layer_routed(L, x_bf16, ids, w, n_tok, k, nthreads, out);
    if (rc == 0) {
        if (ids_out)
            memcpy(ids_out, ids, sizeof(int32_t) * (size_t)(n_tok * k));
        if (w_out)
            memcpy(w_out, w, sizeof(double) * (size_t)(n_tok * k));
    }
    free(ids);
    free(w);
    return rc;
}

/* The dense SwiGLU FFN [C34] for n_tok tokens.  Weights are given unsliced:
 * gate [I, H], up [I, H], down [H, I] in weight_format 0 (MXFP4 codes and
 * E8M0 scales), 1 (BF16 bits) or 2 (group-32 INT4 codes, FP16 scales, zero
 * points or NULL).  With n_slices == 0 the FFN is evaluated as one block;
 * with n_slices > 0 it is evaluated as the sum over n_slices all-active slices
 * of width I / n_slices, each with unit weight (Eq. 2).  out [n_tok, H] double.
 * Returns 0, -1 (a scale the format rejects), -3 (bad args). */
int oracle_dense_ffn(int weight_format, const void *g_codes, const void *g_scales, const uint8_t *g_zeros,
                     const void *u_codes, const void *u_scales, const uint8_t *u_zeros, const void *d_codes,
                     const void *d_scales, const uint8_t *d_zeros, int H, int I, int n_slices,
                     const uint16_t *x_bf16, int64_t n_tok, int nthreads, double *out)
{
    if (H % 32 || I % 32)
        return -3;
    int ns = n_slices > 0 ? n_slices : 1;
    if (I % ns || (I / ns) % 32)
        return -3;
    const int Is = I / ns;
    int rc = 0;
    /* gate and up stacked as one [2I, H] block so a slice's gate and up rows
     * sit at rows [j*Is, (j+1)*Is) and I + [j*Is, (j+1)*Is). */
    float *Wgu = (float *)malloc(sizeof(float) * (size_t)2 * I * H);
    float *Wd = (float *)malloc(sizeof(float) * (size_t)H * I);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n_tok * H + 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)(n_tok * H + 1));
    rc = decode_matrix(weight_format, g_codes, g_scales, g_zeros, I, H, Wgu);
    if (rc == 0)
        rc = decode_matrix(weight_format, u_codes, u_scales, u_zeros, I, H, Wgu + (int64_t)I * H);
    if (rc == 0)
        rc = decode_matrix(weight_format, d_codes, d_scales, d_zeros, H, I, Wd);
    if (rc == 0) {
        for (int64_t i = 0; i < n_tok * H; ++i) {
            uint32_t u = (uint32_t)x_bf16[i] << 16;
            float f;
            memcpy(&f, &u, 4);
            x[i] = (double)f;
            out[i] = 0.0;
        }
        for (int j = 0; j < ns; ++j) {
            /* slice j: gate/up rows [j*Is, (j+1)*Is), down columns likewise */
            const float *Wg_j = Wgu + (int64_t)j * Is * H;
            const float *Wu_j = Wgu + (int64_t)I * H + (int64_t)j * Is * H;
            const float *Wd_j = Wd + (int64_t)j * Is;
            for (int64_t t = 0; t < n_tok; ++t) {
                oracle_swiglu_ffn(Wg_j, Wu_j, H, Wd_j, I, H, Is, x + t * H, y + t * H);
                for (int m = 0; m < H; ++m)
                    out[t * H + m] += y[t * H + m];
            }
        }
    }
    (void)nthreads;
    free(Wgu);
    free(Wd);
    free(x);
    free(y);
    return rc;
}
