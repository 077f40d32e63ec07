/*
 * moe_oracle.c -- plain, slow CPU oracle of the decode-time MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library: every number format, the alignment and the expert FFN are
 * written out here again from their definitions.
 *
 * Everything floating point is computed in double.  Each function names the
 * passage it follows:
 *   [ALIGN]  "nbxtensor/ops/moe_align.py" (page 1): module docstring (worst-case
 *            sizing, deterministic rank), moe_align_stage1_kernel (counts,
 *            block padding, exclusive offsets, total), moe_align_stage2_kernel
 *            (sentinel fill, block -> expert map), moe_align_stage3_kernel
 *            (rank = number of earlier slots with the same expert; scatter).
 *   [SORT]   "metrale_model_layers/layers/ops/fp8_moe_grouped.rs" (page 3):
 *            moe_fp8_grouped_sort (token_to_perm, ascending active-expert
 *            list and its count), fp8_grouped_active_cap (cap = min(n, E)),
 *            moe_expert_gate_up_act_fp8_grouped (SiLU(gate) * up product per
 *            sorted position), moe_expert_down_act_fp8_grouped (down over the
 *            product), moe_weighted_sum_blend_fp8_grouped (blend through
 *            token_to_perm, shared-expert output added).
 *   [LAYER]  "metrale_model_layers/layers/moe/forward_nvfp4_grouped_decode.rs"
 *            (page 2): forward_nvfp4_grouped_decode (route -> sort -> gate+up
 *            -> down -> blend; NVFP4 tables = packed codes, per-16 scales and
 *            one fp32 global scale per projection).
 *   [ROUTER] the same page: the router matrix-vector product named in
 *            nvfp4_grouped_decode_ok (router_gemv_batchm) ahead of grouped_route.
 *   [GATE]   the same page and moe_weighted_sum_blend_fp8_grouped of page 3:
 *            the blend takes the layer input and shared_expert_gate.weight
 *            (NULL: ungated shared expert).
 *   [VEC]    "nbxtensor/ops/moe_decode_vec.py" (page 1): the SwiGLU epilogue
 *            h = silu(g) * u in pure fp32 (here: double), fixed-order
 *            combine of the router-weighted expert outputs.
 * Readings where the pages are silent are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* OCP 8-bit float E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); no infinities; S.1111.111
 * is NaN.  The pages name the format only ("FP8 E4M3"). */
double oracle_e4m3_value(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP 4-bit float E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent
 * field 0 is subnormal (m * 0.5).  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_value(uint8_t nibble)
{
    int s = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 3;
    int m = nibble & 1;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* Round a double to bfloat16 (8-bit exponent, 7 stored mantissa bits), nearest,
 * ties to even, in one rounding step.  Returns the 16-bit pattern. */
uint16_t oracle_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int ex;
    frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) -> a = 1.x * 2^(ex-1) */
    int E = ex - 1;
    if (E < -126)
        E = -126;           /* subnormal range: fixed spacing 2^-133 */
    double q = ldexp(1.0, E - 7);       /* spacing of bf16 values near a */
    double r = nearbyint(a / q);         /* default mode: nearest, ties to even */
    double res = r * q;
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (res > ldexp(2.0 - ldexp(1.0, -7), 127))
        return sign | 0x7F80;
    float f = (float)res;   /* exact: res has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

double oracle_bf16_value(uint16_t bits)
{
    uint32_t b = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Router logits: the matrix-vector product ahead of the top-k              */
/* ------------------------------------------------------------------------ */

/* logits[t][e] = sum_c x[t][c] * W[e][c], in double, for M rows of bf16 x
 * [M][H] and bf16 router weights W [E][H] (row-major).  The pages name the
 * kernel (forward_nvfp4_grouped_decode: nvfp4_grouped_decode_ok requires
 * router_gemv_batchm; grouped_route takes the hidden input) but print no
 * arithmetic; this is the plainest reading of a router that maps hidden
 * states to one logit per expert: no bias, no normalisation. */
void oracle_router_logits(const uint16_t *x, const uint16_t *W, int M, int H, int E,
                          double *logits)
{
    for (int t = 0; t < M; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += oracle_bf16_value(x[(size_t)t * H + c]) *
                       oracle_bf16_value(W[(size_t)e * H + c]);
            logits[(size_t)t * E + e] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Routing: softmax over the experts, top-k, renormalised                   */
/* ------------------------------------------------------------------------ */

/* Per row t: p = softmax(logits[t, :]) over all E experts; the k experts with
 * the largest logits are selected (equal logits: the lower expert id first);
 * the selected probabilities are renormalised to sum to 1.  The pages run a
 * per-row top-k softmax router (forward_nvfp4_grouped_decode: grouped_route
 * with GroupedRouting::PerRow, kernel moe_topk_softmax_rows); the
 * precise order of operations is the workload's statement ("softmax then
 * top-k renormalised").  ids[t*k + j] lists the selection in descending
 * logit order.  Logits must be finite. */
void oracle_topk_softmax(const float *logits, int M, int E, int k,
                         int32_t *ids, double *w)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int t = 0; t < M; ++t) {
        const float *l = logits + (size_t)t * E;
        double mx = -INFINITY;
        for (int e = 0; e < E; ++e)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < E; ++e)
            p[e] /= z;
        memset(taken, 0, (size_t)E);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])   /* strict: ties keep the lower id */
                    best = e;
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
            sel += p[best];
        }
        for (int j = 0; j < k; ++j)
            w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / sel;
    }
    free(p);
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* Alignment                                                                */
/* ------------------------------------------------------------------------ */

/* Worst-case sizes [ALIGN, module docstring; SORT, fp8_grouped_active_cap]:
 *   max_total  = min(n*BS, n + E*(BS-1)) rounded up to a multiple of BS
 *   max_blocks = max_total / BS
 *   cap        = min(n, E)                                                  */
void oracle_align_sizes(int n, int E, int BS, int64_t *max_total,
                        int64_t *max_blocks, int64_t *cap)
{
    int64_t a = (int64_t)n * BS;
    int64_t b = (int64_t)n + (int64_t)E * (BS - 1);
    int64_t m = a < b ? a : b;
    int64_t mt = (m + BS - 1) / BS * BS;
    *max_total = mt;
    *max_blocks = mt / BS;
    *cap = n < E ? n : E;
}

/* The alignment tables of n flat slots ids[0..n) (slot i = token*top_k + j).
 * Follows [ALIGN] stage by stage:
 *  stage 1: counts[e] = #{i : ids[i] == e}; padded[e] = ceil(counts/BS)*BS;
 *           offsets[e] = sum_{f<e} padded[f]; total = sum padded.
 *  stage 2: sorted_token_ids[p] = n (sentinel) for every p < max_total;
 *           sorted_expert_ids[b] = the e with offsets[e] <= b*BS <
 *           offsets[e]+padded[e], else -1 (blocks at or past the total).
 *  stage 3: rank(i) = #{j < i : ids[j] == ids[i]};
 *           sorted_token_ids[offsets[ids[i]] + rank(i)] = i.
 * plus [SORT]: token_to_perm[i] = the position slot i went to;
 * active_experts[0..count) = the experts with counts > 0, ascending.
 * Readings: offsets has E+1 entries, offsets[E] = total; ids outside [0, E)
 * are skipped everywhere (token_to_perm = -1) and counted in the return
 * value; the active list's tail up to cap is -1.  Rank is computed with one
 * running counter per expert, visiting slots in increasing i, which is the
 * count of earlier equal slots by definition. */
int oracle_align(const int64_t *ids, int n, int E, int BS,
                 int32_t *sorted_token_ids, int32_t *sorted_expert_ids,
                 int32_t *expert_offsets, int32_t *token_to_perm,
                 int32_t *active_experts, int32_t *active_count,
                 int32_t *num_tokens_post_padded, int32_t *counts_out)
{
    int64_t max_total, max_blocks, cap;
    oracle_align_sizes(n, E, BS, &max_total, &max_blocks, &cap);
    int64_t *counts = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t *padded = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t *seen = (int64_t *)calloc((size_t)E + 1, sizeof(int64_t));
    int bad = 0;

    /* stage 1 */
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) {
            ++bad;
            continue;
        }
        counts[ids[i]] += 1;
    }
    int64_t total = 0;
    for (int e = 0; e < E; ++e) {
        padded[e] = (counts[e] + BS - 1) / BS * BS;
        expert_offsets[e] = (int32_t)total;
        total += padded[e];
    }
    expert_offsets[E] = (int32_t)total;
    *num_tokens_post_padded = (int32_t)total;

    /* stage 2 */
    for (int64_t p = 0; p < max_total; ++p)
        sorted_token_ids[p] = n;
    for (int64_t b = 0; b < max_blocks; ++b) {
        int64_t start = b * BS;
        int32_t owner = -1;
        for (int e = 0; e < E; ++e)
            if (expert_offsets[e] <= start && start < expert_offsets[e] + padded[e])
                owner = e;
        sorted_expert_ids[b] = owner;
    }

    /* stage 3 */
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) {
            token_to_perm[i] = -1;
            continue;
        }
        int64_t e = ids[i];
        int64_t pos = expert_offsets[e] + seen[e];
        seen[e] += 1;
        sorted_token_ids[pos] = i;
        token_to_perm[i] = (int32_t)pos;
    }

    /* active-expert list */
    int32_t count = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0)
            active_experts[count++] = e;
    for (int64_t a = count; a < cap; ++a)
        active_experts[a] = -1;
    *active_count = count;
    if (counts_out)
        for (int e = 0; e < E; ++e)
            counts_out[e] = (int32_t)counts[e];
    free(counts);
    free(padded);
    free(seen);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Expert weights                                                           */
/* ------------------------------------------------------------------------ */

/* One projection of E experts, weights [E][rows][cols] row-major (rows =
 * output features, cols = input features, the "row-major decode layout").
 *  fmt 1 (FP8, 128x128 blocks): codes uint8 E4M3 [E][rows][cols];
 *        scale fp32 [E][ceil(rows/128)][ceil(cols/128)];
 *        w[o][i] = e4m3(code) * scale[o/128][i/128].
 *  fmt 2 (NVFP4, per-16 groups): codes uint8 [E][rows][cols/2], element i in
 *        the low nibble when i is even, the high nibble when odd;
 *        scale uint8 E4M3 [E][rows][cols/16]; global fp32 [E];
 *        w[o][i] = e2m1(code) * e4m3(scale[o][i/16]) * global.
 * The pages give the FP8 block and the NVFP4 tables' names (packed_ptrs,
 * scale_ptrs, scale2_vals) but not their layout or whether the scale
 * multiplies or divides: the reading here is multiply, row-major. */
typedef struct {
    int fmt;
    int rows, cols;
    const uint8_t *codes;
    const void *scale;
    const float *global;
} oracle_proj;

void oracle_dequant_proj(const oracle_proj *P, int e, double *out)
{
    int R = P->rows, C = P->cols;
    if (P->fmt == 1) {
        int sr = (R + 127) / 128, sc = (C + 127) / 128;
        const uint8_t *q = P->codes + (size_t)e * R * C;
        const float *s = (const float *)P->scale + (size_t)e * sr * sc;
        for (int o = 0; o < R; ++o)
            for (int i = 0; i < C; ++i)
                out[(size_t)o * C + i] = oracle_e4m3_value(q[(size_t)o * C + i])
                                         * (double)s[(o / 128) * sc + i / 128];
    } else {
        const uint8_t *q = P->codes + (size_t)e * R * (C / 2);
        const uint8_t *s = (const uint8_t *)P->scale + (size_t)e * R * (C / 16);
        double g = (double)P->global[e];
        for (int o = 0; o < R; ++o)
            for (int i = 0; i < C; ++i) {
                uint8_t byte = q[(size_t)o * (C / 2) + i / 2];
                uint8_t nib = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
                out[(size_t)o * C + i] = oracle_e2m1_value(nib)
                                         * oracle_e4m3_value(s[(size_t)o * (C / 16) + i / 16]) * g;
            }
    }
}

/* An expert set: gate and up are [I][H], down is [H][I]. */
typedef struct {
    int E, H, I;
    oracle_proj gate, up, down;
} oracle_experts;

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* [SORT moe_expert_gate_up_act_fp8_grouped; VEC SwiGLU epilogue]
 * For every active expert e and every real slot s at a sorted position p of
 * its run (sorted_token_ids[p] != n), with token t = s / top_k:
 *     g = Wg[e] x[t],  u = Wu[e] x[t],  h[p][o] = silu(g[o]) * u[o].
 * With a shared expert (may be NULL): h_sh[t][o] the same for every token.
 * x is bf16 [M][H]; h is [max_total][I] by sorted position; untouched rows
 * (padding) are left as they are. */
void oracle_grouped_gate_up(const oracle_experts *X, const oracle_experts *S,
                            const uint16_t *x, int M, int top_k,
                            const int32_t *sorted_token_ids, const int32_t *expert_offsets,
                            const int32_t *active_experts, int active_count,
                            double *h, double *h_sh)
{
    int H = X->H, I = X->I, n = M * top_k;
    double *xd = (double *)malloc(sizeof(double) * (size_t)M * H);
    for (size_t i = 0; i < (size_t)M * H; ++i)
        xd[i] = oracle_bf16_value(x[i]);
    double *wg = (double *)malloc(sizeof(double) * (size_t)I * H);
    double *wu = (double *)malloc(sizeof(double) * (size_t)I * H);
    for (int a = 0; a < active_count; ++a) {
        int e = active_experts[a];
        oracle_dequant_proj(&X->gate, e, wg);
        oracle_dequant_proj(&X->up, e, wu);
        for (int p = expert_offsets[e]; p < expert_offsets[e + 1]; ++p) {
            int s = sorted_token_ids[p];
            if (s >= n)
                continue;                       /* sentinel: padding */
            const double *xt = xd + (size_t)(s / top_k) * H;
            for (int o = 0; o < I; ++o) {
                double g = 0.0, u = 0.0;
                for (int i = 0; i < H; ++i) {
                    g += wg[(size_t)o * H + i] * xt[i];
                    u += wu[(size_t)o * H + i] * xt[i];
                }
                h[(size_t)p * I + o] = silu(g) * u;
            }
        }
    }
    free(wg);
    free(wu);
    if (S) {
        int Is = S->I;
        double *sg = (double *)malloc(sizeof(double) * (size_t)Is * H);
        double *su = (double *)malloc(sizeof(double) * (size_t)Is * H);
        oracle_dequant_proj(&S->gate, 0, sg);
        oracle_dequant_proj(&S->up, 0, su);
        for (int t = 0; t < M; ++t)
            for (int o = 0; o < Is; ++o) {
                double g = 0.0, u = 0.0;
                for (int i = 0; i < H; ++i) {
                    g += sg[(size_t)o * H + i] * xd[(size_t)t * H + i];
                    u += su[(size_t)o * H + i] * xd[(size_t)t * H + i];
                }
                h_sh[(size_t)t * Is + o] = silu(g) * u;
            }
        free(sg);
        free(su);
    }
    free(xd);
}

/* [SORT moe_expert_down_act_fp8_grouped] y[p][c] = sum_i Wd[e][c][i] h[p][i]
 * for every real position p of every active expert e; shared: y_sh[t]. */
void oracle_grouped_down(const oracle_experts *X, const oracle_experts *S,
                         const double *h, const double *h_sh, int M, int top_k,
                         const int32_t *sorted_token_ids, const int32_t *expert_offsets,
                         const int32_t *active_experts, int active_count,
                         double *y, double *y_sh)
{
    int H = X->H, I = X->I, n = M * top_k;
    double *wd = (double *)malloc(sizeof(double) * (size_t)H * I);
    for (int a = 0; a < active_count; ++a) {
        int e = active_experts[a];
        oracle_dequant_proj(&X->down, e, wd);
        for (int p = expert_offsets[e]; p < expert_offsets[e + 1]; ++p) {
            if (sorted_token_ids[p] >= n)
                continue;
            for (int c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int i = 0; i < I; ++i)
                    acc += wd[(size_t)c * I + i] * h[(size_t)p * I + i];
                y[(size_t)p * H + c] = acc;
            }
        }
    }
    free(wd);
    if (S) {
        int Is = S->I;
        double *sd = (double *)malloc(sizeof(double) * (size_t)H * Is);
        oracle_dequant_proj(&S->down, 0, sd);
        for (int t = 0; t < M; ++t)
            for (int c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int i = 0; i < Is; ++i)
                    acc += sd[(size_t)c * Is + i] * h_sh[(size_t)t * Is + i];
                y_sh[(size_t)t * H + c] = acc;
            }
        free(sd);
    }
}

/* [GATE] The shared expert's gate per token.  The pages pass the layer
 * input and shared_expert_gate.weight to the blend and print no formula; the
 * plain reading of a one-output gate layer: g[t] = sigmoid(sum_c x[t][c] *
 * gate_w[c]) with bf16 x [M][H] and bf16 gate_w [H], no bias,
 * sigmoid(z) = 1 / (1 + exp(-z)). */
void oracle_shared_gate(const uint16_t *x, const uint16_t *gate_w, int M, int H, double *g)
{
    for (int t = 0; t < M; ++t) {
        double z = 0.0;
        for (int c = 0; c < H; ++c)
            z += oracle_bf16_value(x[(size_t)t * H + c]) * oracle_bf16_value(gate_w[c]);
        g[t] = 1.0 / (1.0 + exp(-z));
    }
}

/* [SORT moe_weighted_sum_blend_fp8_grouped; VEC fixed-order combine]
 * out[t][c] = bf16( sum_{j=0..k-1} w[t][j] * y[token_to_perm[t*k+j]][c]
 *                   + gate[t] * y_sh[t][c] ), j in increasing order, one
 * rounding to bf16 at the end.  Slots with token_to_perm = -1 (an
 * out-of-range id) contribute nothing.  y_sh may be NULL (no shared expert);
 * gate may be NULL (an ungated shared expert: gate[t] = 1).  out_d keeps the
 * unrounded double. */
void oracle_blend(const double *y, const double *w, const int32_t *token_to_perm,
                  const double *y_sh, const double *gate, int M, int top_k, int H,
                  double *out_d, uint16_t *out_bf16)
{
    for (int t = 0; t < M; ++t)
        for (int c = 0; c < H; ++c) {
            double acc = 0.0;
            for (int j = 0; j < top_k; ++j) {
                int32_t p = token_to_perm[(size_t)t * top_k + j];
                if (p < 0)
                    continue;
                acc += w[(size_t)t * top_k + j] * y[(size_t)p * H + c];
            }
            if (y_sh)
                acc += (gate ? gate[t] : 1.0) * y_sh[(size_t)t * H + c];
            if (out_d)
                out_d[(size_t)t * H + c] = acc;
            if (out_bf16)
                out_bf16[(size_t)t * H + c] = oracle_bf16_rne(acc);
        }
}

/* [LAYER forward_nvfp4_grouped_decode] the whole layer: route (when logits
 * are given; else the caller's ids and weights), align, gate+up, down,
 * blend.  shared_gate_w ([H] bf16, or NULL: ungated) gates the shared
 * expert.  Returns the number of out-of-range ids the alignment skipped. */
int oracle_moe_layer(const oracle_experts *X, const oracle_experts *S,
                     const uint16_t *shared_gate_w,
                     const uint16_t *x, int M, int top_k, int BS,
                     const float *logits, const int32_t *ids_in, const double *w_in,
                     double *out_d, uint16_t *out_bf16)
{
    int E = X->E, H = X->H, I = X->I, n = M * top_k;
    int64_t max_total, max_blocks, cap;
    oracle_align_sizes(n, E, BS, &max_total, &max_blocks, &cap);
    int32_t *ids32 = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    if (logits) {
        oracle_topk_softmax(logits, M, E, top_k, ids32, w);
    } else {
        memcpy(ids32, ids_in, sizeof(int32_t) * (size_t)n);
        memcpy(w, w_in, sizeof(double) * (size_t)n);
    }
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    for (int i = 0; i < n; ++i)
        ids[i] = ids32[i];
    int32_t *sti = (int32_t *)malloc(sizeof(int32_t) * (size_t)(max_total + 1));
    int32_t *sei = (int32_t *)malloc(sizeof(int32_t) * (size_t)(max_blocks + 1));
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *ttp = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *act = (int32_t *)malloc(sizeof(int32_t) * (size_t)(cap + 1));
    int32_t count, ntpp;
    int bad = oracle_align(ids, n, E, BS, sti, sei, off, ttp, act, &count, &ntpp, NULL);
    double *h = (double *)calloc((size_t)max_total * I + 1, sizeof(double));
    double *y = (double *)calloc((size_t)max_total * H + 1, sizeof(double));
    double *h_sh = NULL, *y_sh = NULL, *gate = NULL;
    if (S) {
        h_sh = (double *)calloc((size_t)M * S->I, sizeof(double));
        y_sh = (double *)calloc((size_t)M * H, sizeof(double));
        if (shared_gate_w) {
            gate = (double *)malloc(sizeof(double) * (size_t)M);
            oracle_shared_gate(x, shared_gate_w, M, H, gate);
        }
    }
    oracle_grouped_gate_up(X, S, x, M, top_k, sti, off, act, count, h, h_sh);
    oracle_grouped_down(X, S, h, h_sh, M, top_k, sti, off, act, count, y, y_sh);
    oracle_blend(y, w, ttp, y_sh, gate, M, top_k, H, out_d, out_bf16);
    free(ids32); free(w); free(ids); free(sti); free(sei); free(off); free(ttp);
    free(act); free(h); free(y); free(h_sh); free(y_sh); free(gate);
    return bad;
}
