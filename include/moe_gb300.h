/*
 * moe_gb300.h -- C ABI of the decode-time Mixture-of-Experts layer on GB300
 * (sm_103a): router top-k ids -> deterministic device-side token alignment ->
 * grouped FP8 / NVFP4 expert FFN (gate+up, SiLU(gate)*up, down) -> weighted
 * blend back to token order.
 *
 * Conventions shared by every entry point
 *  - All array arguments are DEVICE pointers unless stated; the caller owns
 *    every buffer (weights, inputs, outputs, workspace).  No entry point
 *    allocates, frees or synchronises.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it and is CUDA-graph
 *    capturable: every launch's grid depends only on the shape arguments, never
 *    on routing results, and nothing is read back to the host.
 *  - Return value: MOE_OK, or an error code.  Host-detected errors (a NULL
 *    pointer, a size or shape outside what is admitted) launch nothing.
 *    MOE_ECUDA means a launch failed; moe_last_cuda_error() gives the
 *    cudaError_t of the calling thread's last failure.
 *  - Device-detected errors never trap: the kernel skips the offending item
 *    and ORs a MOE_ERR_* bit into *err_word (if err_word is not NULL), which
 *    the caller reads when it chooses.
 *  - Matrices are row-major.  bf16 values are passed as their uint16 bit
 *    patterns.
 *
 * Sources.  The operations are those of three pages:
 *   "nbxtensor/ops/moe_align.py" (alignment stages 1-3 and the worst-case
 *   sizing in its module docstring), "nbxtensor/ops/moe_decode_vec.py" (SiLU
 *   product in fp32, fixed-order combine), "metrale_model_layers/layers/ops/
 *   fp8_moe_grouped.rs" (moe_fp8_grouped_sort, the grouped gate+up/down
 *   launchers, fp8_grouped_active_cap, the blend) and "metrale_model_layers/
 *   layers/moe/forward_nvfp4_grouped_decode.rs" (the layer's sequence and
 *   its shape admission).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK 0
#define MOE_EINVAL 1        /* NULL pointer, negative/zero size, bad enum */
#define MOE_EUNSUPPORTED 2  /* shape valid but not admitted by the kernels */
#define MOE_ECUDA 3         /* a CUDA runtime call or launch failed */

/* ---- device error bits, ORed into *err_word ----------------------------- */
#define MOE_ERR_BAD_ID 0x1u   /* an expert id outside [0, E): slot skipped */
#define MOE_ERR_TIMEOUT 0x2u  /* a bounded pipeline wait gave up: outputs invalid */

/* ---- formats and paths -------------------------------------------------- */
#define MOE_FMT_FP8_B128 1  /* E4M3 codes, fp32 scale per 128x128 block      */
#define MOE_FMT_NVFP4_G16 2 /* E2M1 codes, E4M3 scale per 16, fp32 global    */
/* The "nvfp4-gate-up" tier ("forward_nvfp4_grouped_decode.rs", module notes
 * and the down-projection choice in forward_nvfp4_grouped_decode): gate and
 * up in NVFP4_G16, the down projection in FP8_B128.  hidden and inter must be
 * multiples of 128. */
#define MOE_FMT_NVFP4_GATE_UP 3

#define MOE_PATH_AUTO 0     /* chosen per shape class (never per routing)    */
#define MOE_PATH_SIMT 1     /* CUDA-core kernels, in-register dequant         */
#define MOE_PATH_TC 2       /* tcgen05 tensor-core kernels (moe_decode_layer) */
#define MOE_PATH_SIMT_STAGED 3 /* moe_decode_layer only: CUDA-core kernels as the
                                  five separate launches (router, align, gate+up,
                                  down, blend) instead of the fused decode pair */

#define MOE_MAX_EXPERTS 1024      /* experts the alignment handles            */
#define MOE_MAX_SLOTS (1 << 20)   /* n = M * top_k the alignment handles      */
#define MOE_MAX_ROWS 128          /* M the expert kernels and layer admit     */
#define MOE_MAX_ROWS_TC 4096      /* M the layer admits on the tensor-core path
                                     (prefill-sized batches of FP8 experts)     */

/* One projection of all experts of a set.  Layout for `rows` x `cols`
 * (gate/up: rows = inter, cols = hidden; down: rows = hidden, cols = inter),
 * by the projection's format (the set's format, except that under
 * MOE_FMT_NVFP4_GATE_UP gate and up are NVFP4_G16 and down is FP8_B128):
 *   FP8_B128:  codes  uint8 [E][rows][cols] E4M3;
 *              scale  float [E][rows/128][cols/128], w = e4m3(code) * scale;
 *              global_scale unused (NULL).
 *   NVFP4_G16: codes  uint8 [E][rows][cols/2], element 2i in the low nibble,
 *              2i+1 in the high nibble, E2M1;
 *              scale  uint8 [E][rows][cols/16] E4M3;
 *              global_scale float [E]; w = e2m1(code) * e4m3(scale) * global.
 * Experts are packed back to back (expert e at e * one expert's size).
 * All three pointers must be 16-byte aligned (scale: 4-byte for FP8). */
typedef struct moe_proj {
    const void *codes;
    const void *scale;
    const float *global_scale;
} moe_proj;

/* An expert set: E experts with gate/up [inter][hidden] and down
 * [hidden][inter].  FP8 needs hidden % 128 == 0 and inter % 128 == 0;
 * NVFP4 needs hidden % 32 == 0 and inter % 32 == 0. */
typedef struct moe_experts {
    int fmt;          /* MOE_FMT_* */
    int num_experts;  /* E (1 for a shared expert) */
    int hidden;       /* H */
    int inter;        /* I */
    moe_proj gate, up, down;
} moe_experts;

/* The layer: routed experts (E <= MOE_MAX_EXPERTS), top_k, alignment block
 * size, an optional shared expert (NULL = none; applied to every row, may
 * have its own format and inter), and the expert-kernel path. */
typedef struct moe_layer_desc {
    int top_k;
    int block_size;
    int path;                    /* MOE_PATH_* */
    moe_experts routed;
    const moe_experts *shared;   /* host pointer to a descriptor, or NULL */
    /* The shared expert's gate weight [hidden] bf16 bits on the device,
     * 16-byte aligned, or NULL (ungated); only with a shared expert.  The
     * blend scales the shared term by sigmoid(x[t] . shared_gate). */
    const uint16_t *shared_gate;
    /* Router weights [num_experts][hidden] bf16 bits on the device, 16-byte
     * aligned, or NULL.  With them, a moe_decode_layer call given neither
     * router logits nor top-k ids computes the logits from x itself
     * (moe_router_logits) into the workspace's router_logits region. */
    const uint16_t *router_weight;
} moe_layer_desc;

/* ---- library information ------------------------------------------------ */
const char *moe_version(void);
const char *moe_status_string(int status);
int moe_last_cuda_error(void);

/* ---- alignment ---------------------------------------------------------- */

/* Host only.  Worst-case table sizes of n = M*top_k slots over E experts with
 * block size BS ("nbxtensor/ops/moe_align.py", module docstring;
 * "fp8_moe_grouped.rs", fp8_grouped_active_cap):
 *   *max_total  = min(n*BS, n + E*(BS-1)) rounded up to a multiple of BS,
 *   *max_blocks = *max_total / BS,   *cap = min(n, E).
 * Returns MOE_EINVAL for n < 0, E < 1, BS < 1 or NULL outputs;
 * MOE_EUNSUPPORTED for n > MOE_MAX_SLOTS or a max_total beyond int32. */
int moe_align_sizes(int n, int num_experts, int block_size,
                    int *max_total, int *max_blocks, int *cap);

/* Device-side token alignment of n flat slots (slot i = token*top_k + j),
 * one launch, no atomics on the tables: results are bit-deterministic.
 * ("nbxtensor/ops/moe_align.py": stage 1 counts / block padding / exclusive
 * offsets / total, stage 2 sentinel fill and block->expert map, stage 3
 * rank = number of earlier slots with the same expert and scatter;
 * "fp8_moe_grouped.rs", moe_fp8_grouped_sort: token_to_perm and the active
 * list.)
 *   topk_ids               [n] int32, or int64 if ids_is_int64
 *   sorted_token_ids  out  [max_total] int32: slot index at its sorted
 *                          position; padding and the tail hold n (sentinel)
 *   sorted_expert_ids out  [max_blocks] int32: expert owning block b, -1 for
 *                          blocks at or past the total
 *   expert_offsets    out  [E+1] int32: exclusive block-padded offsets,
 *                          expert_offsets[E] = total
 *   token_to_perm     out  [n] int32: sorted position of slot i (-1 if its id
 *                          is out of range)
 *   active_experts    out  [cap] int32: experts with >= 1 slot, ascending,
 *                          then -1 up to cap
 *   active_count      out  [1] int32
 *   num_tokens_post_padded out [1] int32: the total (= expert_offsets[E])
 *   err_word               [1] uint32 or NULL: MOE_ERR_BAD_ID is ORed in
 *                          when an id lies outside [0, E); that slot is
 *                          skipped everywhere.
 * n == 0 is valid (writes the offsets, counts and total as zero).
 * Errors: MOE_EINVAL (NULL table pointer, n < 0, E < 1, BS < 1),
 * MOE_EUNSUPPORTED (E > MOE_MAX_EXPERTS, n > MOE_MAX_SLOTS). */
int moe_align(const void *topk_ids, int ids_is_int64, int n, int num_experts,
              int block_size, int32_t *sorted_token_ids,
              int32_t *sorted_expert_ids, int32_t *expert_offsets,
              int32_t *token_to_perm, int32_t *active_experts,
              int32_t *active_count, int32_t *num_tokens_post_padded,
              uint32_t *err_word, void *stream);

/* ---- routing ------------------------------------------------------------ */

/* Per-row router: for each of M rows of fp32 logits [M][E] select the top_k
 * largest logits (equal logits: the lower expert id first) and write their
 * ids in descending order and their softmax weights renormalised over the
 * selection (= softmax over all E, top-k, renormalised), fp32
 * ("forward_nvfp4_grouped_decode.rs": grouped_route, GroupedRouting::PerRow;
 * the top-k softmax kernel moe_topk_softmax_rows).  Logits must be finite.
 *   topk_ids out [M][top_k] int32, topk_w out [M][top_k] float.
 * Errors: MOE_EINVAL (NULL, M < 1, top_k < 1, top_k > E),
 * MOE_EUNSUPPORTED (E > MOE_MAX_EXPERTS, top_k > 32). */
int moe_topk_softmax(const float *logits, int M, int num_experts, int top_k,
                     int32_t *topk_ids, float *topk_w, void *stream);

/* Router logits, the matrix-vector product ahead of the top-k
 * ("forward_nvfp4_grouped_decode.rs": the router_gemv_batchm kernel that
 * nvfp4_grouped_decode_ok requires; grouped_route takes the hidden input).
 * The pages print no arithmetic; the plain reading, with no bias:
 *   logits[t][e] = sum_c x[t][c] * router_weight[e][c]
 * accumulated in fp32 in an order that depends on hidden alone: run to run,
 * and for every M, a row's logits are the same bits.
 *   x [M][hidden] bf16 bits; router_weight [num_experts][hidden] bf16 bits,
 *   both 16-byte aligned; logits out [M][num_experts] float.
 * Errors: MOE_EINVAL (NULL, M, hidden or num_experts < 1), MOE_EUNSUPPORTED
 * (hidden not a multiple of 8, x or weights misaligned). */
int moe_router_logits(const uint16_t *x, const uint16_t *router_weight, int M,
                      int hidden, int num_experts, float *logits, void *stream);

/* ---- grouped expert FFN ------------------------------------------------- */

/* Grouped gate+up and SiLU ("fp8_moe_grouped.rs",
 * moe_expert_gate_up_act_fp8_grouped; the SwiGLU epilogue of
 * "moe_decode_vec.py").  For every active expert e = active_experts[a]
 * (a < *active_count) and every real position p of its run
 * (expert_offsets[e] <= p < expert_offsets[e+1], sorted_token_ids[p] < n),
 * token t = sorted_token_ids[p] / top_k:
 *     h[p][o] = silu(g) * u,  g = Wg[e][o] . x[t],  u = Wu[e][o] . x[t]
 * in fp32 (no intermediate bf16 rounding).  Each weight row is read once per
 * pass for all rows routed to its expert.  With a shared expert S (host
 * descriptor, may be NULL): h_shared[t][o] = the same with S, for every t.
 *   x        [M][H] bf16 bits;  the tables as written by moe_align for
 *            n = M*top_k slots and E = routed->num_experts
 *   h    out [max_total][I] float, rows by sorted position (padding rows
 *            untouched)
 *   h_shared out [M][S->inter] float (NULL iff shared is NULL)
 *   path     MOE_PATH_AUTO / _SIMT / _TC; the grid is a function of
 *            (M, top_k, E, H, I, path).
 * Errors: MOE_EINVAL (NULL, M < 1 or > MOE_MAX_ROWS, bad fmt/path),
 * MOE_EUNSUPPORTED (shape not admitted; MOE_PATH_TC, which only
 * moe_decode_layer serves: its activation terms live in the layer workspace). */
int moe_grouped_gate_up(const moe_experts *routed, const moe_experts *shared,
                        const uint16_t *x, int M, int top_k,
                        const int32_t *expert_offsets,
                        const int32_t *sorted_token_ids,
                        const int32_t *active_experts,
                        const int32_t *active_count, float *h,
                        float *h_shared, int path, void *stream);

/* Grouped down projection over the SiLU product ("fp8_moe_grouped.rs",
 * moe_expert_down_act_fp8_grouped): y[p][c] = Wd[e][c] . h[p] in fp32 for
 * every real position p of every active expert e; y_shared[t] = WdS .
 * h_shared[t] for every token.  Rows of h and y are sorted positions.
 *   h [max_total][I], h_shared [M][S->inter], y out [max_total][H],
 *   y_shared out [M][H] (NULL iff shared is NULL).
 * Errors as moe_grouped_gate_up. */
int moe_grouped_down(const moe_experts *routed, const moe_experts *shared,
                     const float *h, const float *h_shared, int M, int top_k,
                     const int32_t *expert_offsets,
                     const int32_t *sorted_token_ids,
                     const int32_t *active_experts,
                     const int32_t *active_count, float *y, float *y_shared,
                     int path, void *stream);

/* Weighted blend back to token order in a fixed order ("fp8_moe_grouped.rs",
 * moe_weighted_sum_blend_fp8_grouped; fixed-order combine of
 * "moe_decode_vec.py"):
 *   out[t][c] = bf16_rn( sum_{j=0..top_k-1} topk_w[t][j] *
 *                        y[token_to_perm[t*top_k+j]][c]  + g[t] * y_shared[t][c] )
 * accumulated in fp32, j ascending, then the shared term; slots with
 * token_to_perm = -1 contribute nothing.  y_shared may be NULL.  The blend
 * takes the layer input and the shared expert's gate weight, as the pages'
 * blend does: with shared_gate ([H] bf16, 16-byte aligned) the shared term
 * is gated, g[t] = sigmoid(x[t] . shared_gate) in fp32 (the pages print no
 * formula: the plain reading of a one-output gate layer, no bias); with
 * shared_gate NULL it is added as it is (x may then be NULL).
 *   x [M][H] bf16 bits; out [M][H] bf16 bits.
 * Errors: MOE_EINVAL (NULL, M < 1, top_k < 1, H < 1, a gate without
 * y_shared or x), MOE_EUNSUPPORTED (H % 4, misaligned; gated: H % 8). */
int moe_blend(const float *y, const float *topk_w, const int32_t *token_to_perm,
              const float *y_shared, const uint16_t *x, const uint16_t *shared_gate,
              uint16_t *out, int M, int top_k, int hidden, void *stream);

/* ---- the layer ---------------------------------------------------------- */

/* Where moe_decode_layer keeps each intermediate inside its workspace, as
 * byte offsets from the workspace base, for M rows (host only). */
typedef struct moe_workspace_view {
    size_t topk_ids, topk_w;                       /* [M*k] int32, float */
    size_t sorted_token_ids, sorted_expert_ids;    /* [max_total], [max_blocks] */
    size_t expert_offsets, token_to_perm;          /* [E+1], [M*k] */
    size_t active_experts, active_count;           /* [cap], [1] */
    size_t num_tokens_post_padded;                 /* [1] */
    size_t h, h_shared, y, y_shared;               /* float tables */
    size_t blend_counters;                         /* internal: [1] uint64 grid-barrier count,
                                                      always at offset 0 */
    size_t router_logits;                          /* [M][E] float: the logits of a call that
                                                      computed them from x (else unwritten) */
    size_t shared_gate;                            /* [M] float: the shared expert's gates
                                                      (fused path, gated layers; else unwritten) */
    /* tensor-core paths only (all 0 on the CUDA-core path): the activation
     * terms they multiply, with power-of-two scales.  FP8 experts: E4M3
     * planes, x = (t0 + t1) * x_scale[p] per sorted row [2][max_total][H] u8
     * and [max_total] float; h = (t0 + t1 + t2) * h_scale[p][c/128]
     * [3][max_total][I] u8 and [max_total][I/128] float.  NVFP4 experts (M <=
     * 32): f16 planes, h = (hi + lo) * h_scale[p][c/128] [2][max_total][I]
     * f16 (then the FP8 shared expert's [2][32][Is] by token, and after the
     * [max_total][I/128] scales its [32][Is/128]), and x by token: tc_x_terms holds [H/128][2][NT][64] f16 (k block,
     * 64-wide half, token, 64 k values; NT = 16 for M <= 16, else 32), x =
     * term * tc_x_scale[t] ([32] float).  The per-token tables are written
     * by extra CTAs of the alignment launch.  Then internal int32 counters
     * (tc_done: [E] per active-list index, the item counter), which every
     * call leaves at zero.  tc_done is
     * always at offset 256 and is kept there for every M whenever the layer
     * runs a tensor-core kernel at some M (also at M the CUDA cores take):
     * the counters that persist between calls sit where M does not move
     * them, so one workspace serves every M up to the one it was sized for. */
    size_t tc_x_terms, tc_x_scale, tc_h_terms, tc_h_scale, tc_done;
    size_t total_bytes;
    int max_total, max_blocks, cap;
    /* tensor-core path only (else 0): the active table the alignment launch
     * writes for it, [cap] x {run offset, expert, slot count, 0} int32.  For
     * M <= 16 the x terms are kept by token instead of by sorted row: the
     * tc_x_terms region holds [H/128][2][16][128] u8 (k block, term, token,
     * 128 k values) and tc_x_scale [16] float. */
    size_t tc_items;
} moe_workspace_view;

/* Host only.  Workspace bytes moe_decode_layer needs for any M <= max_M
 * (the largest layout over 1..max_M; 0 if the descriptor is invalid).  One
 * workspace of this size serves calls at any M <= max_M, in any order. */
size_t moe_decode_layer_workspace_bytes(const moe_layer_desc *layer, int max_M);

/* Host only.  The workspace layout for M rows.  Returns MOE_EINVAL /
 * MOE_EUNSUPPORTED as moe_decode_layer would. */
int moe_decode_layer_workspace_view(const moe_layer_desc *layer, int M,
                                    moe_workspace_view *view);

/* Host only.  The number of kernels moe_decode_layer enqueues for M rows
 * (1 on the fused decode path; 3 with router logits, 2 with given ids on the
 * tensor-core paths; otherwise 5 and 4), or -1 if the call would be
 * rejected.  with_logits: 0 ids given, 1 logits given, 2 logits computed from
 * x and the layer's router_weight (one launch more than 1). */
int moe_decode_layer_launches(const moe_layer_desc *layer, int M, int with_logits);

/* The decode MoE layer of M rows ("forward_nvfp4_grouped_decode.rs",
 * forward_nvfp4_grouped_decode): route (when router_logits is not NULL:
 * moe_topk_softmax; when both router_logits and topk_ids are NULL and the
 * layer has router_weight: moe_router_logits of x into the workspace, then
 * moe_topk_softmax -- grouped_route's hidden input; otherwise topk_ids [M][k]
 * int32 and topk_w [M][k] float are taken as given), moe_align,
 * moe_grouped_gate_up, moe_grouped_down, moe_blend, all enqueued on `stream`
 * with no host read.
 * On the CUDA-core path, when M*top_k <= 256, M <= 32, and hidden, inter and
 * the shared inter are multiples of 128 in [256, 2048] (NVFP4: of 256), the
 * same results come from one cooperative persistent kernel (gate+up, a grid
 * barrier, down, a grid barrier, the blend) instead of five launches; every
 * table and intermediate is still written to the workspace.  MOE_PATH_SIMT_STAGED
 * forces the five.
 * On the tensor-core path (MOE_PATH_TC, and MOE_PATH_AUTO whenever the routed
 * experts are FP8 with hidden a multiple of 256 up to 8192, inter a multiple
 * of 256 up to 4096 and there is no shared expert; MOE_PATH_SIMT keeps such a
 * layer on the CUDA cores) gate+up, down and the blend run as one cooperative
 * persistent kernel of tcgen05 MMAs after the alignment ("fp8_moe_grouped.rs",
 * the tensor-core twins of the grouped launchers): E4M3 weight codes times
 * exact E4M3 splits of x and h, each 128-wide k block promoted to fp32 times
 * its block scale.  NVFP4 routed experts (and the nvfp4-gate-up tier, its
 * FP8 down projection decoded like the shared expert) with M <= 32, hidden
 * and inter multiples of 256 (hidden up to 8192, inter up to 4096) run the
 * NVFP4 twin
 * ("forward_nvfp4_grouped_decode.rs", the NVFP4 grouped launchers): each
 * E2M1 code times its E4M3 scale decoded exactly to f16 into tensor memory,
 * tcgen05 kind::f16 MMAs against an f16 x table by token and f16 hi/lo
 * splits of h, the fp32 globals applied once per item; an FP8 shared expert
 * (inter a multiple of 128 up to 4096) runs in the same kernel, its E4M3
 * codes decoded to f16 and its block scale applied per k block.  Either kernel's h and y are the same
 * quantities as on the CUDA-core path, within the layer tolerance.
 *   x [M][H] bf16 bits; out [M][H] bf16 bits;
 *   workspace: device, >= moe_decode_layer_workspace_bytes(layer, M) bytes,
 *   256-byte aligned, used only by this call (its intermediates can be read
 *   back through moe_decode_layer_workspace_view).  ZERO-FILL it once before
 *   its first use: the fused path keeps a grid-barrier arrival count in it
 *   (the blend_counters region) that every call leaves consistent for the
 *   next.  After a call that reported MOE_ERR_TIMEOUT, zero it again.
 * Shape admission (host, nothing launched on failure):
 *   1 <= M <= MOE_MAX_ROWS (MOE_MAX_ROWS_TC when the layer runs on the
 *   tensor-core path), 1 <= top_k <= min(E, 32), E <= MOE_MAX_EXPERTS,
 *   block_size >= 1, and the format's hidden/inter rules.
 * Errors: MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA. */
int moe_decode_layer(const moe_layer_desc *layer, const uint16_t *x, int M,
                     const float *router_logits, const int32_t *topk_ids,
                     const float *topk_w, uint16_t *out, void *workspace,
                     size_t workspace_bytes, uint32_t *err_word, void *stream);

/* The expert half of moe_decode_layer ("fp8_moe_grouped.rs": the grouped
 * gate+up and down launchers and moe_weighted_sum_blend_fp8_grouped, which
 * run after moe_fp8_grouped_sort): the same grouped gate+up, down and blend,
 * on the routing and alignment tables that an earlier moe_decode_layer call
 * with the same layer and M left in this workspace (topk_ids, topk_w,
 * token_to_perm, sorted_token_ids, the active list and, on the tensor-core
 * paths, the active table of tc_items), with the x given here.  The kernels
 * and the results are those of moe_decode_layer on the same tables: one
 * launch on the fused CUDA-core path (which aligns the ids again, to the
 * same tables); on the tensor-core paths the per-token x table of this x
 * (one launch, when the batch uses one: FP8 up to 16 rows, NVFP4 always)
 * then the expert kernel; three on the staged path (gate+up, down, blend).
 * The workspace rules are moe_decode_layer's.
 * Errors: MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA (as moe_decode_layer). */
int moe_decode_experts(const moe_layer_desc *layer, const uint16_t *x, int M,
                       uint16_t *out, void *workspace, size_t workspace_bytes,
                       uint32_t *err_word, void *stream);

/* ---- the layer without allocation --------------------------------------- */

/* Bytes of the fixed device array that moe_decode_layer_noalloc uses as its
 * workspace (held on every GPU that loads the library until it is unloaded). */
#define MOE_NOALLOC_SCRATCH_BYTES (32u << 20)

/* moe_decode_layer for callers that cannot allocate device memory when they
 * run the layer (code running inside another framework's captured graph or
 * stream callback, plugins whose host forbids device allocation after
 * start-up, embedded runtimes with a device-memory budget fixed at load).
 * The pages have no counterpart: it is the same layer, same arguments and
 * same results as moe_decode_layer, with the workspace taken from a
 * file-scope device array of MOE_NOALLOC_SCRATCH_BYTES instead of a caller
 * buffer.  It calls no allocating routine.
 *   The first call on a device looks up the array's device address (once per
 *   device), so make that call before capturing any stream that contains it.
 *   Every call on a device shares the array and leaves its contents there:
 *   calls that overlap on the GPU race on it, so order them on one stream.
 *   The intermediates are not readable through a workspace view.
 * Errors: as moe_decode_layer, and MOE_EUNSUPPORTED when the layer's
 * workspace for M rows (moe_decode_layer_workspace_bytes) exceeds
 * MOE_NOALLOC_SCRATCH_BYTES; nothing is launched then. */
int moe_decode_layer_noalloc(const moe_layer_desc *layer, const uint16_t *x, int M,
                             const float *router_logits, const int32_t *topk_ids,
                             const float *topk_w, uint16_t *out, uint32_t *err_word,
                             void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
