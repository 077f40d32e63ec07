// layer.cu -- the grouped expert entry points (path dispatch) and the decode
// layer: route -> align -> gate+up -> down -> blend on one stream
// ("metrale_model_layers/layers/moe/forward_nvfp4_grouped_decode.rs",
// forward_nvfp4_grouped_decode; every step enqueued, no host read).
#include "common.cuh"
#include "xprep.cuh"

namespace moe {

int validate_experts(const moe_experts *X, bool shared);
int simt_gate_up(const moe_experts *routed, const moe_experts *shared, const uint16_t *x, int M,
                 int top_k, const int32_t *off, const int32_t *sti, const int32_t *act,
                 const int32_t *act_count, float *h, float *h_sh, void *stream);
int simt_down(const moe_experts *routed, const moe_experts *shared, const float *h,
              const float *h_sh, int M, int top_k, const int32_t *off, const int32_t *sti,
              const int32_t *act, const int32_t *act_count, float *y, float *y_sh, void *stream);
int launch_topk(const float *logits, int M, int E, int k, int32_t *ids, float *w, void *stream);
int launch_router(const uint16_t *x, const uint16_t *W, int M, int H, int E, float *logits,
                  void *stream);
int launch_blend(const float *y, const float *w, const int32_t *ttp, const float *y_sh,
                 const uint16_t *x, const uint16_t *gate_w, uint16_t *out, int M, int k, int H,
                 void *stream);
bool fused_fits(const moe_layer_desc *L, int M, int sms);
bool tc_fits(const moe_layer_desc *L, int M);
void tc_workspace(const moe_layer_desc *L, int M, int max_total, int cap, size_t (&bytes)[5]);
size_t tc_counter_ints(const moe_layer_desc *L);
int launch_tc(const moe_layer_desc *L, const uint16_t *x, int M, const float *w,
              const int32_t *ttp, const int32_t *act_count, uint16_t *out, void *ws,
              const moe_workspace_view &v, uint32_t *err, void *stream);
int align_launch(const void *topk_ids, int ids_is_int64, int n, int num_experts, int block_size,
                 int32_t *sorted_token_ids, int32_t *sorted_expert_ids, int32_t *expert_offsets,
                 int32_t *token_to_perm, int32_t *active_experts, int32_t *active_count,
                 int32_t *num_tokens_post_padded, uint32_t *err_word, int4 *items,
                 const XPrep *xp, void *stream);
int xprep_launch(const XPrep &p, void *stream);
bool f4_fits(const moe_layer_desc *L, int M);
void f4_workspace(const moe_layer_desc *L, int max_total, int cap, size_t (&bytes)[5]);
size_t f4_counter_ints(const moe_layer_desc *L);
int launch_f4(const moe_layer_desc *L, const uint16_t *x, int M, const float *w,
              const int32_t *ttp, const int32_t *act_count, uint16_t *out, void *ws,
              const moe_workspace_view &v, uint32_t *err, void *stream);
int launch_fused(const moe_layer_desc *L, const uint16_t *x, int M, const float *logits,
                 const int32_t *ids, const float *w, uint16_t *out, void *ws,
                 const moe_workspace_view &v, uint32_t *err, void *stream);

int run_experts(const moe_layer_desc *layer, int run, const uint16_t *x, int M,
                const int32_t *ids, const float *w, uint16_t *out, void *workspace,
                const moe_workspace_view &v, uint32_t *err_word, void *stream);

// The expert-kernel path of the grouped entry points.  The tensor-core
// kernels keep their activation terms in the layer workspace, so only
// moe_decode_layer runs them.
static int resolve_path(const moe_experts *routed, int M, int top_k, int path) {
  (void)routed;
  (void)M;
  (void)top_k;
  if (path == MOE_PATH_TC) return -1;
  if (path == MOE_PATH_SIMT_STAGED) return MOE_PATH_SIMT_STAGED;
  return MOE_PATH_SIMT;
}

// How moe_decode_layer runs a shape class: the fused CUDA-core kernel, the
// FP8 tensor-core kernel, the staged CUDA-core kernels, or the NVFP4
// tensor-core kernel (which also runs an FP8 shared expert).  It
// depends on the shapes only, never on the routing, so a captured graph stays
// valid for every routing.
enum { kRunFused = 0, kRunTc = 1, kRunStaged = 2, kRunTcF4 = 3 };

static int layer_run(const moe_layer_desc *L, int M) {
  switch (L->path) {
    case MOE_PATH_TC:
      if (tc_fits(L, M)) return kRunTc;
      return f4_fits(L, M) ? kRunTcF4 : -1;
    case MOE_PATH_SIMT_STAGED:
      return kRunStaged;
    case MOE_PATH_SIMT:
      return fused_fits(L, M, sm_count()) ? kRunFused : kRunStaged;
    default:   // the tensor cores for every shape they admit, else CUDA cores
      if (tc_fits(L, M)) return kRunTc;
      if (f4_fits(L, M)) return kRunTcF4;
      return fused_fits(L, M, sm_count()) ? kRunFused : kRunStaged;
  }
}

static bool is_tc(int run) { return run == kRunTc || run == kRunTcF4; }

// The per-token x table a tensor-core run reads (the FP8 kernel's up to 16
// rows, the NVFP4 kernel's up to 32), else mode none.
static XPrep token_table(const moe_layer_desc *L, int run, const uint16_t *x, int M, char *ws,
                         const moe_workspace_view &v) {
  XPrep p{};
  if (run == kRunTc && M <= 16) {
    p.mode = kXPrepE4M3;
    p.NT = 16;
  } else if (run == kRunTcF4) {
    p.mode = kXPrepF16;
    p.NT = M <= 16 ? 16 : 32;
    if (L->shared && L->shared_gate) {
      p.gate_w = L->shared_gate;
      p.gate_vals = reinterpret_cast<float *>(ws + v.shared_gate);
    }
  } else {
    return p;
  }
  p.M = M;
  p.H = L->routed.hidden;
  p.x = x;
  p.table = reinterpret_cast<uint8_t *>(ws + v.tc_x_terms);
  p.scale = reinterpret_cast<float *>(ws + v.tc_x_scale);
  return p;
}

// Whether the layer runs a tensor-core kernel at some M: its counters then
// have their place at offset 256 for every M, so that calls at M the
// CUDA cores take do not overwrite them.
static bool tc_layer(const moe_layer_desc *L) {
  if (L->path != MOE_PATH_AUTO && L->path != MOE_PATH_TC) return false;
  return tc_fits(L, 1) || f4_fits(L, 1);
}

// Bytes of the tensor-core kernels' counters (each call leaves them
// consistent for the next): sized by the layer alone.
size_t tc_counter_bytes(const moe_layer_desc *L) {
  const bool f4 = L->routed.fmt == MOE_FMT_NVFP4_G16 || L->routed.fmt == MOE_FMT_NVFP4_GATE_UP;
  return 4 * (f4 ? f4_counter_ints(L) : tc_counter_ints(L));
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int layout(const moe_layer_desc *L, int M, moe_workspace_view *v) {
  if (!L || !v) return MOE_EINVAL;
  int st = validate_experts(&L->routed, false);
  if (st) return st;
  if (L->shared) {
    st = validate_experts(L->shared, true);
    if (st) return st;
    if (L->shared->hidden != L->routed.hidden) return MOE_EINVAL;
  }
  if (L->shared_gate && (!L->shared || ((uintptr_t)L->shared_gate & 15))) return MOE_EINVAL;
  const int E = L->routed.num_experts, k = L->top_k;
  if (M < 1 || k < 1 || k > E || L->block_size < 1) return MOE_EINVAL;
  if (k > 32 || M > MOE_MAX_ROWS_TC) return MOE_EUNSUPPORTED;
  // above MOE_MAX_ROWS only the tensor-core path (prefill-sized batches)
  if (M > MOE_MAX_ROWS && layer_run(L, M) != kRunTc) return MOE_EUNSUPPORTED;
  const int n = M * k;
  int max_total, max_blocks, cap;
  st = moe_align_sizes(n, E, L->block_size, &max_total, &max_blocks, &cap);
  if (st) return st;
  const int H = L->routed.hidden, I = L->routed.inter;
  const int Is = L->shared ? L->shared->inter : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  // The counters that persist from call to call come first, at offsets and
  // sizes that do not depend on M, so that one workspace serves every M up to
  // the one it was sized for: the grid-barrier count at 0, then the
  // tensor-core path's counters (sized by the layer alone).
  v->blend_counters = take(8);
  if (L->path != MOE_PATH_AUTO && L->path != MOE_PATH_SIMT && L->path != MOE_PATH_TC &&
      L->path != MOE_PATH_SIMT_STAGED)
    return MOE_EINVAL;
  const int run = layer_run(L, M);
  v->tc_done = tc_layer(L) ? take(tc_counter_bytes(L)) : 0;
  v->topk_ids = take((size_t)n * 4);
  v->topk_w = take((size_t)n * 4);
  v->sorted_token_ids = take((size_t)max_total * 4);
  v->sorted_expert_ids = take((size_t)max_blocks * 4);
  v->expert_offsets = take((size_t)(E + 1) * 4);
  v->token_to_perm = take((size_t)n * 4);
  v->active_experts = take((size_t)cap * 4);
  v->active_count = take(4);
  v->num_tokens_post_padded = take(4);
  v->h = take((size_t)max_total * I * 4);
  v->h_shared = take((size_t)M * Is * 4);
  v->y = take((size_t)max_total * H * 4);
  v->y_shared = take((size_t)M * H * 4);
  v->router_logits = take((size_t)M * E * 4);
  v->shared_gate = take((size_t)M * 4);
  v->tc_x_terms = v->tc_x_scale = v->tc_h_terms = v->tc_h_scale = 0;
  v->tc_items = 0;
  if (is_tc(run)) {
    size_t b[5];
    if (run == kRunTc)
      tc_workspace(L, M, max_total, cap, b);
    else
      f4_workspace(L, max_total, cap, b);
    v->tc_x_terms = take(b[0]);
    v->tc_x_scale = take(b[1]);
    v->tc_h_terms = take(b[2]);
    v->tc_h_scale = take(b[3]);
    v->tc_items = take(b[4]);
  }
  v->total_bytes = off;
  v->max_total = max_total;
  v->max_blocks = max_blocks;
  v->cap = cap;
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_grouped_gate_up(const moe_experts *routed, const moe_experts *shared,
                                   const uint16_t *x, int M, int top_k,
                                   const int32_t *expert_offsets, const int32_t *sorted_token_ids,
                                   const int32_t *active_experts, const int32_t *active_count,
                                   float *h, float *h_shared, int path, void *stream) {
  if (!routed) return MOE_EINVAL;
  const int p = moe::resolve_path(routed, M, top_k, path);
  if (p < 0) return MOE_EUNSUPPORTED;
  return moe::simt_gate_up(routed, shared, x, M, top_k, expert_offsets, sorted_token_ids,
                           active_experts, active_count, h, h_shared, stream);
}

extern "C" int moe_grouped_down(const moe_experts *routed, const moe_experts *shared,
                                const float *h, const float *h_shared, int M, int top_k,
                                const int32_t *expert_offsets, const int32_t *sorted_token_ids,
                                const int32_t *active_experts, const int32_t *active_count,
                                float *y, float *y_shared, int path, void *stream) {
  if (!routed) return MOE_EINVAL;
  const int p = moe::resolve_path(routed, M, top_k, path);
  if (p < 0) return MOE_EUNSUPPORTED;
  return moe::simt_down(routed, shared, h, h_shared, M, top_k, expert_offsets, sorted_token_ids,
                        active_experts, active_count, y, y_shared, stream);
}

extern "C" size_t moe_decode_layer_workspace_bytes(const moe_layer_desc *layer, int max_M) {
  moe_workspace_view v;
  if (moe::layout(layer, max_M, &v) != MOE_OK) return 0;
  size_t most = v.total_bytes;
  for (int m = 1; m < max_M; ++m)
    if (moe::layout(layer, m, &v) == MOE_OK && v.total_bytes > most) most = v.total_bytes;
  return most;
}

extern "C" int moe_decode_layer_workspace_view(const moe_layer_desc *layer, int M,
                                               moe_workspace_view *view) {
  return moe::layout(layer, M, view);
}

extern "C" int moe_decode_layer_launches(const moe_layer_desc *layer, int M, int with_logits) {
  moe_workspace_view v;
  if (moe::layout(layer, M, &v) != MOE_OK) return -1;
  const int run = moe::layer_run(layer, M);
  if (run < 0) return -1;
  if (with_logits == 2 && !layer->router_weight) return -1;
  const int router = with_logits == 2;   // the logits kernel ahead of the route
  if (run == moe::kRunFused) return 1 + router;
  if (moe::is_tc(run)) return (with_logits ? 3 : 2) + router;
  return (with_logits ? 5 : 4) + router;
}

namespace moe {

// Every host check of a moe_decode_layer call except those on the workspace:
// the descriptor and M (through the layout, returned in *v), the inputs, the
// output, and that a path admits the shape.  MOE_OK or the status to return.
int check_layer_call(const moe_layer_desc *layer, const uint16_t *x, int M,
                     const float *router_logits, const int32_t *topk_ids, const float *topk_w,
                     const uint16_t *out, moe_workspace_view *v) {
  int st = layout(layer, M, v);
  if (st) return st;
  if (!x || !out) return MOE_EINVAL;
  // hidden in: the logits come from x and the layer's router weights
  const bool hidden_in = !router_logits && !topk_ids && layer->router_weight;
  if (!router_logits && !hidden_in && (!topk_ids || !topk_w)) return MOE_EINVAL;
  if (hidden_in && ((uintptr_t)layer->router_weight & 15)) return MOE_EINVAL;
  if (((uintptr_t)x & 15) || ((uintptr_t)out & 7)) return MOE_EINVAL;
  if (layer_run(layer, M) < 0) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_decode_layer(const moe_layer_desc *layer, const uint16_t *x, int M,
                                const float *router_logits, const int32_t *topk_ids,
                                const float *topk_w, uint16_t *out, void *workspace,
                                size_t workspace_bytes, uint32_t *err_word, void *stream) {
  moe_workspace_view v;
  int st = moe::check_layer_call(layer, x, M, router_logits, topk_ids, topk_w, out, &v);
  if (st) return st;
  if (!workspace) return MOE_EINVAL;
  if (workspace_bytes < v.total_bytes || ((uintptr_t)workspace & 255)) return MOE_EINVAL;
  const bool hidden_in = !router_logits && !topk_ids && layer->router_weight;
  const int run = moe::layer_run(layer, M);

  char *ws = reinterpret_cast<char *>(workspace);
  auto I32 = [&](size_t o) { return reinterpret_cast<int32_t *>(ws + o); };
  auto F32 = [&](size_t o) { return reinterpret_cast<float *>(ws + o); };
  const int E = layer->routed.num_experts, k = layer->top_k, H = layer->routed.hidden;

  if (hidden_in) {
    st = moe::launch_router(x, layer->router_weight, M, H, E, F32(v.router_logits), stream);
    if (st) return st;
    router_logits = F32(v.router_logits);
  }
  if (run == moe::kRunFused)
    return moe::launch_fused(layer, x, M, router_logits, topk_ids, topk_w, out, workspace, v,
                             err_word, stream);

  const int32_t *ids = topk_ids;
  const float *w = topk_w;
  if (router_logits) {
    st = moe::launch_topk(router_logits, M, E, k, I32(v.topk_ids), F32(v.topk_w), stream);
    if (st) return st;
    ids = I32(v.topk_ids);
    w = F32(v.topk_w);
  }
  // the tensor-core kernels also take the active table (offset, expert and
  // slot count of each active expert) and their per-token x table from the
  // alignment launch
  const moe::XPrep xp = moe::token_table(layer, run, x, M, ws, v);
  st = moe::align_launch(ids, 0, M * k, E, layer->block_size, I32(v.sorted_token_ids),
                         I32(v.sorted_expert_ids), I32(v.expert_offsets), I32(v.token_to_perm),
                         I32(v.active_experts), I32(v.active_count),
                         I32(v.num_tokens_post_padded), err_word,
                         moe::is_tc(run) ? reinterpret_cast<int4 *>(ws + v.tc_items) : nullptr,
                         &xp, stream);
  if (st) return st;
  return moe::run_experts(layer, run, x, M, ids, w, out, workspace, v, err_word, stream);
}

namespace moe {

// The expert half of a layer call, after the routing and the alignment
// tables are in the workspace: a tensor-core kernel, or the staged gate+up,
// down and blend.
int run_experts(const moe_layer_desc *layer, int run, const uint16_t *x, int M,
                const int32_t *ids, const float *w, uint16_t *out, void *workspace,
                const moe_workspace_view &v, uint32_t *err_word, void *stream) {
  char *ws = reinterpret_cast<char *>(workspace);
  auto I32 = [&](size_t o) { return reinterpret_cast<int32_t *>(ws + o); };
  auto F32 = [&](size_t o) { return reinterpret_cast<float *>(ws + o); };
  const int k = layer->top_k, H = layer->routed.hidden;
  const moe_experts *S = layer->shared;
  (void)ids;
  if (run == kRunTc)
    return launch_tc(layer, x, M, w, I32(v.token_to_perm), I32(v.active_count), out, workspace,
                     v, err_word, stream);
  if (run == kRunTcF4)
    return launch_f4(layer, x, M, w, I32(v.token_to_perm), I32(v.active_count), out, workspace,
                     v, err_word, stream);
  int st = simt_gate_up(&layer->routed, S, x, M, k, I32(v.expert_offsets),
                        I32(v.sorted_token_ids), I32(v.active_experts), I32(v.active_count),
                        F32(v.h), S ? F32(v.h_shared) : nullptr, stream);
  if (st) return st;
  st = simt_down(&layer->routed, S, F32(v.h), S ? F32(v.h_shared) : nullptr, M, k,
                 I32(v.expert_offsets), I32(v.sorted_token_ids), I32(v.active_experts),
                 I32(v.active_count), F32(v.y), S ? F32(v.y_shared) : nullptr, stream);
  if (st) return st;
  return launch_blend(F32(v.y), w, I32(v.token_to_perm), S ? F32(v.y_shared) : nullptr, x,
                      S ? layer->shared_gate : nullptr, out, M, k, H, stream);
}

}  // namespace moe

extern "C" int moe_decode_experts(const moe_layer_desc *layer, const uint16_t *x, int M,
                                  uint16_t *out, void *workspace, size_t workspace_bytes,
                                  uint32_t *err_word, void *stream) {
  moe_workspace_view v;
  int st = moe::layout(layer, M, &v);
  if (st) return st;
  if (!x || !out || !workspace) return MOE_EINVAL;
  if (((uintptr_t)x & 15) || ((uintptr_t)out & 7)) return MOE_EINVAL;
  if (workspace_bytes < v.total_bytes || ((uintptr_t)workspace & 255)) return MOE_EINVAL;
  const int run = moe::layer_run(layer, M);
  if (run < 0) return MOE_EUNSUPPORTED;
  char *ws = reinterpret_cast<char *>(workspace);
  const int32_t *ids = reinterpret_cast<const int32_t *>(ws + v.topk_ids);
  const float *w = reinterpret_cast<const float *>(ws + v.topk_w);
  if (run == moe::kRunFused)   // it aligns the given ids again, to the same tables
    return moe::launch_fused(layer, x, M, nullptr, ids, w, out, workspace, v, err_word, stream);
  // the tensor-core runs' per-token x table of this x (one launch more)
  st = moe::xprep_launch(moe::token_table(layer, run, x, M, ws, v), stream);
  if (st) return st;
  return moe::run_experts(layer, run, x, M, ids, w, out, workspace, v, err_word, stream);
}
