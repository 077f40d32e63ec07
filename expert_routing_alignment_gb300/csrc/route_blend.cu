// route_blend.cu -- per-row top-k softmax router (moe_topk_softmax) and the
// fixed-order weighted blend back to token order (moe_blend).
#include <math.h>

#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// top-k softmax: one warp per row
// ---------------------------------------------------------------------------
//
// What ("forward_nvfp4_grouped_decode.rs", grouped_route with
// GroupedRouting::PerRow; the workload's "softmax then top-k renormalised"):
// the k largest logits of the row (equal logits: lower expert id first), in
// descending order, with weights exp(l_j - l_max) / sum over the k selected
// (= softmax over all E, restricted to the selection, renormalised).
// How: a warp keeps the row in registers (E <= 1024 -> up to 32 values per
// lane) and runs k rounds of a warp arg-max on (value, -id); selection
// compares fp32 values exactly, so the chosen ids are the oracle's.

constexpr int kTopkWarps = 4;

template <int VPL>   // logits per lane: E <= 32 * VPL
__global__ void __launch_bounds__(32 * kTopkWarps) topk_softmax_kernel(const float *logits, int M,
                                                                       int E, int k, int32_t *ids,
                                                                       float *w) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  topk_softmax_row<VPL>(logits + (size_t)row * E, E, k, ids + (size_t)row * k,
                        w + (size_t)row * k);
}

// ---------------------------------------------------------------------------
// blend
// ---------------------------------------------------------------------------
//
// What ("fp8_moe_grouped.rs", moe_weighted_sum_blend_fp8_grouped; the fixed
// order of "moe_decode_vec.py"'s combine): out[t][c] = bf16_rn(sum_j w[t][j] *
// y[token_to_perm[t*k+j]][c] + y_sh[t][c]), fp32, j ascending, then the shared
// term.  How: grid (ceil(H/1024), M), each thread 4 consecutive columns with
// 16-byte loads; no atomics.

__global__ void __launch_bounds__(256) blend_kernel(const float *y, const float *w,
                                                    const int32_t *ttp, const float *y_sh,
                                                    uint16_t *out, int M, int k, int H) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int c = (blockIdx.x * 256 + threadIdx.x) * 4;
  if (c >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int p = __ldcg(ttp + (size_t)t * k + j);
    if (p < 0) continue;
    const float wj = __ldcg(w + (size_t)t * k + j);
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)p * H + c));
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  if (y_sh) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(y_sh + (size_t)t * H + c));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const uint32_t lo = (uint32_t)float_to_bf16_rn(acc.x) | ((uint32_t)float_to_bf16_rn(acc.y) << 16);
  const uint32_t hi = (uint32_t)float_to_bf16_rn(acc.z) | ((uint32_t)float_to_bf16_rn(acc.w) << 16);
  *reinterpret_cast<uint2 *>(out + (size_t)t * H + c) = make_uint2(lo, hi);
}

}  // namespace

int launch_topk(const float *logits, int M, int E, int k, int32_t *ids, float *w, void *stream) {
  const dim3 grid((M + kTopkWarps - 1) / kTopkWarps), block(32 * kTopkWarps);
  if (E <= 32) return launch_pdl(topk_softmax_kernel<1>, grid, block, 0, stream, logits, M, E, k, ids, w);
  if (E <= 64) return launch_pdl(topk_softmax_kernel<2>, grid, block, 0, stream, logits, M, E, k, ids, w);
  if (E <= 128) return launch_pdl(topk_softmax_kernel<4>, grid, block, 0, stream, logits, M, E, k, ids, w);
  if (E <= 256) return launch_pdl(topk_softmax_kernel<8>, grid, block, 0, stream, logits, M, E, k, ids, w);
  if (E <= 512) return launch_pdl(topk_softmax_kernel<16>, grid, block, 0, stream, logits, M, E, k, ids, w);
  return launch_pdl(topk_softmax_kernel<32>, grid, block, 0, stream, logits, M, E, k, ids, w);
}

int launch_blend(const float *y, const float *w, const int32_t *ttp, const float *y_sh,
                 uint16_t *out, int M, int k, int H, void *stream) {
  const dim3 grid((H / 4 + 255) / 256, M);
  return launch_pdl(blend_kernel, grid, dim3(256), 0, stream, y, w, ttp, y_sh, out, M, k, H);
}

}  // namespace moe

extern "C" int moe_topk_softmax(const float *logits, int M, int num_experts, int top_k,
                                int32_t *topk_ids, float *topk_w, void *stream) {
  if (!logits || !topk_ids || !topk_w || M < 1 || num_experts < 1 || top_k < 1 ||
      top_k > num_experts)
    return MOE_EINVAL;
  if (num_experts > MOE_MAX_EXPERTS || top_k > 32) return MOE_EUNSUPPORTED;
  return moe::launch_topk(logits, M, num_experts, top_k, topk_ids, topk_w, stream);
}

extern "C" int moe_blend(const float *y, const float *topk_w, const int32_t *token_to_perm,
                         const float *y_shared, uint16_t *out, int M, int top_k, int hidden,
                         void *stream) {
  if (!y || !topk_w || !token_to_perm || !out || M < 1 || top_k < 1 || hidden < 1)
    return MOE_EINVAL;
  if (hidden % 4 != 0 || ((uintptr_t)y & 15) || ((uintptr_t)out & 7) ||
      (y_shared && ((uintptr_t)y_shared & 15)))
    return MOE_EUNSUPPORTED;
  return moe::launch_blend(y, topk_w, token_to_perm, y_shared, out, M, top_k, hidden, stream);
}
