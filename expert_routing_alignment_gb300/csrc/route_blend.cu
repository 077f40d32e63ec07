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
// router logits: the k dimension split over a block's threads
// ---------------------------------------------------------------------------
//
// What (the router matrix-vector product ahead of the top-k; the pages name
// router_gemv_batchm in nvfp4_grouped_decode_ok of
// "forward_nvfp4_grouped_decode.rs"): logits[t][e] = sum_c x[t][c] * W[e][c]
// for bf16 x [M][H] and bf16 W [E][H], fp32 result.
// How: a block owns RE (1, 2 or 4) expert rows and 8 x rows.  Thread i of the block takes
// the 16-byte chunks i, i + 256, ... of every row, so each row of W is read
// once per 8 x rows, in whole-block coalesced lines, and x comes from L2.
// Each thread keeps RE x 8 fp32 partial sums (fmaf in chunk order, elements
// ascending); a warp ends them with a reduce-scatter butterfly (xor 16, 8, 4,
// 2, 1: the pairing tree of a plain butterfly, so every sum is added in the
// same tree) and the 8 warps' sums are added in warp order.  The order of
// every addition depends on H alone: a row's logits are the same bits for
// every M, every RE and every run.  Products of two bf16 values are exact in
// fp32.

constexpr int kRouterThreads = 256;
constexpr int kRouterRows = 8;   // x rows per block

template <int RE>   // expert rows per block
__global__ void __launch_bounds__(kRouterThreads)
    router_logits_kernel(const uint16_t *x, const uint16_t *W, int M, int H, int E,
                         float *logits) {
  constexpr int N = RE * kRouterRows;   // partial sums per thread, index re * 8 + r
  __shared__ float red[kRouterThreads / 32][N];
  pdl_wait();
  pdl_trigger();
  const int e0 = blockIdx.x * RE, t0 = blockIdx.y * kRouterRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = H / 8;   // 16-byte chunks per row
  float acc[N];
#pragma unroll
  for (int i = 0; i < N; ++i) acc[i] = 0.f;
  // U chunks' loads are issued before any is used (the decode widths are
  // bound by load latency); the sums still take the chunks in ascending order
  constexpr int U = RE == 1 ? 4 : RE == 2 ? 2 : 1;
  for (int c0 = tid; c0 < chunks; c0 += U * kRouterThreads) {
    uint4 wv[U][RE], xv[U][kRouterRows];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * kRouterThreads;
#pragma unroll
      for (int re = 0; re < RE; ++re)
        wv[u][re] = c < chunks && e0 + re < E
                        ? ld_stream16(reinterpret_cast<const uint4 *>(W + (size_t)(e0 + re) * H) + c)
                        : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < kRouterRows; ++r)
        xv[u][r] = c < chunks && t0 + r < M
                       ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + r) * H) + c)
                       : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + u * kRouterThreads >= chunks) break;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float wl[RE], wh[RE], xl[kRouterRows], xh[kRouterRows];
#pragma unroll
        for (int re = 0; re < RE; ++re) {
          const uint4 q = wv[u][re];
          const uint32_t v = h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w;
          wl[re] = __uint_as_float(v << 16);
          wh[re] = __uint_as_float(v & 0xFFFF0000u);
        }
#pragma unroll
        for (int r = 0; r < kRouterRows; ++r) {
          const uint4 q = xv[u][r];
          const uint32_t v = h == 0 ? q.x : h == 1 ? q.y : h == 2 ? q.z : q.w;
          xl[r] = __uint_as_float(v << 16);
          xh[r] = __uint_as_float(v & 0xFFFF0000u);
        }
#pragma unroll
        for (int re = 0; re < RE; ++re)
#pragma unroll
          for (int r = 0; r < kRouterRows; ++r) {
            float &v = acc[re * kRouterRows + r];
            v = fmaf(wl[re], xl[r], v);
            v = fmaf(wh[re], xh[r], v);
          }
      }
    }
  }
  // reduce-scatter: while a lane holds more than one sum it keeps half of them
  // (the upper half where its lane bit is set) and adds the partner's copy
  int idx = 0;   // the first sum this lane ends with
  int cnt = N;
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    if (cnt > 1) {
      const bool up = lane & m;
      const int half = cnt / 2;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = up ? acc[i] : acc[i + half];
          const float keep = up ? acc[i + half] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
        }
      }
      if (up) idx += half;
      cnt = half;
    } else {
      acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], m);
    }
  }
  // lanes that hold the same sums (N < 32) wrote equal values; one writes
  if ((lane & (32 * cnt / N - 1)) == 0)
#pragma unroll
    for (int i = 0; i < (N >= 32 ? N / 32 : 1); ++i) red[warp][idx + i] = acc[i];
  __syncthreads();
  if (tid < N) {
    float v = red[0][tid];
#pragma unroll
    for (int w = 1; w < kRouterThreads / 32; ++w) v += red[w][tid];
    const int re = tid / kRouterRows, r = tid - re * kRouterRows;
    if (e0 + re < E && t0 + r < M) logits[(size_t)(t0 + r) * E + e0 + re] = v;
  }
}

// ---------------------------------------------------------------------------
// blend
// ---------------------------------------------------------------------------
//
// What ("fp8_moe_grouped.rs", moe_weighted_sum_blend_fp8_grouped; the fixed
// order of "moe_decode_vec.py"'s combine): out[t][c] = bf16_rn(sum_j w[t][j] *
// y[token_to_perm[t*k+j]][c] + g[t] * y_sh[t][c]), fp32, j ascending, then the
// shared term; g[t] = sigmoid(x[t] . gate_w) when the shared expert is gated
// (shared_gate_warp), else the term is added as it is.  How: grid
// (ceil(H/1024), M), each thread 4 consecutive columns with 16-byte loads; no
// atomics.  Warp 0 of each block computes its token's gate.

__global__ void __launch_bounds__(256) blend_kernel(const float *y, const float *w,
                                                    const int32_t *ttp, const float *y_sh,
                                                    const uint16_t *x, const uint16_t *gate_w,
                                                    uint16_t *out, int M, int k, int H) {
  __shared__ float gate_s;
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  if (gate_w) {
    if (threadIdx.x < 32) {
      const float g = shared_gate_warp(x + (size_t)t * H, gate_w, H);
      if (threadIdx.x == 0) gate_s = g;
    }
    __syncthreads();
  }
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
    if (gate_w) {
      const float g = gate_s;
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    } else {
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
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
                 const uint16_t *x, const uint16_t *gate_w, uint16_t *out, int M, int k, int H,
                 void *stream) {
  const dim3 grid((H / 4 + 255) / 256, M);
  return launch_pdl(blend_kernel, grid, dim3(256), 0, stream, y, w, ttp, y_sh, x, gate_w, out, M,
                    k, H);
}

// Expert rows per block: the most (up to 4, for the fewest re-reads of x; 8
// holds too many registers for two blocks per SM) that still leave two blocks
// per SM; 1 when even that is too few blocks.
int launch_router(const uint16_t *x, const uint16_t *W, int M, int H, int E, float *logits,
                  void *stream) {
  const int row_blocks = (M + kRouterRows - 1) / kRouterRows;
  const int want = 2 * sm_count();
  auto blocks = [&](int re) { return ((E + re - 1) / re) * row_blocks; };
  const dim3 block(kRouterThreads);
  if (blocks(4) >= want)
    return launch_pdl(router_logits_kernel<4>, dim3((E + 3) / 4, row_blocks), block, 0, stream, x,
                      W, M, H, E, logits);
  if (blocks(2) >= want)
    return launch_pdl(router_logits_kernel<2>, dim3((E + 1) / 2, row_blocks), block, 0, stream, x,
                      W, M, H, E, logits);
  return launch_pdl(router_logits_kernel<1>, dim3(E, row_blocks), block, 0, stream, x, W, M, H, E,
                    logits);
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

extern "C" int moe_router_logits(const uint16_t *x, const uint16_t *router_weight, int M,
                                 int hidden, int num_experts, float *logits, void *stream) {
  if (!x || !router_weight || !logits || M < 1 || hidden < 1 || num_experts < 1)
    return MOE_EINVAL;
  if (hidden % 8 || ((uintptr_t)x & 15) || ((uintptr_t)router_weight & 15))
    return MOE_EUNSUPPORTED;
  return moe::launch_router(x, router_weight, M, hidden, num_experts, logits, stream);
}

extern "C" int moe_blend(const float *y, const float *topk_w, const int32_t *token_to_perm,
                         const float *y_shared, const uint16_t *x, const uint16_t *shared_gate,
                         uint16_t *out, int M, int top_k, int hidden, void *stream) {
  if (!y || !topk_w || !token_to_perm || !out || M < 1 || top_k < 1 || hidden < 1)
    return MOE_EINVAL;
  if (shared_gate && (!y_shared || !x)) return MOE_EINVAL;
  if (hidden % 4 != 0 || ((uintptr_t)y & 15) || ((uintptr_t)out & 7) ||
      (y_shared && ((uintptr_t)y_shared & 15)))
    return MOE_EUNSUPPORTED;
  if (shared_gate && (hidden % 8 != 0 || ((uintptr_t)x & 15) || ((uintptr_t)shared_gate & 15)))
    return MOE_EUNSUPPORTED;
  return moe::launch_blend(y, topk_w, token_to_perm, y_shared, x, shared_gate, out, M, top_k,
                           hidden, stream);
}
