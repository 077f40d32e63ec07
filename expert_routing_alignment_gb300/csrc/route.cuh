// route.cuh -- the per-row top-k softmax router as a warp-level device
// function, shared by the router kernel and the fused decode kernels so that
// both produce the same ids and weight bits.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// Order-preserving map of a float to an unsigned key (larger float, larger
// key; -0.0 is taken as +0.0 so that the two compare equal).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp routes one row of fp32 logits [E] ("forward_nvfp4_grouped_decode.rs",
// grouped_route with GroupedRouting::PerRow; the workload's "softmax then
// top-k renormalised"): the k largest logits (equal logits: lower expert id
// first) in descending order, weights exp(l_j - l_max) / sum over the k
// selected.  Each selection round takes the warp's largest key with one
// redux.sync and, among the lanes holding it, the lowest expert id with a
// second.  The weight sum runs as an xor butterfly over the 32 lanes (fixed
// order).  ids[j] / w[j] for j < k are written by lane j.  Requires
// E <= 32 * VPL and k <= 32.
template <int VPL>
__device__ __forceinline__ void topk_softmax_row(const float *l, int E, int k, int32_t *ids,
                                                 float *w) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) / 32;   // logits per lane actually present
  uint32_t key[VPL];              // 0: absent (below every real logit)
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = (j < nv && e < E) ? order_key(__ldcg(l + e)) : 0u;
  }
  unsigned taken = 0;   // bit j: this lane's j-th value already selected
  float mine = 0.f, vmax = 0.f;
  int myid = 0;
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (j >= nv) break;
      if (!((taken >> j) & 1u) && key[j] > bk) {   // strict: the lower id wins a tie
        bk = key[j];
        bj = j;
      }
    }
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bj >= 0 && bk == wk) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
    const uint32_t wid = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(wid & 31u) == lane) taken |= 1u << (wid >> 5);
    const float wv = key_value(wk);
    if (r == 0) vmax = wv;
    if (lane == r) {       // lane r keeps the r-th selection
      mine = wv;
      myid = (int)wid;
    }
  }
  const float ex = lane < k ? expf(mine - vmax) : 0.f;
  float z = ex;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  if (lane < k) {
    ids[lane] = myid;
    w[lane] = ex / z;
  }
}

// The shared expert's gate of one token, by one warp ("fp8_moe_grouped.rs":
// moe_weighted_sum_blend_fp8_grouped takes the layer input and
// shared_expert_gate.weight; read as a one-output gate layer):
// sigmoid(sum_c x[c] * g[c]) over bf16 x [H] and bf16 g [H], H % 8 == 0, both
// 16-byte aligned.  Lane l sums the 16-byte chunks l, l + 32, ... with fmaf
// (elements ascending), an xor butterfly ends the sum, so the blend kernel and
// the fused kernel get the same bits.  Every lane returns the gate.
__device__ __forceinline__ float shared_gate_warp(const uint16_t *x, const uint16_t *g, int H) {
  const int lane = threadIdx.x & 31;
  float z = 0.f;
#pragma unroll 4
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x) + c);
    const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(g) + c);
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, gs[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z = fmaf(__uint_as_float(xs[i] << 16), __uint_as_float(gs[i] << 16), z);
      z = fmaf(__uint_as_float(xs[i] & 0xFFFF0000u), __uint_as_float(gs[i] & 0xFFFF0000u), z);
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  return 1.f / (1.f + expf(-z));
}

}  // namespace moe
