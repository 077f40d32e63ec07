// route.cuh -- the per-row top-k softmax router as a warp-level device
// function, shared by the router kernel and the fused decode kernels so that
// both produce the same ids and weight bits.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// One warp routes one row of fp32 logits [E] ("forward_nvfp4_grouped_decode.rs",
// grouped_route with GroupedRouting::PerRow; the workload's "softmax then
// top-k renormalised"): the k largest logits (equal logits: lower expert id
// first) in descending order, weights exp(l_j - l_max) / sum over the k
// selected.  Selection compares fp32 values exactly; the weight sum runs as an
// xor butterfly over the 32 lanes (fixed order).  ids[j] / w[j] for j < k are
// written by lane j.  Requires E <= 32 * VPL and k <= 32.
template <int VPL>
__device__ __forceinline__ void topk_softmax_row(const float *l, int E, int k, int32_t *ids,
                                                 float *w) {
  const int lane = threadIdx.x & 31;
  const int nv = (E + 31) / 32;   // logits per lane actually present
  float v[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    v[j] = (j < nv && e < E) ? __ldcg(l + e) : -INFINITY;
  }
  unsigned taken = 0;   // bit j: this lane's j-th value already selected
  float mine = 0.f, vmax = 0.f;
  int myid = 0;
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      if (j >= nv) break;
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (v[j] > bv || bid == 0x7fffffff)) {
        bv = v[j];
        bid = e;
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, d);
      if (oid != 0x7fffffff && (bid == 0x7fffffff || ov > bv || (ov == bv && oid < bid))) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (r == 0) vmax = bv;
    if (lane == r) {       // lane r keeps the r-th selection
      mine = bv;
      myid = bid;
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

}  // namespace moe
