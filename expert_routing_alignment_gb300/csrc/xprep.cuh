// xprep.cuh -- the per-token x tables of the tensor-core expert kernels,
// written by extra CTAs of the alignment launch (or by a launch of their
// own), so that the expert kernels find them complete when their
// programmatic-dependency wait returns: no flags, no fences, no wait for
// another CTA inside the expert kernels.
//
// Two formats, one CTA per token t < M (the first 128 threads compute, so the
// results do not depend on the width of the launch):
//  * FP8 kernel (M <= 16): two E4M3 terms x * 2^s = t0 + t1 (exact for bf16
//    x), s putting max|x[t]| in [128, 256); term r of element c at byte
//    (c/128 * 2 + r) * 16 * 128 + t * 128 + c % 128; scale[t] = 2^-s.
//  * NVFP4 kernel (M <= 32): one f16 term x * 2^s (exact), s putting max|x[t]|
//    in [2^14, 2^15); element c at byte ((c/128 * 2 + (c % 128) / 64) * NT + t)
//    * 128 + (c % 64) * 2 for NT = 16 or 32 token columns; scale[t] = 2^-s;
//    with a gated shared expert also gate_vals[t] = sigmoid(x[t] . gate_w),
//    the fp32 dot summed per thread, then by a fixed warp tree, then over the
//    warps in order.
#pragma once

#include "tc_common.cuh"

namespace moe {

enum { kXPrepNone = 0, kXPrepE4M3 = 1, kXPrepF16 = 2 };

struct XPrep {
  int mode;        // kXPrep*
  int M, H, NT;    // rows, hidden, token columns of the table (E4M3: 16)
  const uint16_t *x;
  uint8_t *table;
  float *scale;
  const uint16_t *gate_w;   // NVFP4 only: [H] bf16 shared gate, or NULL
  float *gate_vals;         // [M]
};

constexpr int kXPrepThreads = 128;

// Token t's row of the table (called by every thread of the CTA; red holds 8
// ints of shared memory).
__device__ inline void xprep_token(const XPrep &p, int t, int *red) {
  using namespace tc;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bool worker = tid < kXPrepThreads;
  const uint16_t *xr = p.x + (size_t)t * p.H;
  uint32_t mx = 0;
  float dot = 0.f;
  const bool gated = p.mode == kXPrepF16 && p.gate_w;
  for (int c = tid * 8; worker && c < p.H; c += kXPrepThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + c));
    const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      mx = max(mx, (xv[h] & 0x7FFFu) << 16);
      mx = max(mx, (xv[h] >> 16 & 0x7FFFu) << 16);
    }
    if (gated) {
      const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(p.gate_w + c));
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        dot = fmaf(bf16_to_float((uint16_t)(xv[h] & 0xFFFFu)),
                   bf16_to_float((uint16_t)(gw[h] & 0xFFFFu)), dot);
        dot = fmaf(bf16_to_float((uint16_t)(xv[h] >> 16)), bf16_to_float((uint16_t)(gw[h] >> 16)),
                   dot);
      }
    }
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, d);
  if (worker && lane == 0) {
    red[w] = (int)mx;
    reinterpret_cast<float *>(red)[4 + w] = dot;
  }
  __syncthreads();
  mx = 0;
  for (int j = 0; j < kXPrepThreads / 32; ++j) mx = max(mx, (uint32_t)red[j]);
  int sh;
  if (p.mode == kXPrepE4M3) {
    sh = term_shift(mx);
  } else {
    sh = 0;
    if (mx) {
      const int e = (int)(mx >> 23) - 127;
      sh = 14 - e;
      sh = sh < -126 ? -126 : (sh > 126 ? 126 : sh);
    }
  }
  const float scl = pow2f(sh);
  if (tid == 0) {
    p.scale[t] = pow2f(-sh);
    if (gated) {
      float z = 0.f;
      for (int j = 0; j < kXPrepThreads / 32; ++j) z += reinterpret_cast<float *>(red)[4 + j];
      p.gate_vals[t] = 1.f / (1.f + expf(-z));
    }
  }
  if (!worker) return;
  if (p.mode == kXPrepE4M3) {
    for (int c = tid * 4; c < p.H; c += kXPrepThreads * 4) {
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(xr + c));
      uint32_t t0a, t1a, t0b, t1b;
      e4m3_split2(bf16_to_float((uint16_t)(v.x & 0xFFFFu)) * scl,
                  bf16_to_float((uint16_t)(v.x >> 16)) * scl, t0a, t1a);
      e4m3_split2(bf16_to_float((uint16_t)(v.y & 0xFFFFu)) * scl,
                  bf16_to_float((uint16_t)(v.y >> 16)) * scl, t0b, t1b);
      uint8_t *dst = p.table + (size_t)(c / 128) * 2 * 16 * 128 + (size_t)t * 128 + c % 128;
      *reinterpret_cast<uint32_t *>(dst) = t0a | (t0b << 16);
      *reinterpret_cast<uint32_t *>(dst + 16 * 128) = t1a | (t1b << 16);
    }
  } else {
    for (int c = tid * 2; c < p.H; c += kXPrepThreads * 2) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(xr + c));
      const uint32_t hv = f16x2_rn(bf16_to_float((uint16_t)(v & 0xFFFFu)) * scl,
                                   bf16_to_float((uint16_t)(v >> 16)) * scl);
      const int kb = c / 128, half = (c % 128) / 64;
      uint8_t *dst = p.table + ((size_t)(kb * 2 + half) * p.NT + t) * 128 + (c % 64) * 2;
      *reinterpret_cast<uint32_t *>(dst) = hv;
    }
  }
}

}  // namespace moe
