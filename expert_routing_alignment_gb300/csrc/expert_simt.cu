// expert_simt.cu -- grouped expert FFN on the CUDA cores (moe_grouped_gate_up,
// moe_grouped_down, SIMT path).
//
// What it computes ("metrale_model_layers/layers/ops/fp8_moe_grouped.rs":
// moe_expert_gate_up_act_fp8_grouped and moe_expert_down_act_fp8_grouped; the
// SwiGLU epilogue of "nbxtensor/ops/moe_decode_vec.py"): a CTA owns one active
// expert and a tile of output features, streams each of those weight rows once
// and applies it to every row routed to that expert (rows live at sorted
// positions).  Grid = (feature tiles, cap [+ 1 for the shared expert]); the
// extent depends on the shape only, CTAs whose slot is not active exit.
//
// How (GB300): each warp owns one weight row per matrix; lane l reads the
// row's 16-byte chunks l, l+32, ... with L1-bypassing vector loads that are
// all issued before any arithmetic (up to 2 x 8 x 16 B in flight per lane).
// Dequantisation happens in registers: E4M3 / E2M1 pairs through the hardware
// cvt to f16x2, then to fp32; the block (FP8) or group (NVFP4) scale
// multiplies each chunk's partial dot product.  The activation rows are staged
// in shared memory as fp32 in a chunk-interleaved layout so that a warp's
// 16-byte reads of one quad of every lane's chunk are consecutive (no bank
// conflicts).  Per output the sum order is fixed (lane-local chunk order, then
// an xor butterfly), and it does not depend on how many rows an expert has:
// every row's result bits are independent of M.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGuFeatures = kWarps;        // gate+up: one feature (gate & up row) per warp
constexpr int kDnRowsPerWarp = 2;          // down: two weight rows per warp
constexpr int kDnFeatures = kWarps * kDnRowsPerWarp;
constexpr int kRowsPerPass = 4;            // activation rows staged per pass

struct ProjDev {
  const uint8_t *codes;
  const void *scale;
  const float *glob;
};

struct ExpertsDev {
  int fmt, E, H, I;
  ProjDev gate, up, down;
};

struct GroupArgs {
  ExpertsDev r, s;            // routed, shared
  int has_shared;
  int M, top_k, n, cap;
  const int32_t *off, *sti, *act, *act_count;
  const uint16_t *x;          // gate+up input [M][H] bf16
  const float *hin, *hin_sh;  // down input
  float *out, *out_sh;        // gate+up: h, h_sh; down: y, y_sh
};

template <int FMT> struct Fmt;
template <> struct Fmt<MOE_FMT_FP8_B128> {
  static constexpr int kElems = 16;     // elements per 16-byte chunk
};
template <> struct Fmt<MOE_FMT_NVFP4_G16> {
  static constexpr int kElems = 32;
};

// Row o of expert e's projection (rows x cols): its first byte.
template <int FMT>
__device__ __forceinline__ const uint8_t *row_ptr(const ProjDev &P, int e, int rows, int cols, int o) {
  const size_t row_bytes = FMT == MOE_FMT_FP8_B128 ? (size_t)cols : (size_t)cols / 2;
  return P.codes + ((size_t)e * rows + o) * row_bytes;
}

// Scale(s) of chunk c of row o: FP8 -> the 128x128 block scale; NVFP4 -> the
// two per-16 E4M3 scales of the chunk as floats.
template <int FMT>
__device__ __forceinline__ float2 chunk_scale(const ProjDev &P, int e, int rows, int cols, int o,
                                              int c) {
  if constexpr (FMT == MOE_FMT_FP8_B128) {
    const int sc = cols / 128;
    const float *s = reinterpret_cast<const float *>(P.scale) + (size_t)e * (rows / 128) * sc;
    return make_float2(__ldg(s + (o / 128) * sc + (c * 16) / 128), 0.f);
  } else {
    const uint8_t *s = reinterpret_cast<const uint8_t *>(P.scale) +
                       ((size_t)e * rows + o) * (cols / 16) + 2 * c;
    const uint32_t two = __ldg(reinterpret_cast<const unsigned short *>(s));
    const float2 f = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)two));
    return f;
  }
}

// Decode one 16-byte chunk into fp32 weights (FP8: 16, NVFP4: 32).
template <int FMT>
__device__ __forceinline__ void decode_chunk(const uint4 &q, float *w) {
  const uint32_t word[4] = {q.x, q.y, q.z, q.w};
  if constexpr (FMT == MOE_FMT_FP8_B128) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)(word[i] & 0xFFFFu)));
      const float2 b = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)(word[i] >> 16)));
      w[4 * i + 0] = a.x;
      w[4 * i + 1] = a.y;
      w[4 * i + 2] = b.x;
      w[4 * i + 3] = b.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 v = f16x2_to_float2(e2m1x2_to_f16x2((word[i] >> (8 * b)) & 0xFFu));
        w[8 * i + 2 * b + 0] = v.x;
        w[8 * i + 2 * b + 1] = v.y;
      }
    }
  }
}

// Partial dot product of one decoded chunk with activation row `xs` (fp32,
// chunk-interleaved: quad q of chunk c at float4 index q * nch + c), scaled.
template <int FMT>
__device__ __forceinline__ float chunk_dot(const float *w, const float4 *xs, int nch, int c,
                                           float2 s) {
  constexpr int Q = Fmt<FMT>::kElems / 4;
  if constexpr (FMT == MOE_FMT_FP8_B128) {
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const float4 xv = xs[q * nch + c];
      part = fmaf(w[4 * q + 0], xv.x, part);
      part = fmaf(w[4 * q + 1], xv.y, part);
      part = fmaf(w[4 * q + 2], xv.z, part);
      part = fmaf(w[4 * q + 3], xv.w, part);
    }
    return part * s.x;
  } else {
    float pa = 0.f, pb = 0.f;
#pragma unroll
    for (int q = 0; q < Q / 2; ++q) {
      const float4 xv = xs[q * nch + c];
      pa = fmaf(w[4 * q + 0], xv.x, pa);
      pa = fmaf(w[4 * q + 1], xv.y, pa);
      pa = fmaf(w[4 * q + 2], xv.z, pa);
      pa = fmaf(w[4 * q + 3], xv.w, pa);
    }
#pragma unroll
    for (int q = Q / 2; q < Q; ++q) {
      const float4 xv = xs[q * nch + c];
      pb = fmaf(w[4 * q + 0], xv.x, pb);
      pb = fmaf(w[4 * q + 1], xv.y, pb);
      pb = fmaf(w[4 * q + 2], xv.z, pb);
      pb = fmaf(w[4 * q + 3], xv.w, pb);
    }
    return fmaf(pa, s.x, pb * s.y);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Index of element k in the chunk-interleaved fp32 layout.
template <int FMT>
__device__ __forceinline__ int xs_index(int k, int nch) {
  constexpr int EPC = Fmt<FMT>::kElems;
  return (((k % EPC) >> 2) * nch + k / EPC) * 4 + (k & 3);
}

// Number of real rows at the start of positions [p0, p1) (sorted_token_ids
// below the sentinel n).  Block-wide; every thread gets the count.
__device__ __forceinline__ int real_rows(const int32_t *sti, int p0, int p1, int n) {
  int cnt = 0;
  for (int base = p0; base < p1; base += kThreads) {
    const int p = base + threadIdx.x;
    cnt += __syncthreads_count(p < p1 && __ldcg(sti + p) < n);
  }
  return cnt;
}

// ---------------------------------------------------------------------------
// gate + up
// ---------------------------------------------------------------------------

// One (expert, feature tile) item: features o_base + warp; rows `nrows` whose
// input token is tok(r) (routed: slot/top_k of position p0 + r; shared: r) and
// whose output row is out + orow(r) * I.
template <int FMT, int CPL>
__device__ __forceinline__ void gate_up_item(const ExpertsDev &X, int e, int o_base,
                                             const uint16_t *x, const int32_t *row_slots,
                                             int top_k, int nrows, float *out, float *xs_smem) {
  const int H = X.H, I = X.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int o = o_base + warp;
  const bool live = o < I;
  constexpr int EPC = Fmt<FMT>::kElems;
  const int nch = H / EPC;

  // issue every weight load of this warp's two rows first
  uint4 wg[CPL], wu[CPL];
  const uint8_t *gr = live ? row_ptr<FMT>(X.gate, e, I, H, o) : nullptr;
  const uint8_t *ur = live ? row_ptr<FMT>(X.up, e, I, H, o) : nullptr;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane + 32 * j;
    if (live && c < nch) {
      wg[j] = ld_stream16(gr + (size_t)c * 16);
      wu[j] = ld_stream16(ur + (size_t)c * 16);
    } else {
      wg[j] = make_uint4(0, 0, 0, 0);
      wu[j] = make_uint4(0, 0, 0, 0);
    }
  }
  float2 sg[CPL], su[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane + 32 * j;
    sg[j] = su[j] = make_float2(0.f, 0.f);
    if (live && c < nch) {
      sg[j] = chunk_scale<FMT>(X.gate, e, I, H, o, c);
      su[j] = chunk_scale<FMT>(X.up, e, I, H, o, c);
    }
  }
  const float gg = (FMT == MOE_FMT_NVFP4_G16 && live) ? __ldg(X.gate.glob + e) : 1.f;
  const float gu = (FMT == MOE_FMT_NVFP4_G16 && live) ? __ldg(X.up.glob + e) : 1.f;

  for (int r0 = 0; r0 < nrows; r0 += kRowsPerPass) {
    const int rows = min(kRowsPerPass, nrows - r0);
    __syncthreads();   // previous pass done with xs
    // stage `rows` activation rows: bf16 -> fp32, chunk-interleaved
    for (int idx = threadIdx.x; idx < rows * (H / 8); idx += kThreads) {
      const int r = idx / (H / 8);
      const int k = (idx % (H / 8)) * 8;
      const int tok = row_slots ? __ldcg(row_slots + r0 + r) / top_k : r0 + r;
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)tok * H + k));
      float *dst = xs_smem + (size_t)r * H;
      // k is a multiple of 8: two whole quads of the interleaved layout
      *reinterpret_cast<float4 *>(dst + xs_index<FMT>(k, nch)) =
          make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                      __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
      *reinterpret_cast<float4 *>(dst + xs_index<FMT>(k + 4, nch)) =
          make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                      __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
    }
    __syncthreads();

    float ag[kRowsPerPass], au[kRowsPerPass];
#pragma unroll
    for (int r = 0; r < kRowsPerPass; ++r) ag[r] = au[r] = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      if (c < nch) {
        float w[EPC];
        decode_chunk<FMT>(wg[j], w);
#pragma unroll
        for (int r = 0; r < kRowsPerPass; ++r)
          if (r < rows)
            ag[r] += chunk_dot<FMT>(w, reinterpret_cast<const float4 *>(xs_smem + (size_t)r * H),
                                    nch, c, sg[j]);
        decode_chunk<FMT>(wu[j], w);
#pragma unroll
        for (int r = 0; r < kRowsPerPass; ++r)
          if (r < rows)
            au[r] += chunk_dot<FMT>(w, reinterpret_cast<const float4 *>(xs_smem + (size_t)r * H),
                                    nch, c, su[j]);
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerPass; ++r) {
      if (r < rows) {
        const float g = warp_sum(ag[r]) * gg;
        const float u = warp_sum(au[r]) * gu;
        if (live && lane == 0) out[(size_t)(r0 + r) * I + o] = silu_f32(g) * u;
      }
    }
  }
}

template <int RFMT, int SFMT, int CPL>
__global__ void __launch_bounds__(kThreads) gate_up_kernel(GroupArgs a) {
  extern __shared__ float4 smem4[];
  float *xs = reinterpret_cast<float *>(smem4);
  pdl_wait();
  pdl_trigger();
  const int slot = blockIdx.y;
  if (slot < a.cap) {
    if (slot >= __ldcg(a.act_count)) return;
    const int e = __ldcg(a.act + slot);
    const int o_base = blockIdx.x * kGuFeatures;
    if (o_base >= a.r.I) return;
    const int p0 = __ldcg(a.off + e), p1 = __ldcg(a.off + e + 1);
    const int nrows = real_rows(a.sti, p0, p1, a.n);
    gate_up_item<RFMT, CPL>(a.r, e, o_base, a.x, a.sti + p0, a.top_k, nrows,
                            a.out + (size_t)p0 * a.r.I, xs);
  } else {
    const int o_base = blockIdx.x * kGuFeatures;
    if (o_base >= a.s.I) return;
    gate_up_item<SFMT, CPL>(a.s, 0, o_base, a.x, nullptr, 1, a.M, a.out_sh, xs);
  }
}

// ---------------------------------------------------------------------------
// down
// ---------------------------------------------------------------------------

template <int FMT, int CPL>
__device__ __forceinline__ void down_item(const ExpertsDev &X, int e, int c_base, const float *hin,
                                          int nrows, float *out, float *xs_smem) {
  const int H = X.H, I = X.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int EPC = Fmt<FMT>::kElems;
  constexpr int RW = kDnRowsPerWarp;
  const int nch = I / EPC;

  uint4 wd[RW][CPL];
  float2 sd[RW][CPL];
  float gd[RW];
#pragma unroll
  for (int q = 0; q < RW; ++q) {
    const int c_out = c_base + warp * RW + q;
    const bool live = c_out < H;
    const uint8_t *dr = live ? row_ptr<FMT>(X.down, e, H, I, c_out) : nullptr;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      wd[q][j] = (live && c < nch) ? ld_stream16(dr + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int q = 0; q < RW; ++q) {
    const int c_out = c_base + warp * RW + q;
    const bool live = c_out < H;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      sd[q][j] = (live && c < nch) ? chunk_scale<FMT>(X.down, e, H, I, c_out, c)
                                   : make_float2(0.f, 0.f);
    }
    gd[q] = (FMT == MOE_FMT_NVFP4_G16 && live) ? __ldg(X.down.glob + e) : 1.f;
  }

  for (int r0 = 0; r0 < nrows; r0 += kRowsPerPass) {
    const int rows = min(kRowsPerPass, nrows - r0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * (I / 4); idx += kThreads) {
      const int r = idx / (I / 4);
      const int k = (idx % (I / 4)) * 4;
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(hin + (size_t)(r0 + r) * I + k));
      float *dst = xs_smem + (size_t)r * I;
      // k is a multiple of 4: the quad lands whole in the interleaved layout
      *reinterpret_cast<float4 *>(dst + xs_index<FMT>(k, nch)) = v;
    }
    __syncthreads();

    float acc[RW][kRowsPerPass];
#pragma unroll
    for (int q = 0; q < RW; ++q)
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r) acc[q][r] = 0.f;
#pragma unroll
    for (int q = 0; q < RW; ++q) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
        if (c < nch) {
          float w[EPC];
          decode_chunk<FMT>(wd[q][j], w);
#pragma unroll
          for (int r = 0; r < kRowsPerPass; ++r)
            if (r < rows)
              acc[q][r] += chunk_dot<FMT>(
                  w, reinterpret_cast<const float4 *>(xs_smem + (size_t)r * I), nch, c, sd[q][j]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < RW; ++q) {
      const int c_out = c_base + warp * RW + q;
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r) {
        if (r < rows) {
          const float v = warp_sum(acc[q][r]) * gd[q];
          if (c_out < H && lane == 0) out[(size_t)(r0 + r) * H + c_out] = v;
        }
      }
    }
  }
}

template <int RFMT, int SFMT, int CPL>
__global__ void __launch_bounds__(kThreads) down_kernel(GroupArgs a) {
  extern __shared__ float4 smem4[];
  float *xs = reinterpret_cast<float *>(smem4);
  pdl_wait();
  pdl_trigger();
  const int slot = blockIdx.y;
  const int c_base = blockIdx.x * kDnFeatures;
  if (slot < a.cap) {
    if (slot >= __ldcg(a.act_count)) return;
    const int e = __ldcg(a.act + slot);
    const int p0 = __ldcg(a.off + e), p1 = __ldcg(a.off + e + 1);
    const int nrows = real_rows(a.sti, p0, p1, a.n);
    down_item<RFMT, CPL>(a.r, e, c_base, a.hin + (size_t)p0 * a.r.I, nrows,
                         a.out + (size_t)p0 * a.r.H, xs);
  } else {
    down_item<SFMT, CPL>(a.s, 0, c_base, a.hin_sh, a.M, a.out_sh, xs);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

int chunks_per_lane(int fmt, int K) {
  const int epc = fmt == MOE_FMT_FP8_B128 ? 16 : 32;
  return (K / epc + 31) / 32;
}

int cpl_bucket(int need) {
  if (need <= 1) return 1;
  if (need <= 2) return 2;
  if (need <= 4) return 4;
  if (need <= 8) return 8;
  return 0;
}

template <int RFMT, int SFMT>
int launch_gate_up_fmt(const GroupArgs &a, int cpl, void *stream) {
  const int feats = a.has_shared ? max(a.r.I, a.s.I) : a.r.I;
  dim3 grid((feats + kGuFeatures - 1) / kGuFeatures, a.cap + (a.has_shared ? 1 : 0));
  const size_t smem = (size_t)kRowsPerPass * a.r.H * sizeof(float);
  auto run = [&](auto kern) -> int {
    const int st = ensure_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (st) return st;
    return launch_pdl(kern, grid, dim3(kThreads), smem, stream, a);
  };
  switch (cpl) {
    case 1: return run(gate_up_kernel<RFMT, SFMT, 1>);
    case 2: return run(gate_up_kernel<RFMT, SFMT, 2>);
    case 4: return run(gate_up_kernel<RFMT, SFMT, 4>);
    case 8: return run(gate_up_kernel<RFMT, SFMT, 8>);
  }
  return MOE_EUNSUPPORTED;
}

template <int RFMT, int SFMT>
int launch_down_fmt(const GroupArgs &a, int cpl, void *stream) {
  dim3 grid((a.r.H + kDnFeatures - 1) / kDnFeatures, a.cap + (a.has_shared ? 1 : 0));
  const int kmax = a.has_shared ? max(a.r.I, a.s.I) : a.r.I;
  const size_t smem = (size_t)kRowsPerPass * kmax * sizeof(float);
  auto run = [&](auto kern) -> int {
    const int st = ensure_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (st) return st;
    return launch_pdl(kern, grid, dim3(kThreads), smem, stream, a);
  };
  switch (cpl) {
    case 1: return run(down_kernel<RFMT, SFMT, 1>);
    case 2: return run(down_kernel<RFMT, SFMT, 2>);
    case 4: return run(down_kernel<RFMT, SFMT, 4>);
    case 8: return run(down_kernel<RFMT, SFMT, 8>);
  }
  return MOE_EUNSUPPORTED;
}

}  // namespace

// Validation shared with the layer: 0 = ok.
int validate_experts(const moe_experts *X, bool shared) {
  if (!X) return MOE_EINVAL;
  if (X->fmt != MOE_FMT_FP8_B128 && X->fmt != MOE_FMT_NVFP4_G16 &&
      X->fmt != MOE_FMT_NVFP4_GATE_UP)
    return MOE_EINVAL;
  if (X->num_experts < 1 || X->hidden < 1 || X->inter < 1) return MOE_EINVAL;
  if (shared && X->num_experts != 1) return MOE_EINVAL;
  if (X->num_experts > MOE_MAX_EXPERTS) return MOE_EUNSUPPORTED;
  const moe_proj *P[3] = {&X->gate, &X->up, &X->down};
  for (int j = 0; j < 3; ++j) {
    const moe_proj *p = P[j];
    const int f = proj_fmt(X->fmt, j);
    if (!p->codes || !p->scale) return MOE_EINVAL;
    if (f == MOE_FMT_NVFP4_G16 && !p->global_scale) return MOE_EINVAL;
    if (((uintptr_t)p->codes & 15) != 0) return MOE_EINVAL;
    if (f == MOE_FMT_NVFP4_G16 && ((uintptr_t)p->scale & 1) != 0) return MOE_EINVAL;
    if (f == MOE_FMT_FP8_B128 && ((uintptr_t)p->scale & 3) != 0) return MOE_EINVAL;
  }
  // FP8 projections need 128-wide blocks on both sides, NVFP4 ones 32
  const int fg = proj_fmt(X->fmt, 0), fd = proj_fmt(X->fmt, 2);
  const int qh = (fg == MOE_FMT_FP8_B128 || fd == MOE_FMT_FP8_B128) ? 128 : 32;
  if (X->hidden % qh || X->inter % qh) return MOE_EUNSUPPORTED;
  if (cpl_bucket(chunks_per_lane(fg, X->hidden)) == 0 ||
      cpl_bucket(chunks_per_lane(fd, X->inter)) == 0)
    return MOE_EUNSUPPORTED;
  if ((size_t)kRowsPerPass * (X->hidden > X->inter ? X->hidden : X->inter) * 4 > 200 * 1024)
    return MOE_EUNSUPPORTED;
  return MOE_OK;
}

static ExpertsDev to_dev(const moe_experts *X) {
  ExpertsDev d = {};
  if (!X) return d;
  d.fmt = X->fmt;
  d.E = X->num_experts;
  d.H = X->hidden;
  d.I = X->inter;
  const moe_proj *src[3] = {&X->gate, &X->up, &X->down};
  ProjDev *dst[3] = {&d.gate, &d.up, &d.down};
  for (int i = 0; i < 3; ++i) {
    dst[i]->codes = reinterpret_cast<const uint8_t *>(src[i]->codes);
    dst[i]->scale = src[i]->scale;
    dst[i]->glob = src[i]->global_scale;
  }
  return d;
}

static int prepare(const moe_experts *routed, const moe_experts *shared, int M, int top_k,
                   const int32_t *off, const int32_t *sti, const int32_t *act,
                   const int32_t *act_count, int path, GroupArgs &a) {
  int st = validate_experts(routed, false);
  if (st) return st;
  if (shared) {
    st = validate_experts(shared, true);
    if (st) return st;
    if (shared->hidden != routed->hidden) return MOE_EINVAL;
  }
  if (M < 1 || top_k < 1 || top_k > routed->num_experts) return MOE_EINVAL;
  if (M > MOE_MAX_ROWS) return MOE_EUNSUPPORTED;
  if (path != MOE_PATH_AUTO && path != MOE_PATH_SIMT && path != MOE_PATH_TC) return MOE_EINVAL;
  if (!off || !sti || !act || !act_count) return MOE_EINVAL;
  a = GroupArgs{};
  a.r = to_dev(routed);
  a.s = to_dev(shared);
  a.has_shared = shared != nullptr;
  a.M = M;
  a.top_k = top_k;
  a.n = M * top_k;
  a.cap = a.n < routed->num_experts ? a.n : routed->num_experts;
  a.off = off;
  a.sti = sti;
  a.act = act;
  a.act_count = act_count;
  return MOE_OK;
}

#define MOE_DISPATCH_FMT(RF, SF, FN, ...)                                              \
  ((RF) == MOE_FMT_FP8_B128                                                           \
       ? ((SF) == MOE_FMT_NVFP4_G16 ? FN<MOE_FMT_FP8_B128, MOE_FMT_NVFP4_G16>(__VA_ARGS__) \
                                    : FN<MOE_FMT_FP8_B128, MOE_FMT_FP8_B128>(__VA_ARGS__))  \
       : ((SF) == MOE_FMT_FP8_B128 ? FN<MOE_FMT_NVFP4_G16, MOE_FMT_FP8_B128>(__VA_ARGS__)  \
                                   : FN<MOE_FMT_NVFP4_G16, MOE_FMT_NVFP4_G16>(__VA_ARGS__)))

int simt_gate_up(const moe_experts *routed, const moe_experts *shared, const uint16_t *x, int M,
                 int top_k, const int32_t *off, const int32_t *sti, const int32_t *act,
                 const int32_t *act_count, float *h, float *h_sh, void *stream) {
  GroupArgs a;
  int st = prepare(routed, shared, M, top_k, off, sti, act, act_count, MOE_PATH_SIMT, a);
  if (st) return st;
  if (!x || !h || (shared && !h_sh)) return MOE_EINVAL;
  a.x = x;
  a.out = h;
  a.out_sh = h_sh;
  const int rf = proj_fmt(routed->fmt, 0);
  const int sf = shared ? proj_fmt(shared->fmt, 0) : rf;
  int need = chunks_per_lane(rf, routed->hidden);
  if (shared) need = max(need, chunks_per_lane(sf, shared->hidden));
  return MOE_DISPATCH_FMT(rf, sf, launch_gate_up_fmt, a, cpl_bucket(need), stream);
}

int simt_down(const moe_experts *routed, const moe_experts *shared, const float *h,
              const float *h_sh, int M, int top_k, const int32_t *off, const int32_t *sti,
              const int32_t *act, const int32_t *act_count, float *y, float *y_sh, void *stream) {
  GroupArgs a;
  int st = prepare(routed, shared, M, top_k, off, sti, act, act_count, MOE_PATH_SIMT, a);
  if (st) return st;
  if (!h || !y || (shared && (!h_sh || !y_sh))) return MOE_EINVAL;
  a.hin = h;
  a.hin_sh = h_sh;
  a.out = y;
  a.out_sh = y_sh;
  const int rf = proj_fmt(routed->fmt, 2);
  const int sf = shared ? proj_fmt(shared->fmt, 2) : rf;
  int need = chunks_per_lane(rf, routed->inter);
  if (shared) need = max(need, chunks_per_lane(sf, shared->inter));
  return MOE_DISPATCH_FMT(rf, sf, launch_down_fmt, a, cpl_bucket(need), stream);
}

}  // namespace moe
