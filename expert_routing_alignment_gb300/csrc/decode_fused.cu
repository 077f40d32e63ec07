// decode_fused.cu -- the decode MoE layer (M * top_k <= 256 slots) as one
// cooperative persistent kernel.
//
// What ("metrale_model_layers/layers/moe/forward_nvfp4_grouped_decode.rs",
// forward_nvfp4_grouped_decode; "fp8_moe_grouped.rs": gate+up and down over
// rows grouped by expert, each weight row read once for all rows routed to it,
// the blend through token_to_perm): route, align, gate+up with SiLU(gate)*up
// in fp32, down, and the fixed-order blend.  The results are those of
// moe_topk_softmax + moe_align + the grouped stages + moe_blend; the routing
// and alignment tables land in the workspace bit-identical to what
// moe_topk_softmax and moe_align write.
//
// How (GB300):
//  * One CTA per SM, all co-resident (cooperative launch).  Every CTA routes
//    the whole batch itself in shared memory from the router logits (warp
//    top-k, then for each slot the count of smaller expert ids and of earlier
//    equal ones: the pairwise rank of "nbxtensor/ops/moe_align.py" stage 3,
//    cheap at n <= 256), so weight streaming starts at once.  CTA 0 also
//    writes the tables.
//  * The (active expert, output feature) list -- and the shared expert's
//    features -- of each projection is split evenly over the CTAs.  A producer
//    warp streams the CTA's gate+up weight rows, then without a pause its down
//    weight rows (and NVFP4 group scales), into one shared-memory ring with
//    cp.async.bulk (mbarrier completion, L2 evict-first), so the down rows are
//    already on chip when the CTA reaches them.  In the fifteen consumer
//    warps, a group of lanes owns one output feature of the stage and deals
//    the row's 16-element units round-robin to its lanes; every unit is
//    decoded once in registers and multiplied with each activation row, the
//    unit's scale multiplies its partial sum, and an xor butterfly over the
//    group finishes the dot product.  Warps run independently through the
//    ring; they meet only when the stage's expert changes, to stage that
//    expert's activation rows (and FP8 block scales) in shared memory.
//  * gate+up: activations are the bf16 rows of x as f16 scaled by a per-row
//    power of two (taken from the row's largest |x| when staged); the
//    mixed-precision fma forms exact f16 x f16 products in fp32.  Epilogue:
//    h = silu(g) * u.
//  * A grid barrier (a monotonic arrival count in the workspace) separates the
//    last h write of any CTA from the first h read.
//  * down: activations are the fp32 h rows; weights are decoded to fp32.
//    Epilogue: y.  At its end a CTA adds, per 64-column tile, how many
//    (expert, column) pairs it wrote to that tile's counter; the CTA whose
//    addition completes a tile blends it for every token in slot order
//    j = 0..k-1 and adds the shared expert.  The counter only decides who
//    blends; the sum is the same whoever does it.
// Every wait is bounded; one that gives up sets MOE_ERR_TIMEOUT.
#include <limits.h>

#include "async.cuh"
#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kCW = 15;                   // consumer warps
constexpr int kCThreads = kCW * 32;
constexpr int kThreads = kCThreads + 32;  // + one producer warp: 16 warps, <= 128 registers
constexpr int kMaxN = 256;                // slots M * top_k on this path
constexpr int kMaxM = 32;
constexpr int kXS = 4;                    // activation rows staged in shared memory
constexpr int kBlendTile = 64;            // output columns per blend tile
constexpr int kNoKey = INT_MAX;

struct Proj {
  const uint8_t *codes;
  const void *scale;
  const float *glob;
};

struct Exp {
  int fmt, I;
  Proj gate, up, down;
};

struct FusedArgs {
  Exp r, s;
  int has_shared;
  int E, H, k, BS, M, n, max_total, max_blocks, cap;
  const float *logits;
  const int32_t *ids_in;
  const float *w_in;
  const uint16_t *x;
  int32_t *topk_ids, *sti, *sei, *off, *ttp, *act, *act_count, *ntpp;
  float *topk_w, *h, *h_sh, *y, *y_sh;
  unsigned long long *grid_ctr;   // grid-barrier arrivals (monotonic; zero before first use)
  int32_t *tile_cnt;              // [ceil(H / kBlendTile)] blend counters, zeroed each call
  uint16_t *out;
  uint32_t *err;
  int stages, slot_bytes;         // the weight ring
  int rounds[2][2];               // lane-group rounds per stage: [gate+up, down][routed, shared]
};

// ---------------------------------------------------------------------------
// routing of the whole batch, in shared memory
// ---------------------------------------------------------------------------

enum { kHdrA = 0, kHdrTotal, kHdrBad, kHdrInts = 8 };

struct Plan {
  int *hdr;        // A, total padded rows, out-of-range slots
  int *key;        // [n] expert id of slot i, kNoKey when out of range
  int *cnth;       // [n] rows of the expert if slot i is its first slot, else 0
  int *pos;        // [n] sorted position of slot i (token_to_perm), -1 if out of range
  float *w;        // [n] routing weight of slot i
  int *act_e;      // [n] active experts, ascending
  int *act_cnt;    // [n] rows of active expert a
  int *act_start;  // [n] first row of active expert a in rowslot
  int *act_off;    // [n] padded offset (sorted position of its row 0)
  int *rowslot;    // [n] slots grouped by expert (ascending), slot order within
};

__host__ __device__ inline size_t plan_bytes(int n) {
  return (((size_t)kHdrInts + 9 * (size_t)n) * 4 + 15) & ~(size_t)15;
}

__device__ __forceinline__ Plan carve_plan(uint8_t *base, int n) {
  Plan P;
  int *q = reinterpret_cast<int *>(base);
  P.hdr = q;
  q += kHdrInts;
  P.key = q;
  q += n;
  P.cnth = q;
  q += n;
  P.pos = q;
  q += n;
  P.w = reinterpret_cast<float *>(q);
  q += n;
  P.act_e = q;
  q += n;
  P.act_cnt = q;
  q += n;
  P.act_start = q;
  q += n;
  P.act_off = q;
  q += n;
  P.rowslot = q;
  return P;
}

__device__ __forceinline__ int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Route every row (top-k softmax, or the given ids and weights) and align.
__device__ void route_local(const Plan &P, const FusedArgs &a) {
  const int tid = threadIdx.x, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int n = a.n;
  if (a.logits) {
    for (int t = warp; t < a.M; t += nwarps)
      topk_softmax_row<32>(a.logits + (size_t)t * a.E, a.E, a.k, P.key + t * a.k, P.w + t * a.k);
  } else {
    for (int i = tid; i < n; i += blockDim.x) {
      P.key[i] = __ldcg(a.ids_in + i);
      P.w[i] = __ldcg(a.w_in + i);
    }
  }
  __syncthreads();
  int my = kNoKey, less = 0, eqb = 0, cnt = 0;
  if (tid < n) {
    my = P.key[tid];
    if (my < 0 || my >= a.E) my = kNoKey;
  }
  __syncthreads();
  if (tid < n) P.key[tid] = my;
  __syncthreads();
  if (tid < n) {
    for (int j = 0; j < n; ++j) {
      const int kj = P.key[j];
      less += kj < my;
      eqb += (kj == my) & (j < tid);
      cnt += kj == my;
    }
    P.cnth[tid] = (my != kNoKey && eqb == 0) ? cnt : 0;
  }
  __syncthreads();
  if (tid < n) {
    int aidx = 0, off = 0;
    for (int j = 0; j < n; ++j) {
      const int c = P.cnth[j];
      if (c > 0 && P.key[j] < my) {
        ++aidx;
        off += round_up(c, a.BS);
      }
    }
    if (my != kNoKey) {
      P.pos[tid] = off + eqb;
      P.rowslot[less + eqb] = tid;
      if (eqb == 0) {
        P.act_e[aidx] = my;
        P.act_cnt[aidx] = cnt;
        P.act_start[aidx] = less;
        P.act_off[aidx] = off;
      }
    } else {
      P.pos[tid] = -1;
    }
  }
  const int A = __syncthreads_count(tid < n && my != kNoKey && eqb == 0);
  const int bad = __syncthreads_count(tid < n && my == kNoKey);
  if (tid == 0) {
    P.hdr[kHdrA] = A;
    P.hdr[kHdrBad] = bad;
    P.hdr[kHdrTotal] = A > 0 ? P.act_off[A - 1] + round_up(P.act_cnt[A - 1], a.BS) : 0;
  }
  __syncthreads();
}

// The routing and alignment tables in the workspace, as moe_topk_softmax and
// moe_align write them.  Run by the first nt threads of the CTA.
__device__ void write_tables(const Plan &P, const FusedArgs &a, int nt) {
  const int tid = threadIdx.x, n = a.n;
  const int A = P.hdr[kHdrA], total = P.hdr[kHdrTotal];
  if (a.logits)
    for (int i = tid; i < n; i += nt) {
      a.topk_ids[i] = P.key[i];
      a.topk_w[i] = P.w[i];
    }
  for (int i = tid; i < n; i += nt) a.ttp[i] = P.pos[i];
  for (int x = tid; x < a.cap; x += nt) a.act[x] = x < A ? P.act_e[x] : -1;
  if (tid == 0) {
    *a.act_count = A;
    *a.ntpp = total;
    if (P.hdr[kHdrBad] && a.err) atomicOr(a.err, MOE_ERR_BAD_ID);
  }
  for (int e = tid; e <= a.E; e += nt) {   // padded rows of the active experts below e
    int lo = 0, hi = A;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (P.act_e[mid] < e) lo = mid + 1; else hi = mid;
    }
    a.off[e] = lo < A ? P.act_off[lo] : total;
  }
  for (int p = tid; p < a.max_total; p += nt) {   // slot at its position, else sentinel n
    int lo = 0, hi = A - 1, owner = -1;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (P.act_off[mid] <= p) {
        owner = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    int v = n;
    if (owner >= 0 && p - P.act_off[owner] < P.act_cnt[owner])
      v = P.rowslot[P.act_start[owner] + p - P.act_off[owner]];
    a.sti[p] = v;
  }
  for (int b = tid; b < a.max_blocks; b += nt) {
    const int start = b * a.BS;
    int owner = -1;
    if (start < total) {
      int lo = 0, hi = A - 1;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        if (P.act_off[mid] <= start) {
          owner = mid;
          lo = mid + 1;
        } else {
          hi = mid - 1;
        }
      }
    }
    a.sei[b] = owner >= 0 ? P.act_e[owner] : -1;
  }
}

// ---------------------------------------------------------------------------
// units of 16 weights
// ---------------------------------------------------------------------------

template <int FMT>
struct Unit {
  static constexpr int kBytes = FMT == MOE_FMT_FP8_B128 ? 16 : 8;
};

__host__ __device__ inline size_t row_bytes(int fmt, int K) {
  return fmt == MOE_FMT_FP8_B128 ? (size_t)K : (size_t)K / 2;
}

// 16 weights (one unit in shared memory) -> 8 f16x2 registers, exact.
template <int FMT>
__device__ __forceinline__ void unit_f16(const uint8_t *src, uint32_t (&wh)[8]) {
  if constexpr (FMT == MOE_FMT_FP8_B128) {
    const uint4 q = *reinterpret_cast<const uint4 *>(src);
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wh[2 * i] = e4m3x2_to_f16x2((uint16_t)(wd[i] & 0xFFFFu));
      wh[2 * i + 1] = e4m3x2_to_f16x2((uint16_t)(wd[i] >> 16));
    }
  } else {
    const uint2 q = *reinterpret_cast<const uint2 *>(src);
    const uint32_t wd[2] = {q.x, q.y};
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) wh[4 * i + b] = e2m1x2_to_f16x2((wd[i] >> (8 * b)) & 0xFFu);
  }
}

// w . x over 16 elements (x as two uint4 of f16): exact f16 x f16 products
// accumulated in fp32; even elements and odd elements in two chains, added at
// the end.
__device__ __forceinline__ float dot16_mixed(const uint32_t (&w)[8], const uint4 &x0,
                                             const uint4 &x1) {
  const uint32_t x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm("{\n\t.reg .f16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w[i]), "r"(x[i]));
  return a0 + a1;
}

// w . h over 16 elements: weights decoded to fp32, fp32 fma, even and odd
// elements in two chains.
__device__ __forceinline__ float dot16_f32(const uint32_t (&w)[8], const float4 (&hv)[4]) {
  const float h[16] = {hv[0].x, hv[0].y, hv[0].z, hv[0].w, hv[1].x, hv[1].y, hv[1].z, hv[1].w,
                       hv[2].x, hv[2].y, hv[2].z, hv[2].w, hv[3].x, hv[3].y, hv[3].z, hv[3].w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = f16x2_to_float2(w[i]);
    a0 = fmaf(f.x, h[2 * i], a0);
    a1 = fmaf(f.y, h[2 * i + 1], a1);
  }
  return a0 + a1;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

// Sum over the lg consecutive lanes of a group (xor butterfly, fixed order).
__device__ __forceinline__ float group_sum(float v, int lg) {
  for (int d = lg >> 1; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// ---------------------------------------------------------------------------
// the engine
// ---------------------------------------------------------------------------

// Lanes that share one weight row: the row's K/16 units of 16 elements are
// dealt round-robin to them (K is a multiple of 128, so K/16 is a multiple
// of 8).
__host__ __device__ inline int lanes_per_row(int K) {
  const int units = K / 16;
  return units % 32 == 0 ? 32 : units % 16 == 0 ? 16 : 8;
}

// Rows of one matrix per lane-group round: consumer warps x (32 / lanes_per_row).
__host__ __device__ inline int stage_feats(int K) { return kCW * (32 / lanes_per_row(K)); }

// A stage: features [o0, o0 + r) of one expert's projection(s).
struct Stage {
  int a, o0, r;   // active index (-1: shared expert), first feature, features
};

// The CTA's stages: its share of the routed (expert, feature) list, then its
// share of the shared expert's features.
struct Iter {
  long long f, f1, sf, sf1;
  int R, fs, fss;
  __device__ bool next(Stage &st) {
    if (f < f1) {
      st.a = (int)(f / R);
      st.o0 = (int)(f % R);
      st.r = (int)min((long long)fs, min(f1 - f, (long long)(R - st.o0)));
      f += st.r;
      return true;
    }
    if (sf < sf1) {
      st.a = -1;
      st.o0 = (int)sf;
      st.r = (int)min((long long)fss, sf1 - sf);
      sf += st.r;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ Iter make_iter(int A, int R, int Rs, int fs, int fss) {
  Iter it;
  const long long T = (long long)A * R;
  it.f = T * blockIdx.x / gridDim.x;
  it.f1 = T * (blockIdx.x + 1) / gridDim.x;
  it.sf = (long long)Rs * blockIdx.x / gridDim.x;
  it.sf1 = (long long)Rs * (blockIdx.x + 1) / gridDim.x;
  it.R = R;
  it.fs = fs;
  it.fss = fss;
  return it;
}

// One lane group's dot products for NR staged activation rows (r0 .. r0+NR)
// against weight row f of the stage (gate+up: gate row f and up row F + f).
// Lane j of the group takes units j, j + lpr, ...; per unit the weights are
// decoded once and used for every row; the unit's scale multiplies its
// partial sum; the group's lanes are then summed by an xor butterfly.  The
// order of every sum is fixed and independent of NR.
template <bool GATE_UP, int FMT, int NR>
__device__ __forceinline__ void row_pass(const uint8_t *stage, int F, int Kb, int K, int lpr,
                                         int upl, const uint8_t *xs, int r0, int f, int j,
                                         bool live, int o0, const float *bscale, float (&acc0)[4],
                                         float (&acc1)[4]) {
  const int U = K / 16;
#pragma unroll
  for (int r = 0; r < 4; ++r) acc0[r] = acc1[r] = 0.f;
  if (live) {
    const uint8_t *s16 = stage + (size_t)(GATE_UP ? 2 : 1) * F * Kb;
#pragma unroll 4
    for (int u = 0; u < upl; ++u) {
      const int c = j + u * lpr;
      uint32_t wa[8], wb[8];
      unit_f16<FMT>(stage + (size_t)f * Kb + (size_t)c * Unit<FMT>::kBytes, wa);
      float sa, sb = 0.f;
      if constexpr (FMT == MOE_FMT_FP8_B128) {
        sa = bscale[((o0 + f) / 128) * (K / 128) + c / 8];
        if (GATE_UP) sb = bscale[256 + ((o0 + f) / 128) * (K / 128) + c / 8];
      } else {
        sa = e4m3_to_float(s16[(size_t)f * (K / 16) + c]);
        if (GATE_UP) sb = e4m3_to_float(s16[(size_t)(F + f) * (K / 16) + c]);
      }
      if constexpr (GATE_UP) {
        unit_f16<FMT>(stage + (size_t)(F + f) * Kb + (size_t)c * Unit<FMT>::kBytes, wb);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const uint4 *xp = reinterpret_cast<const uint4 *>(xs) + (size_t)(r0 + r) * 2 * U + c;
          const uint4 x0 = xp[0], x1 = xp[U];
          acc0[r] = fmaf(dot16_mixed(wa, x0, x1), sa, acc0[r]);
          acc1[r] = fmaf(dot16_mixed(wb, x0, x1), sb, acc1[r]);
        }
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float4 *hp = reinterpret_cast<const float4 *>(xs) + (size_t)(r0 + r) * 4 * U + c;
          const float4 hv[4] = {hp[0], hp[U], hp[2 * U], hp[3 * U]};
          acc0[r] = fmaf(dot16_f32(wa, hv), sa, acc0[r]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    acc0[r] = group_sum(acc0[r], lpr);
    if (GATE_UP) acc1[r] = group_sum(acc1[r], lpr);
  }
}

// Shared-memory carve-up of the layer kernel.
struct Smem {
  uint8_t *ring;
  uint64_t *full, *empty;
  Plan P;
  float *bscale;    // FP8 block scales of the current expert [2][256]
  uint32_t *xmax;   // [kXS] staged-row |x| maxima
  int *xexp;        // [kXS] their f16 exponents
  int *misc;        // [64] tile counts / flags
  uint8_t *xs;      // [kXS] staged activation rows
};

__host__ __device__ inline size_t xs_bytes(int H, int kd_max) {
  const size_t g = (size_t)kXS * H * 2, d = (size_t)kXS * kd_max * 4;
  return g > d ? g : d;
}

__device__ __forceinline__ Smem carve(uint8_t *smem, const FusedArgs &a, int kd_max) {
  Smem S;
  size_t o = 0;
  S.ring = smem;
  o += (size_t)a.stages * a.slot_bytes;
  S.full = reinterpret_cast<uint64_t *>(smem + o);
  S.empty = S.full + a.stages;
  o += 16 * (size_t)a.stages;
  S.P = carve_plan(smem + o, a.n);
  o += plan_bytes(a.n);
  S.bscale = reinterpret_cast<float *>(smem + o);
  o += 2 * 256 * 4;
  S.xmax = reinterpret_cast<uint32_t *>(smem + o);
  S.xexp = reinterpret_cast<int *>(S.xmax + kXS);
  S.misc = S.xexp + kXS;
  o += (2 * kXS + 64) * 4;
  S.xs = smem + o;
  (void)kd_max;
  return S;
}

// Geometry of one phase's stage for a projection with K inputs.
struct Geo {
  int K, U, Kb, lpr, upl, rpw, fu, F;   // fu: features per lane-group round; F = rounds * fu
};

__device__ __forceinline__ Geo geo(int fmt, int K, int rounds) {
  Geo g;
  g.K = K;
  g.U = K / 16;
  g.Kb = (int)row_bytes(fmt, K);
  g.lpr = lanes_per_row(K);
  g.upl = g.U / g.lpr;
  g.rpw = 32 / g.lpr;
  g.fu = kCW * g.rpw;
  g.F = rounds * g.fu;
  return g;
}

// Producer: stream one phase's stages into the ring, continuing the stage
// counter s.  False when a wait gave up.
template <bool GATE_UP, int RF, int SF>
__device__ bool produce(const FusedArgs &a, const Smem &S, int A, int &s, uint64_t pol) {
  constexpr int kMats = GATE_UP ? 2 : 1;
  const int p = GATE_UP ? 0 : 1;
  const int Kr = GATE_UP ? a.H : a.r.I, Ks = a.has_shared ? (GATE_UP ? a.H : a.s.I) : 0;
  const Geo gr = geo(RF, Kr, a.rounds[p][0]);
  const Geo gs = geo(SF, a.has_shared ? Ks : 256, a.rounds[p][1]);
  const int R = GATE_UP ? a.r.I : a.H, Rs = a.has_shared ? (GATE_UP ? a.s.I : a.H) : 0;
  Iter it = make_iter(A, R, Rs, gr.F, gs.F);
  Stage st;
  while (it.next(st)) {
    const int slot = s % a.stages;
    if (!mbar_wait(&S.empty[slot], ((uint32_t)(s / a.stages) & 1u) ^ 1u)) return false;
    const bool sh = st.a < 0;
    const Exp &X = sh ? a.s : a.r;
    const int fmt = sh ? SF : RF;
    const Geo &g = sh ? gs : gr;
    const int e = sh ? 0 : S.P.act_e[st.a];
    const int rows = GATE_UP ? X.I : a.H;   // rows of each matrix
    const uint32_t wbytes = (uint32_t)(st.r * g.Kb);
    const uint32_t sbytes = fmt == MOE_FMT_NVFP4_G16 ? (uint32_t)(st.r * (g.K / 16)) : 0u;
    uint8_t *dst = S.ring + (size_t)slot * a.slot_bytes;
    mbar_expect_tx(&S.full[slot], kMats * (wbytes + sbytes));
#pragma unroll
    for (int m = 0; m < kMats; ++m) {
      const Proj &Pj = GATE_UP ? (m == 0 ? X.gate : X.up) : X.down;
      bulk_g2s(dst + (size_t)m * g.F * g.Kb, Pj.codes + ((size_t)e * rows + st.o0) * g.Kb,
               wbytes, &S.full[slot], pol);
      if (sbytes)
        bulk_g2s(dst + (size_t)kMats * g.F * g.Kb + (size_t)m * g.F * (g.K / 16),
                 reinterpret_cast<const uint8_t *>(Pj.scale) + ((size_t)e * rows + st.o0) * (g.K / 16),
                 sbytes, &S.full[slot], pol);
    }
    ++s;
  }
  return true;
}

// Consumers: one phase's stages, continuing the stage counter s.
template <bool GATE_UP, int RF, int SF>
__device__ void consume(const FusedArgs &a, const Smem &S, int A, int &s, bool &failed) {
  constexpr int kMats = GATE_UP ? 2 : 1;
  const int p = GATE_UP ? 0 : 1;
  const Plan &P = S.P;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Kr = GATE_UP ? a.H : a.r.I, Ks = a.has_shared ? (GATE_UP ? a.H : a.s.I) : 0;
  const Geo gr = geo(RF, Kr, a.rounds[p][0]);
  const Geo gs = geo(SF, a.has_shared ? Ks : 256, a.rounds[p][1]);
  const int R = GATE_UP ? a.r.I : a.H, Rs = a.has_shared ? (GATE_UP ? a.s.I : a.H) : 0;
  Iter it = make_iter(A, R, Rs, gr.F, gs.F);
  Stage st;
  int cur_a = INT_MIN, cur_x0 = -1;
  uint8_t *xs = S.xs;
  while (it.next(st)) {
    const int slot = s % a.stages;
    const uint32_t par = (uint32_t)(s / a.stages) & 1u;
    const bool sh = st.a < 0;
    const Exp &X = sh ? a.s : a.r;
    const int fmt = sh ? SF : RF;
    const Geo &g = sh ? gs : gr;
    const int e = sh ? 0 : P.act_e[st.a];
    const int K = g.K, U = g.U;
    const int rows = sh ? a.M : P.act_cnt[st.a];    // activation rows of this expert
    const int mrows = GATE_UP ? X.I : a.H;          // rows of each weight matrix
    const int gi = lane / g.lpr, j = lane % g.lpr;
    bool waited = false;
    for (int x0 = 0; x0 < rows; x0 += kXS) {
      const int xn = min(kXS, rows - x0);
      if (st.a != cur_a || x0 != cur_x0) {
        // stage rows x0 .. x0+xn of this expert's activations (and, on a new
        // expert, its FP8 block scales); every consumer warp reaches here
        named_sync(kCThreads);
        if (GATE_UP) {
          // bf16 x rows -> f16 * 2^-s, s from the row's largest |x|, stored
          // as [row][half][unit] x 16 bytes
          if (tid < kXS) S.xmax[tid] = 0u;
          named_sync(kCThreads);
          uint4 held[kXS];
#pragma unroll
          for (int r = 0; r < kXS; ++r) {
            const int k8 = tid * 8;
            held[r] = make_uint4(0, 0, 0, 0);
            if (r < xn && k8 < K) {
              const int tok = sh ? x0 + r : P.rowslot[P.act_start[st.a] + x0 + r] / a.k;
              held[r] = __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * a.H + k8));
            }
            const uint32_t wd[4] = {held[r].x, held[r].y, held[r].z, held[r].w};
            uint32_t mx = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = max(mx, max(wd[i] & 0x7FFFu, (wd[i] >> 16) & 0x7FFFu));
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
            if (lane == 0 && r < xn) atomicMax(&S.xmax[r], mx);
          }
          // rows longer than the thread count: the remaining chunks
          for (int k8 = (tid + kCThreads) * 8; k8 < K; k8 += kCThreads * 8)
            for (int r = 0; r < xn; ++r) {
              const int tok = sh ? x0 + r : P.rowslot[P.act_start[st.a] + x0 + r] / a.k;
              const uint4 q = __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * a.H + k8));
              const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
              uint32_t mx = 0;
              for (int i = 0; i < 4; ++i) mx = max(mx, max(wd[i] & 0x7FFFu, (wd[i] >> 16) & 0x7FFFu));
              atomicMax(&S.xmax[r], mx);
            }
          named_sync(kCThreads);
          if (tid < xn) S.xexp[tid] = max(0, (int)((S.xmax[tid] >> 7) & 0xFF) - 127 - 14);
          for (int k8 = tid * 8; k8 < K; k8 += kCThreads * 8) {
#pragma unroll
            for (int r = 0; r < kXS; ++r) {
              if (r >= xn) break;
              uint4 q;
              if (k8 == tid * 8) {
                q = held[r];
              } else {
                const int tok = sh ? x0 + r : P.rowslot[P.act_start[st.a] + x0 + r] / a.k;
                q = __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * a.H + k8));
              }
              const float m = pow2f(-max(0, (int)((S.xmax[r] >> 7) & 0xFF) - 127 - 14));
              uint4 hv;
              hv.x = pack_f16x2(__uint_as_float(q.x << 16) * m, __uint_as_float(q.x & 0xFFFF0000u) * m);
              hv.y = pack_f16x2(__uint_as_float(q.y << 16) * m, __uint_as_float(q.y & 0xFFFF0000u) * m);
              hv.z = pack_f16x2(__uint_as_float(q.z << 16) * m, __uint_as_float(q.z & 0xFFFF0000u) * m);
              hv.w = pack_f16x2(__uint_as_float(q.w << 16) * m, __uint_as_float(q.w & 0xFFFF0000u) * m);
              const int c = k8 / 16, half = (k8 / 8) & 1;
              reinterpret_cast<uint4 *>(xs)[((size_t)r * 2 + half) * U + c] = hv;
            }
          }
        } else {
          // fp32 h rows, stored as [row][quarter][unit] x 16 bytes
          const float *src = sh ? a.h_sh + (size_t)x0 * K
                                : a.h + (size_t)(P.act_off[st.a] + x0) * K;
          for (int v = tid; v < xn * (K / 4); v += kCThreads) {
            const int r = v / (K / 4), k4 = (v % (K / 4)) * 4;
            const int c = k4 / 16, qd = (k4 / 4) & 3;
            reinterpret_cast<float4 *>(xs)[((size_t)r * 4 + qd) * U + c] =
                __ldcg(reinterpret_cast<const float4 *>(src + (size_t)r * K + k4));
          }
        }
        if (fmt == MOE_FMT_FP8_B128 && st.a != cur_a) {
          const int nb = (mrows / 128) * (K / 128);
#pragma unroll
          for (int m = 0; m < kMats; ++m) {
            const Proj &Pj = GATE_UP ? (m == 0 ? X.gate : X.up) : X.down;
            const float *sp = reinterpret_cast<const float *>(Pj.scale) + (size_t)e * nb;
            for (int v = tid; v < nb; v += kCThreads) S.bscale[m * 256 + v] = __ldg(sp + v);
          }
        }
        named_sync(kCThreads);
        cur_a = st.a;
        cur_x0 = x0;
      }
      if (!waited) {
        if (!failed && !mbar_wait(&S.full[slot], par)) {
          failed = true;
          if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
        }
        waited = true;
      }
      const uint8_t *stage = S.ring + (size_t)slot * a.slot_bytes;
      const float gg = (fmt == MOE_FMT_NVFP4_G16) ? __ldg((GATE_UP ? X.gate : X.down).glob + e) : 1.f;
      const float gu = (GATE_UP && fmt == MOE_FMT_NVFP4_G16) ? __ldg(X.up.glob + e) : 1.f;
      for (int q = 0; q < g.F / g.fu; ++q) {   // lane-group rounds of the stage
        const int f = q * g.fu + warp * g.rpw + gi;   // this lane group's feature
        const bool go = f < st.r && !failed;
        if (q * g.fu >= st.r) break;
        for (int r0 = 0; r0 < xn; r0 += 4) {
          const int nr = min(4, xn - r0);
          float acc0[4], acc1[4];
#define MOE_ROWS(F_, NR)                                                                        \
  row_pass<GATE_UP, F_, NR>(stage, g.F, g.Kb, K, g.lpr, g.upl, xs, r0, f, j, go, st.o0, S.bscale, \
                            acc0, acc1)
          if (fmt == MOE_FMT_FP8_B128) {
            if (nr == 1) MOE_ROWS(MOE_FMT_FP8_B128, 1);
            else if (nr == 2) MOE_ROWS(MOE_FMT_FP8_B128, 2);
            else MOE_ROWS(MOE_FMT_FP8_B128, 4);
          } else {
            if (nr == 1) MOE_ROWS(MOE_FMT_NVFP4_G16, 1);
            else if (nr == 2) MOE_ROWS(MOE_FMT_NVFP4_G16, 2);
            else MOE_ROWS(MOE_FMT_NVFP4_G16, 4);
          }
#undef MOE_ROWS
          if (j == 0 && go) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              if (r >= nr) break;
              const int row = x0 + r0 + r;   // activation row of the expert
              if (GATE_UP) {
                const float mx = pow2f(S.xexp[r0 + r]);
                const float hv = silu_f32(acc0[r] * gg * mx) * (acc1[r] * gu * mx);
                if (sh)
                  a.h_sh[(size_t)row * X.I + st.o0 + f] = hv;
                else
                  a.h[(size_t)(P.act_off[st.a] + row) * X.I + st.o0 + f] = hv;
              } else {
                const float yv = acc0[r] * gg;
                if (sh)
                  a.y_sh[(size_t)row * a.H + st.o0 + f] = yv;
                else
                  a.y[(size_t)(P.act_off[st.a] + row) * a.H + st.o0 + f] = yv;
              }
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);   // this warp is done with the stage
    ++s;
  }
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Barrier over the consumer threads of every CTA of the (co-resident) grid.
// The counter only grows: each CTA adds one per call, so the CTAs of a call
// all see arrival numbers inside the same window [c*G, (c+1)*G).  False when
// the wait gave up.
__device__ bool grid_barrier(unsigned long long *ctr, int *flag) {
  __threadfence();
  named_sync(kCThreads);
  if (threadIdx.x == 0) {
    const unsigned long long G = gridDim.x;
    const unsigned long long v = atomicAdd(ctr, 1ull);
    const unsigned long long target = (v / G + 1) * G;
    bool ok = false;
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
      if (ld_acquire_u64(ctr) >= target) {
        ok = true;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *flag = ok;
  }
  named_sync(kCThreads);
  return *flag != 0;
}

template <int RF, int SF>
__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Smem S = carve(smem, a, 0);
  const Plan &P = S.P;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_wait();      // x and the router logits are final
  pdl_trigger();   // the next kernel on the stream may be scheduled
  if (tid == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kCW);
    }
    fence_mbar_init();
  }
  route_local(P, a);
  const int A = P.hdr[kHdrA];

  if (warp == kCW) {
    // ---------------- producer: gate+up stages, then down stages ----------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      bool ok = produce<true, RF, SF>(a, S, A, s, pol);
      if (ok) ok = produce<false, RF, SF>(a, S, A, s, pol);
      if (!ok) {
        if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
        for (int q = max(0, s - a.stages); q < s; ++q)   // the last fill of each slot lands
          (void)mbar_wait(&S.full[q % a.stages], (uint32_t)(q / a.stages) & 1u);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ntiles = (a.H + kBlendTile - 1) / kBlendTile;
  if (blockIdx.x == 0)   // read only after the grid barrier below
    for (int t = tid; t < ntiles; t += kCThreads) a.tile_cnt[t] = 0;
  int s = 0;
  bool failed = false;
  consume<true, RF, SF>(a, S, A, s, failed);
  // every h row of every CTA is written before any CTA reads one
  if (!grid_barrier(a.grid_ctr, S.misc + 32)) {
    failed = true;
    if (tid == 0 && a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
  }
  consume<false, RF, SF>(a, S, A, s, failed);

  // ---------------- blend ----------------
  int *tiles = S.misc;   // [32]
  if (A == 0 && !a.has_shared) {   // every slot out of range: the blend is zero
    const int c0 = (int)((long long)a.H * blockIdx.x / gridDim.x);
    const int c1 = (int)((long long)a.H * (blockIdx.x + 1) / gridDim.x);
    for (int t = tid; t < a.M * (c1 - c0); t += kCThreads)
      a.out[(size_t)(t / (c1 - c0)) * a.H + c0 + t % (c1 - c0)] = 0;
  } else {
    // Publish how many (expert, column) pairs of each 64-column tile this CTA
    // wrote; the CTA whose count completes a tile blends it, in slot order.
    __threadfence();          // this thread's y writes are visible device-wide
    if (tid < 32) tiles[tid] = 0;
    named_sync(kCThreads);
    if (tid == 0) {
      const int Ks = a.has_shared ? a.s.I : 256;
      Iter it2 = make_iter(A, a.H, a.has_shared ? a.H : 0,
                           geo(RF, a.r.I, a.rounds[1][0]).F, geo(SF, Ks, a.rounds[1][1]).F);
      Stage s2;
      while (it2.next(s2))
        for (int tcol = s2.o0 / kBlendTile; tcol * kBlendTile < s2.o0 + s2.r; ++tcol)
          tiles[tcol] += min(s2.o0 + s2.r, (tcol + 1) * kBlendTile) - max(s2.o0, tcol * kBlendTile);
    }
    named_sync(kCThreads);
    if (tid < ntiles) {
      const int mine = tiles[tid];
      int last = 0;
      if (mine > 0) {
        const int width = min(kBlendTile, a.H - tid * kBlendTile);
        const int target = (A + (a.has_shared ? 1 : 0)) * width;
        last = atomicAdd(&a.tile_cnt[tid], mine) + mine == target;
      }
      __threadfence();
      tiles[tid] = last;
    }
    named_sync(kCThreads);
    for (int tcol = 0; tcol < ntiles; ++tcol) {
      if (!tiles[tcol]) continue;
      const int c0 = tcol * kBlendTile, width = min(kBlendTile, a.H - c0);
      for (int t = tid; t < a.M * width; t += kCThreads) {
        const int tok = t / width, cc = c0 + t % width;
        float acc = 0.f;
        for (int jj = 0; jj < a.k; ++jj) {
          const int slot_j = tok * a.k + jj;
          const int pj = P.pos[slot_j];
          if (pj < 0) continue;
          acc = fmaf(P.w[slot_j], __ldcg(a.y + (size_t)pj * a.H + cc), acc);
        }
        if (a.has_shared) acc += __ldcg(a.y_sh + (size_t)tok * a.H + cc);
        a.out[(size_t)tok * a.H + cc] = float_to_bf16_rn(acc);
      }
    }
  }
  if (blockIdx.x == 0) write_tables(P, a, kCThreads);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr size_t kSmemMax = 227 * 1024;

struct Shape {
  int stages, slot_bytes, rounds[2][2];
  size_t smem;
};

// Bytes of one lane-group round of a stage: every lane group one row of each
// matrix (and the NVFP4 group scales of those rows).
size_t round_bytes(bool gate_up, int fmt, int K) {
  const size_t per_row = row_bytes(fmt, K) + (fmt == MOE_FMT_NVFP4_G16 ? (size_t)K / 16 : 0);
  return (size_t)(gate_up ? 2 : 1) * stage_feats(K) * per_row;
}

bool plan_shape(const moe_layer_desc *L, int M, int sms, Shape &sp) {
  const moe_experts &R = L->routed;
  const moe_experts *S = L->shared;
  const int n = M * L->top_k;
  if (n > kMaxN || M > kMaxM || L->top_k > 32 || sms < 1) return false;
  const int H = R.hidden;
  // K in [256, 2048], a multiple of 128 (at most 4 units of 16 per lane, FP8
  // block scales of at most 16 x 16 blocks); NVFP4 group scales are copied by
  // rows, so K/16 bytes must be a multiple of 16.
  auto k_ok = [](int K, int fmt) {
    return K % 128 == 0 && K >= 256 && K <= 2048 && (fmt == MOE_FMT_FP8_B128 || K % 256 == 0);
  };
  if (!k_ok(H, R.fmt) || !k_ok(R.inter, R.fmt)) return false;
  if (S && (!k_ok(H, S->fmt) || !k_ok(S->inter, S->fmt))) return false;
  if ((H + kBlendTile - 1) / kBlendTile > 32) return false;
  // NVFP4 group scales are bulk-copied: 16-byte aligned tables
  auto scales_ok = [](const moe_experts *X) {
    if (!X || X->fmt != MOE_FMT_NVFP4_G16) return true;
    return ((uintptr_t)X->gate.scale & 15) == 0 && ((uintptr_t)X->up.scale & 15) == 0 &&
           ((uintptr_t)X->down.scale & 15) == 0;
  };
  if (!scales_ok(&R) || !scales_ok(S)) return false;
  // a ring slot holds one gate+up round; down stages take as many rounds as fit
  size_t slot = round_bytes(true, R.fmt, H);
  if (S && round_bytes(true, S->fmt, H) > slot) slot = round_bytes(true, S->fmt, H);
  const size_t dr = round_bytes(false, R.fmt, R.inter);
  const size_t ds = S ? round_bytes(false, S->fmt, S->inter) : 0;
  if (dr > slot) slot = dr;
  if (ds > slot) slot = ds;
  slot = (slot + 127) & ~(size_t)127;
  sp.rounds[0][0] = sp.rounds[0][1] = 1;
  sp.rounds[1][0] = (int)(slot / dr);
  sp.rounds[1][1] = S ? (int)(slot / ds) : 1;
  const int kd_max = S && S->inter > R.inter ? S->inter : R.inter;
  const size_t fixed = plan_bytes(n) + 2 * 256 * 4 + (2 * kXS + 64) * 4 + xs_bytes(H, kd_max);
  if (fixed + 2 * (slot + 16) > kSmemMax) return false;
  int ns = (int)((kSmemMax - fixed) / (slot + 16));
  if (ns > 16) ns = 16;
  sp.stages = ns;
  sp.slot_bytes = (int)slot;
  sp.smem = (size_t)ns * slot + 16 * (size_t)ns + fixed;
  return true;
}

}  // namespace

// Whether the fused decode path serves this layer call.
bool fused_fits(const moe_layer_desc *L, int M, int sms) {
  Shape sp;
  return plan_shape(L, M, sms, sp);
}

int launch_fused(const moe_layer_desc *L, const uint16_t *x, int M, const float *logits,
                 const int32_t *ids, const float *w, uint16_t *out, void *ws,
                 const moe_workspace_view &v, uint32_t *err, void *stream) {
  const int sms = sm_count();
  Shape sp;
  if (!plan_shape(L, M, sms, sp)) return MOE_EUNSUPPORTED;
  FusedArgs a = {};
  auto conv = [](const moe_experts *X) {
    Exp d = {};
    if (!X) return d;
    d.fmt = X->fmt;
    d.I = X->inter;
    const moe_proj *src[3] = {&X->gate, &X->up, &X->down};
    Proj *dst[3] = {&d.gate, &d.up, &d.down};
    for (int i = 0; i < 3; ++i) {
      dst[i]->codes = reinterpret_cast<const uint8_t *>(src[i]->codes);
      dst[i]->scale = src[i]->scale;
      dst[i]->glob = src[i]->global_scale;
    }
    return d;
  };
  a.r = conv(&L->routed);
  a.s = conv(L->shared);
  a.has_shared = L->shared != nullptr;
  a.E = L->routed.num_experts;
  a.H = L->routed.hidden;
  a.k = L->top_k;
  a.BS = L->block_size;
  a.M = M;
  a.n = M * L->top_k;
  a.max_total = v.max_total;
  a.max_blocks = v.max_blocks;
  a.cap = v.cap;
  a.logits = logits;
  a.ids_in = ids;
  a.w_in = w;
  a.x = x;
  char *base = reinterpret_cast<char *>(ws);
  a.topk_ids = reinterpret_cast<int32_t *>(base + v.topk_ids);
  a.topk_w = reinterpret_cast<float *>(base + v.topk_w);
  a.sti = reinterpret_cast<int32_t *>(base + v.sorted_token_ids);
  a.sei = reinterpret_cast<int32_t *>(base + v.sorted_expert_ids);
  a.off = reinterpret_cast<int32_t *>(base + v.expert_offsets);
  a.ttp = reinterpret_cast<int32_t *>(base + v.token_to_perm);
  a.act = reinterpret_cast<int32_t *>(base + v.active_experts);
  a.act_count = reinterpret_cast<int32_t *>(base + v.active_count);
  a.ntpp = reinterpret_cast<int32_t *>(base + v.num_tokens_post_padded);
  a.h = reinterpret_cast<float *>(base + v.h);
  a.h_sh = reinterpret_cast<float *>(base + v.h_shared);
  a.y = reinterpret_cast<float *>(base + v.y);
  a.y_sh = reinterpret_cast<float *>(base + v.y_shared);
  a.grid_ctr = reinterpret_cast<unsigned long long *>(base + v.blend_counters);
  a.tile_cnt = reinterpret_cast<int32_t *>(base + v.blend_counters + 8);
  a.out = out;
  a.err = err;
  a.stages = sp.stages;
  a.slot_bytes = sp.slot_bytes;
  for (int p = 0; p < 2; ++p)
    for (int q = 0; q < 2; ++q) a.rounds[p][q] = sp.rounds[p][q];
  const int rf = L->routed.fmt, sf = L->shared ? L->shared->fmt : rf;
  auto go = [&](auto kern) -> int {
    int st = ensure_max_carveout(reinterpret_cast<const void *>(kern));
    if (st) return st;
    st = ensure_smem_limit(reinterpret_cast<const void *>(kern), sp.smem);
    if (st) return st;
    // cooperative: all CTAs are co-resident, which the grid barrier needs
    return launch_pdl_coop(kern, dim3(sms), dim3(kThreads), sp.smem, stream, a);
  };
  constexpr int F8 = MOE_FMT_FP8_B128, F4 = MOE_FMT_NVFP4_G16;
  if (rf == F8 && sf == F8) return go(decode_layer_kernel<F8, F8>);
  if (rf == F4 && sf == F8) return go(decode_layer_kernel<F4, F8>);
  if (rf == F8 && sf == F4) return go(decode_layer_kernel<F8, F4>);
  return go(decode_layer_kernel<F4, F4>);
}

}  // namespace moe
