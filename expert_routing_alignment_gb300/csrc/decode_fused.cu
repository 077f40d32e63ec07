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
//    top-k by redux.sync; then one warp ranks the slots of each expert in slot
//    order with match.any and scans the per-expert counts), so weight
//    streaming starts at once.  CTA 0 also writes the tables.
//  * Work unit: a tile of 16 output features of one expert.  The tiles of
//    each projection (and of the shared expert) are split evenly over the
//    CTAs.  A stage of the weight stream is a group of tiles x a part of K,
//    up to 32 KB of codes: one 3-D tensor copy per tile (cp.async.bulk.tensor;
//    16 rows x the K part as 128-byte column blocks, 128-byte swizzle, L2
//    evict-first) issued by one producer thread into a ring of stages in
//    shared memory (mbarrier completion).  The producer streams the gate+up stages and then, without
//    a pause, the down stages.
//  * Sixteen consumer warps each take one (tile, K-range) item of a stage and
//    run mma.sync m16n8k16 (f16 x f16 -> fp32) with the tile's 16 features as
//    the MMA rows and up to 8 activation rows as its columns.  Weights are
//    decoded in registers (E4M3 / E2M1 -> f16, exact; NVFP4 codes times their
//    E4M3 group scale, exact in f16); the K order inside each MMA is a fixed
//    permutation shared by both operands; the rows of a tile are taken in an
//    order that makes the swizzled shared-memory reads conflict-free.  FP8
//    block scales multiply each 64-wide K piece's fp32 partial sum.  After
//    a tile group's last K part the warps' partial tiles meet in shared
//    memory and are summed in a fixed order.
//  * gate+up: activations are the bf16 rows of x as f16 scaled by a per-row
//    power of two (exact); epilogue h = silu(g) * u.  down: the fp32 h rows
//    are split into two f16 terms (hi + lo, per-row power-of-two scale), so the
//    product keeps about 22 bits of h; epilogue y.
//  * Grid barriers (a monotonic arrival count in the workspace) separate the
//    last h write of any CTA from the first h read, and the last y write from
//    the blend.  Then every CTA blends an equal share of the M x H outputs,
//    each in slot order j = 0..k-1 plus the shared expert (times its gate
//    when gated: CTA t computes token t's gate before the barrier), and
//    writes a share of the tables.
// Every result depends only on its own row's data: the K split, the order of
// every sum and the MMA shapes are fixed by the layer's shapes, never by the
// batch.  Every wait is bounded; one that gives up sets MOE_ERR_TIMEOUT.
#include <limits.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "async.cuh"
#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kCW = 16;                   // consumer warps
constexpr int kCThreads = kCW * 32;
constexpr int kThreads = kCThreads + 32;  // + one producer warp
constexpr int kMaxN = 256;                // slots M * top_k on this path
constexpr int kMaxM = 32;
constexpr int kRows = 8;                  // activation rows per pass (the MMA's n)
constexpr int kNoKey = INT_MAX;
constexpr int kBoxBytes = 16 * 128;       // one code box: 16 rows x 128 bytes
constexpr int kSBoxBytes = 16 * 16;       // one NVFP4 scale box: 16 rows x 16 bytes

// Stage geometry of one projection (host-computed).  A half-chunk (hc) is 64
// bytes of a weight row: FP8 64 inputs, NVFP4 128.  Each consumer warp takes
// cpw half-chunks of one tile per stage; wpt warps share a tile; a stage holds
// mt tiles x kr half-chunks (kr even: whole 128-byte boxes) of every matrix;
// K is covered in nkp stages.
struct PGeo {
  int fmt, K, R, Kb, nhc, cpw, kr, wpt, mt, nkp, code_bytes, stage_bytes;
};

struct Exp {
  int fmt, I;
  const float *bscale[3];   // FP8 block scales of gate, up, down
  const float *glob[3];     // NVFP4 global scales
};

struct FusedArgs {
  Exp r, s;
  int has_shared;
  int E, H, k, BS, M, n, max_total, max_blocks, cap;
  const float *logits;
  const int32_t *ids_in;
  const float *w_in;
  const uint16_t *x;
  const uint16_t *gate_w;   // the shared expert's gate weight [H], or NULL (ungated)
  float *gate_vals;         // [M] the shared expert's gates (workspace)
  int32_t *topk_ids, *sti, *sei, *off, *ttp, *act, *act_count, *ntpp;
  float *topk_w, *h, *h_sh, *y, *y_sh;
  unsigned long long *grid_ctr;   // grid-barrier arrivals (monotonic; zero before first use)
  uint16_t *out;
  uint32_t *err;
  PGeo geo[2][2];                 // [gate+up, down][routed, shared]
  int stages, slot_bytes, xs_row_bytes;
};

// Tensor maps of the weight codes and NVFP4 group scales:
// [routed, shared][gate, up, down][codes, scales].
struct Maps {
  CUtensorMap m[2][3][2];
};

// ---------------------------------------------------------------------------
// routing of the whole batch, in shared memory
// ---------------------------------------------------------------------------

enum { kHdrA = 0, kHdrTotal, kHdrBad, kHdrInts = 8 };

struct Plan {
  int *hdr;        // A, total padded rows, out-of-range slots
  int *key;        // [n] expert id of slot i, kNoKey when out of range
  int *pos;        // [n] sorted position of slot i (token_to_perm), -1 if out of range
  float *w;        // [n] routing weight of slot i
  int *act_e;      // [n] active experts, ascending
  int *act_cnt;    // [n] rows of active expert a
  int *act_start;  // [n] first row of active expert a in rowslot
  int *act_off;    // [n] padded offset (sorted position of its row 0)
  int *rowslot;    // [n] slots grouped by expert (ascending), slot order within
};

__host__ __device__ inline size_t plan_bytes(int n) {
  return (((size_t)kHdrInts + 8 * (size_t)n) * 4 + 15) & ~(size_t)15;
}

__device__ __forceinline__ Plan carve_plan(uint8_t *base, int n) {
  Plan P;
  int *q = reinterpret_cast<int *>(base);
  P.hdr = q;
  q += kHdrInts;
  P.key = q;
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
// scratch: 3 * E ints of shared memory, free for the duration of the call.
__device__ void route_local(const Plan &P, const FusedArgs &a, int *scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int n = a.n, E = a.E;
  int *cnt = scratch, *less = scratch + E, *poff = scratch + 2 * E;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
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
  if (warp == 0) {
    // Rank of each slot among the earlier slots of its expert (slot order)
    // and the per-expert counts: 32 slots at a time, in slot order.
    int bad = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      int key = kNoKey;
      if (i < n) {
        key = P.key[i];
        if (key < 0 || key >= E) key = kNoKey;
        P.key[i] = key;
      }
      const bool real = i < n && key != kNoKey;
      bad += __popc(__ballot_sync(0xffffffffu, i < n && !real));
      const unsigned grp = __match_any_sync(0xffffffffu, key);
      const int before = __popc(grp & lanemask_lt());
      const int base = real ? cnt[key] : 0;
      __syncwarp();
      if (real) {
        P.pos[i] = base + before;   // rank for now; the sorted position below
        if (before == 0) cnt[key] = base + __popc(grp);
      }
      __syncwarp();
    }
    // Exclusive scans over the experts: rows below (less), padded rows below
    // (poff) and active experts below; lane L owns experts [L*per, L*per+per).
    const int per = (E + 31) / 32, e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int c = 0, na = 0, po = 0;
    for (int e = e0; e < e1; ++e) {
      const int v = cnt[e];
      c += v;
      na += v > 0;
      po += round_up(v, a.BS);
    }
    int ci = c, nai = na, poi = po;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int c2 = __shfl_up_sync(0xffffffffu, ci, d);
      const int n2 = __shfl_up_sync(0xffffffffu, nai, d);
      const int p2 = __shfl_up_sync(0xffffffffu, poi, d);
      if (lane >= d) {
        ci += c2;
        nai += n2;
        poi += p2;
      }
    }
    int cr = ci - c, ar = nai - na, pr = poi - po;
    for (int e = e0; e < e1; ++e) {
      const int v = cnt[e];
      less[e] = cr;
      poff[e] = pr;
      if (v > 0) {
        P.act_e[ar] = e;
        P.act_cnt[ar] = v;
        P.act_start[ar] = cr;
        P.act_off[ar] = pr;
        ++ar;
      }
      cr += v;
      pr += round_up(v, a.BS);
    }
    if (lane == 31) {
      P.hdr[kHdrA] = nai;
      P.hdr[kHdrTotal] = poi;
      P.hdr[kHdrBad] = bad;
    }
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int key = P.key[i];
    if (key == kNoKey) {
      P.pos[i] = -1;
    } else {
      const int rank = P.pos[i];
      P.pos[i] = poff[key] + rank;
      P.rowslot[less[key] + rank] = i;
    }
  }
  __syncthreads();
}

// The routing and alignment tables in the workspace, as moe_topk_softmax and
// moe_align write them; thread tid of nt (over the whole grid: every CTA
// holds the same plan).
__device__ void write_tables(const Plan &P, const FusedArgs &a, int tid, int nt) {
  const int n = a.n;
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
// the stage walk: the same sequence for the producer and the consumers
// ---------------------------------------------------------------------------

struct Stage {
  int seg;        // 0 routed, 1 shared
  int ai;         // active index (routed), -1 shared
  int e;          // expert id (0 for the shared expert)
  int x0, xn;     // activation rows [x0, x0 + xn) of the expert
  int tg, nt;     // first tile within the expert, tiles in this group
  int kp;         // K part
  bool new_rows;  // first stage of (expert, x0): stage its activation rows
};

// The CTA's stages of one projection: its share of the routed tile list (all
// active experts' tiles, expert-major), then its share of the shared expert's
// tiles; per expert, row passes of kRows rows, tile groups of mt tiles, K
// parts.  fn(Stage) is called for each.
template <class Fn>
__device__ __forceinline__ void walk(const FusedArgs &a, const Plan &P, int A, int phase, Fn &&fn) {
  for (int seg = 0; seg < 2; ++seg) {
    if (seg == 1 && !a.has_shared) break;
    const PGeo &g = a.geo[phase][seg];
    const int RT = g.R / 16;
    const long long T = seg == 0 ? (long long)A * RT : RT;
    const long long t1 = T * (blockIdx.x + 1) / gridDim.x;
    long long t = T * blockIdx.x / gridDim.x;
    while (t < t1) {
      const int ai = seg == 0 ? (int)(t / RT) : -1;
      const int et0 = (int)(t % RT);
      const long long ebase = t - et0;
      const int et1 = (int)min((long long)RT, t1 - ebase);
      const int rows = seg == 0 ? P.act_cnt[ai] : a.M;
      const int e = seg == 0 ? P.act_e[ai] : 0;
      for (int x0 = 0; x0 < rows; x0 += kRows)
        for (int tg = et0; tg < et1; tg += g.mt)
          for (int kp = 0; kp < g.nkp; ++kp) {
            Stage st;
            st.seg = seg;
            st.ai = ai;
            st.e = e;
            st.x0 = x0;
            st.xn = min(kRows, rows - x0);
            st.tg = tg;
            st.nt = min(g.mt, et1 - tg);
            st.kp = kp;
            st.new_rows = tg == et0 && kp == 0;
            fn(st);
          }
      t = ebase + et1;
    }
  }
}

// ---------------------------------------------------------------------------
// producer
// ---------------------------------------------------------------------------

// One box of a 3-D tensor map (x: bytes within a 128-byte column block,
// y: row, z: column block) into shared memory.
__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                       uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// Stream one projection's stages into the ring, continuing the stage counter
// s.  False when a wait gave up.
template <int RF, int SF>
__device__ bool produce(const FusedArgs &a, const Maps &maps, uint8_t *ring, uint64_t *full,
                        uint64_t *empty, const Plan &P, int A, int phase, int &s,
                        uint64_t pol) {
  const int kMats = phase == 0 ? 2 : 1;
  bool ok = true;
  walk(a, P, A, phase, [&](const Stage &st) {
    if (!ok) return;
    const int slot = s % a.stages;
    if (!mbar_wait(&empty[slot], ((uint32_t)(s / a.stages) & 1u) ^ 1u)) {
      ok = false;
      return;
    }
    const PGeo &g = a.geo[phase][st.seg];
    const bool f4 = (st.seg == 0 ? RF : SF) == MOE_FMT_NVFP4_G16;
    const int boxes = g.kr >> 1;
    const uint32_t bytes =
        (uint32_t)(kMats * st.nt * boxes * (kBoxBytes + (f4 ? kSBoxBytes : 0)));
    mbar_expect_tx(&full[slot], bytes);
    uint8_t *dst = ring + (size_t)slot * a.slot_bytes;
    for (int m = 0; m < kMats; ++m) {
      const int proj = phase == 0 ? m : 2;
      const CUtensorMap *cm = &maps.m[st.seg][proj][0];
      const CUtensorMap *sm = &maps.m[st.seg][proj][1];
      // one copy per tile: 16 rows x kr/2 column blocks of 128 bytes (and
      // of 16 scale bytes), column block b at b * 16 rows
      for (int i = 0; i < st.nt; ++i) {
        const int row = st.e * g.R + (st.tg + i) * 16;
        const int blk = (m * g.mt + i) * boxes;
        tma_3d(dst + (size_t)blk * kBoxBytes, cm, 0, row, st.kp * boxes, &full[slot], pol);
        if (f4)
          tma_3d(dst + g.code_bytes + (size_t)blk * kSBoxBytes, sm, 0, row, st.kp * boxes,
                 &full[slot], pol);
      }
    }
    ++s;
  });
  return ok;
}

// ---------------------------------------------------------------------------
// consumers: MMA over a stage
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

// 16-byte activation pieces per lane per half-chunk: FP8 16 inputs (2), NVFP4
// 32 inputs (4).
template <int FMT>
struct Frag {
  static constexpr int kQ = FMT == MOE_FMT_FP8_B128 ? 2 : 4;
};

// Index (in 16-byte units) of activation piece q of lane (g, t) in half-chunk
// hc.  The pieces a warp reads together are 512 contiguous bytes.
__device__ __forceinline__ int xs_unit(int hc, int q, int g, int t, int kQ) {
  return ((hc * kQ + q) * 8 + g) * 4 + t;
}

// Tile rows in MMA-row order: MMA rows 2p and 2p+1 sit in tile rows p and
// p + 4, whose 128-byte-swizzled pieces fall in opposite bank halves.
__device__ __forceinline__ int tile_row(int mrow) {
  const int lo = mrow & 7;
  return ((lo >> 1) | ((lo & 1) << 2)) + (mrow & 8);
}

// One warp's item of a stage: tile ti, half-chunks [hl0, hl0 + CPW) of the
// stage (global half-chunk hg0 + ...).  The item's weight pieces are loaded
// into registers first and the stage released (empty barrier) before any
// MMA, so the slot refills while the warp computes.  acc[m] accumulates
// matrix m's 16 x 8 tile.  FP8: sc[m][0], sc[m][1] are the block scales of
// the 128-input blocks hg0 / 2 and hg0 / 2 + 1 (CPW <= 2 spans at most two).
template <bool GU, int FMT, int CPW>
__device__ __forceinline__ void stage_mma(const uint8_t *stage, uint64_t *empty, const PGeo &g,
                                          int ti, int hl0, int hg0, const uint4 *xs_hi,
                                          const uint4 *xs_lo, bool xrow, const float (&sc)[2][2],
                                          float (&acc)[2][4]) {
  constexpr int kMats = GU ? 2 : 1;
  constexpr int kQ = Frag<FMT>::kQ;
  const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
  const int ra = tile_row(gq);   // tile rows of MMA rows gq and gq + 8: ra, ra + 8
  const int boxes = g.kr >> 1;
  uint4 wa[CPW][kMats], wb[CPW][kMats];
  uint32_t s_a[CPW][kMats], s_b[CPW][kMats];
#pragma unroll
  for (int c = 0; c < CPW; ++c) {
    const int hl = hl0 + c, b = hl >> 1, half = hl & 1;
    const int u = (((half << 2) | t) ^ (ra & 7)) << 4;   // swizzled byte offset in the row
#pragma unroll
    for (int m = 0; m < kMats; ++m) {
      const int blk = (m * g.mt + ti) * boxes + b;
      const uint8_t *box = stage + (size_t)blk * kBoxBytes;
      wa[c][m] = lds128(box + ra * 128 + u);
      wb[c][m] = lds128(box + (ra + 8) * 128 + u);
      if constexpr (FMT == MOE_FMT_NVFP4_G16) {
        const uint8_t *sbox = stage + g.code_bytes + (size_t)blk * kSBoxBytes;
        s_a[c][m] = *reinterpret_cast<const uint16_t *>(sbox + ra * 16 + half * 8 + 2 * t);
        s_b[c][m] = *reinterpret_cast<const uint16_t *>(sbox + (ra + 8) * 16 + half * 8 + 2 * t);
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);   // the stage is in registers
#pragma unroll
  for (int c = 0; c < CPW; ++c) {
    const int hg = hg0 + c;
    uint4 xh[kQ], xl[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      xh[q] = make_uint4(0, 0, 0, 0);
      xl[q] = make_uint4(0, 0, 0, 0);
      if (xrow) {
        xh[q] = xs_hi[xs_unit(hg, q, gq, t, kQ)];
        if (!GU) xl[q] = xs_lo[xs_unit(hg, q, gq, t, kQ)];
      }
    }
#pragma unroll
    for (int m = 0; m < kMats; ++m) {
      const uint32_t wa4[4] = {wa[c][m].x, wa[c][m].y, wa[c][m].z, wa[c][m].w};
      const uint32_t wb4[4] = {wb[c][m].x, wb[c][m].y, wb[c][m].z, wb[c][m].w};
      if constexpr (FMT == MOE_FMT_FP8_B128) {
        // 16 inputs per row: MMA j takes inputs 4j .. 4j+3 of the lane's span
        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a0 = e4m3x2_to_f16x2((uint16_t)(wa4[j] & 0xFFFFu));
          const uint32_t a1 = e4m3x2_to_f16x2((uint16_t)(wb4[j] & 0xFFFFu));
          const uint32_t a2 = e4m3x2_to_f16x2((uint16_t)(wa4[j] >> 16));
          const uint32_t a3 = e4m3x2_to_f16x2((uint16_t)(wb4[j] >> 16));
          const uint4 &xq = xh[j >> 1];
          mma16816(tmp, a0, a1, a2, a3, (j & 1) ? xq.z : xq.x, (j & 1) ? xq.w : xq.y);
          if (!GU) {
            const uint4 &lq = xl[j >> 1];
            mma16816(tmp, a0, a1, a2, a3, (j & 1) ? lq.z : lq.x, (j & 1) ? lq.w : lq.y);
          }
        }
        const float sk = ((hg >> 1) != (hg0 >> 1)) ? sc[m][1] : sc[m][0];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[m][r] = fmaf(tmp[r], sk, acc[m][r]);
      } else {
        // 32 inputs per row in two 16-input groups, each with its E4M3 scale
        const uint32_t sA = e4m3x2_to_f16x2((uint16_t)s_a[c][m]);
        const uint32_t sB = e4m3x2_to_f16x2((uint16_t)s_b[c][m]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t sa = prmt(sA, sA, j < 4 ? 0x1010u : 0x3232u);
          const uint32_t sb = prmt(sB, sB, j < 4 ? 0x1010u : 0x3232u);
          const int sh = (j & 1) * 16;
          const uint32_t wA = wa4[j >> 1] >> sh, wB = wb4[j >> 1] >> sh;
          const uint32_t a0 = hmul2(e2m1x2_to_f16x2(wA & 0xFFu), sa);
          const uint32_t a1 = hmul2(e2m1x2_to_f16x2(wB & 0xFFu), sb);
          const uint32_t a2 = hmul2(e2m1x2_to_f16x2((wA >> 8) & 0xFFu), sa);
          const uint32_t a3 = hmul2(e2m1x2_to_f16x2((wB >> 8) & 0xFFu), sb);
          const uint4 &xq = xh[j >> 1];
          mma16816(acc[m], a0, a1, a2, a3, (j & 1) ? xq.z : xq.x, (j & 1) ? xq.w : xq.y);
          if (!GU) {
            const uint4 &lq = xl[j >> 1];
            mma16816(acc[m], a0, a1, a2, a3, (j & 1) ? lq.z : lq.x, (j & 1) ? lq.w : lq.y);
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

struct Smem {
  uint8_t *ring;
  uint64_t *full, *empty;
  Plan P;
  uint8_t *xs;      // staged activation rows (permuted f16 pieces)
  uint32_t *xmax;   // [kRows] row |max| bits
  int *xexp;        // [kRows] row power-of-two exponents
  float4 *red;      // [2][kCW][32] partial tiles
  float *bsc;       // [2][256] FP8 block scales of the staged expert's matrices
  float *gsc;       // [4] NVFP4 global scales of the staged expert's matrices
  int *misc;        // [64] flags
};

__host__ __device__ inline size_t fixed_smem(int n, int xs_row_bytes) {
  return plan_bytes(n) + (size_t)kRows * xs_row_bytes + 2 * kRows * 4 +
         (size_t)2 * kCW * 32 * 16 + (2 * 256 + 4) * 4 + 64 * 4;
}

__device__ __forceinline__ Smem carve(uint8_t *smem, const FusedArgs &a) {
  Smem S;
  // the 128-byte swizzle of the code boxes wants 1024-byte aligned boxes
  const uint32_t base = smem_addr(smem);
  uint8_t *p = smem + ((1024u - (base & 1023u)) & 1023u);
  S.ring = p;
  p += (size_t)a.stages * a.slot_bytes;
  S.full = reinterpret_cast<uint64_t *>(p);
  S.empty = S.full + a.stages;
  p += 16 * (size_t)a.stages;
  S.P = carve_plan(p, a.n);
  p += plan_bytes(a.n);
  S.xs = p;
  p += (size_t)kRows * a.xs_row_bytes;
  S.xmax = reinterpret_cast<uint32_t *>(p);
  S.xexp = reinterpret_cast<int *>(S.xmax + kRows);
  p += 2 * kRows * 4;
  S.red = reinterpret_cast<float4 *>(p);
  p += (size_t)2 * kCW * 32 * 16;
  S.bsc = reinterpret_cast<float *>(p);
  S.gsc = S.bsc + 2 * 256;
  p += (2 * 256 + 4) * 4;
  S.misc = reinterpret_cast<int *>(p);
  return S;
}

// The power-of-two exponent s of a row whose largest |value| has exponent
// field exp_field (fp32 layout): |values| * 2^-s < 2^15, the largest in
// [2^14, 2^15).
__device__ __forceinline__ int row_shift(uint32_t exp_field) {
  const int s = (int)exp_field - 127 - 14;
  return max(-100, min(100, s));
}

// Stage activation rows [x0, x0 + xn) of the stage's expert as permuted f16
// pieces.  gate+up: bf16 x rows; down: fp32 h rows as hi + lo.  All consumer
// threads.
template <bool GU, int FMT>
__device__ void stage_rows(const FusedArgs &a, const Smem &S, const Stage &st, const PGeo &g) {
  constexpr int kQ = Frag<FMT>::kQ;
  constexpr int kMats = GU ? 2 : 1;
  const int K = g.K;
  const int tid = threadIdx.x;
  const Plan &P = S.P;
  // the expert's scales, read once here rather than per stage
  const Exp &X = st.seg == 0 ? a.r : a.s;
  if constexpr (FMT == MOE_FMT_FP8_B128) {
    const int nb = (g.R / 128) * (K / 128);   // <= 16 x 16
#pragma unroll
    for (int m = 0; m < kMats; ++m)
      for (int v = tid; v < nb; v += kCThreads)
        S.bsc[m * 256 + v] = __ldg(X.bscale[GU ? m : 2] + (size_t)st.e * nb + v);
  } else {
    if (tid < kMats) S.gsc[tid] = __ldg(X.glob[GU ? tid : 2] + st.e);
  }
  if (tid < kRows) S.xmax[tid] = 0u;
  named_sync(kCThreads);
  const int upr = K / 8;                 // 8-input units per row
  const int units = st.xn * upr;
  // pass 1: the rows' largest |value| (the loads are repeated in pass 2,
  // from L2, rather than held in registers)
  for (int v = tid; v < units; v += kCThreads) {
    const int r = v / upr, k8 = (v % upr) * 8;
    uint32_t mx = 0;
    if (GU) {
      const int tok = st.seg == 0 ? P.rowslot[P.act_start[st.ai] + st.x0 + r] / a.k : st.x0 + r;
      const uint4 q4 = __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * a.H + k8));
      const uint32_t wd[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) mx = max(mx, max((wd[q] & 0x7FFFu) << 16, wd[q] & 0x7FFF0000u));
    } else {
      const float *src = st.seg == 0 ? a.h + (size_t)(P.act_off[st.ai] + st.x0 + r) * K
                                     : a.h_sh + (size_t)(st.x0 + r) * K;
      const uint4 q0 = __ldcg(reinterpret_cast<const uint4 *>(src + k8));
      const uint4 q1 = __ldcg(reinterpret_cast<const uint4 *>(src + k8 + 4));
      const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) mx = max(mx, wd[q] & 0x7FFFFFFFu);
    }
    atomicMax(&S.xmax[r], mx);
  }
  named_sync(kCThreads);
  if (tid < st.xn) S.xexp[tid] = row_shift((S.xmax[tid] >> 23) & 0xFFu);
  named_sync(kCThreads);
  uint4 *xs_hi = reinterpret_cast<uint4 *>(S.xs);
  uint4 *xs_lo = xs_hi + (size_t)kRows * K / 8;
  for (int v = tid; v < units; v += kCThreads) {
    const int r = v / upr, k = (v % upr) * 8;
    const float m = pow2f(-S.xexp[r]);
    float f[8];
    if (GU) {
      const int tok = st.seg == 0 ? P.rowslot[P.act_start[st.ai] + st.x0 + r] / a.k : st.x0 + r;
      const uint4 q4 = __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * a.H + k));
      const uint32_t wd[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[2 * q] = __uint_as_float(wd[q] << 16) * m;
        f[2 * q + 1] = __uint_as_float(wd[q] & 0xFFFF0000u) * m;
      }
    } else {
      const float *src = st.seg == 0 ? a.h + (size_t)(P.act_off[st.ai] + st.x0 + r) * K
                                     : a.h_sh + (size_t)(st.x0 + r) * K;
      const uint4 q0 = __ldcg(reinterpret_cast<const uint4 *>(src + k));
      const uint4 q1 = __ldcg(reinterpret_cast<const uint4 *>(src + k + 4));
      const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(wd[q]) * m;
    }
    // piece (hc, q, t) of row r: 8 inputs starting at k
    const int span = 8 * kQ;                      // inputs per lane per half-chunk
    const int hc = k / (4 * span), t = (k / span) & 3, q = (k / 8) % kQ;
    const int unit = xs_unit(hc, q, r, t, kQ);
    uint4 hv;
    hv.x = pack_f16x2(f[0], f[1]);
    hv.y = pack_f16x2(f[2], f[3]);
    hv.z = pack_f16x2(f[4], f[5]);
    hv.w = pack_f16x2(f[6], f[7]);
    xs_hi[unit] = hv;
    if (!GU) {
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
      uint32_t lw[4];
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 hf = f16x2_to_float2(hw[q2]);
        lw[q2] = pack_f16x2(f[2 * q2] - hf.x, f[2 * q2 + 1] - hf.y);
      }
      xs_lo[unit] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  named_sync(kCThreads);
}

// One projection's stages on the consumer side, continuing the stage counter s.
template <bool GU, int RF, int SF>
__device__ void consume(const FusedArgs &a, const Smem &S, int A, int &s, bool &failed) {
  constexpr int kMats = GU ? 2 : 1;
  const int phase = GU ? 0 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Plan &P = S.P;
  float acc[2][4];
  int cur_ai = INT_MIN, cur_seg = -1, cur_x0 = -1;
  walk(a, P, A, phase, [&](const Stage &st) {
    const PGeo &g = a.geo[phase][st.seg];
    const int fmt = st.seg == 0 ? RF : SF;
    const Exp &X = st.seg == 0 ? a.r : a.s;
    const int slot = s % a.stages;
    const uint32_t par = (uint32_t)(s / a.stages) & 1u;
    if (st.seg != cur_seg || st.ai != cur_ai || st.x0 != cur_x0) {
      named_sync(kCThreads);   // nobody still reads the previous rows
      if (fmt == MOE_FMT_FP8_B128)
        stage_rows<GU, MOE_FMT_FP8_B128>(a, S, st, g);
      else
        stage_rows<GU, MOE_FMT_NVFP4_G16>(a, S, st, g);
      cur_seg = st.seg;
      cur_ai = st.ai;
      cur_x0 = st.x0;
    }
    if (st.kp == 0)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[m][r] = 0.f;
    const int ti = warp / g.wpt, wi = warp % g.wpt;
    const bool active = ti < st.nt;
    const int hl0 = wi * g.cpw, hg0 = st.kp * g.kr + hl0;
    float sc[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
    if (active && fmt == MOE_FMT_FP8_B128) {
      const int nkb = g.K / 128;
      const int fb = ((st.tg + ti) * 16) / 128, kb = hg0 / 2;
#pragma unroll
      for (int m = 0; m < kMats; ++m) {
        sc[m][0] = S.bsc[m * 256 + fb * nkb + kb];
        if (kb + 1 < nkb) sc[m][1] = S.bsc[m * 256 + fb * nkb + kb + 1];
      }
    }
    if (!failed && !mbar_wait(&S.full[slot], par)) {
      failed = true;
      if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
    }
    if (active && !failed) {
      uint64_t *empty = &S.empty[slot];
      const uint8_t *stage = S.ring + (size_t)slot * a.slot_bytes;
      const uint4 *xh = reinterpret_cast<const uint4 *>(S.xs);
      const uint4 *xl = xh + (size_t)kRows * g.K / 8;
      const bool xrow = (lane >> 2) < st.xn;
#define MOE_MMA(F_, C_) \
  stage_mma<GU, F_, C_>(stage, empty, g, ti, hl0, hg0, xh, xl, xrow, sc, acc)
      // gate+up items are one half-chunk of both matrices; down items one
      // or two half-chunks of one matrix (a warp's weights in registers)
      if (fmt == MOE_FMT_FP8_B128) {
        if (GU || g.cpw == 1) MOE_MMA(MOE_FMT_FP8_B128, 1);
        else MOE_MMA(MOE_FMT_FP8_B128, GU ? 1 : 2);
      } else {
        if (GU || g.cpw == 1) MOE_MMA(MOE_FMT_NVFP4_G16, 1);
        else MOE_MMA(MOE_FMT_NVFP4_G16, GU ? 1 : 2);
      }
#undef MOE_MMA
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);   // nothing of this stage for this warp
    }
    ++s;
    if (st.kp == g.nkp - 1) {
      // the group's partial tiles -> shared memory -> fixed-order sums
      named_sync(kCThreads);   // the previous group's sums are done
      if (active)
#pragma unroll
        for (int m = 0; m < kMats; ++m)
          S.red[(m * kCW + warp) * 32 + lane] =
              make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      named_sync(kCThreads);
      const float g0 = fmt == MOE_FMT_NVFP4_G16 ? S.gsc[0] : 1.f;
      const float g1 = (GU && fmt == MOE_FMT_NVFP4_G16) ? S.gsc[1] : 1.f;
      const float *red = reinterpret_cast<const float *>(S.red);
      for (int o = tid; o < st.nt * 128; o += kCThreads) {
        const int i = o >> 7, mr = (o >> 3) & 15, n = o & 7;
        if (n >= st.xn) continue;
        const int ln = 4 * (mr & 7) + (n >> 1), rg = ((mr >> 3) << 1) | (n & 1);
        float v0 = 0.f, v1 = 0.f;
        for (int w2 = 0; w2 < g.wpt; ++w2) {
          const int wv = i * g.wpt + w2;
          v0 += red[((0 * kCW + wv) * 32 + ln) * 4 + rg];
          if (GU) v1 += red[((1 * kCW + wv) * 32 + ln) * 4 + rg];
        }
        const float mx = pow2f(S.xexp[n]);
        const int feat = (st.tg + i) * 16 + tile_row(mr);
        const int row = st.x0 + n;
        if (GU) {
          const float hv = silu_f32(v0 * mx * g0) * (v1 * mx * g1);
          if (st.seg == 0)
            a.h[(size_t)(P.act_off[st.ai] + row) * X.I + feat] = hv;
          else
            a.h_sh[(size_t)row * X.I + feat] = hv;
        } else {
          const float yv = v0 * mx * g0;
          if (st.seg == 0)
            a.y[(size_t)(P.act_off[st.ai] + row) * a.H + feat] = yv;
          else
            a.y_sh[(size_t)row * a.H + feat] = yv;
        }
      }
    }
  });
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
    for (uint32_t i = 0; i < (1u << 24); ++i) {   // about a second at most
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
__global__ void __launch_bounds__(kThreads, 1)
    decode_layer_kernel(const __grid_constant__ FusedArgs a, const __grid_constant__ Maps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem S = carve(smem, a);
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
  // the ring is idle until the producer starts: routing scratch
  route_local(P, a, reinterpret_cast<int *>(S.ring));
  const int A = P.hdr[kHdrA];

  if (warp == kCW) {
    // ---------------- producer: gate+up stages, then down stages ----------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      bool ok = produce<RF, SF>(a, maps, S.ring, S.full, S.empty, P, A, 0, s, pol);
      if (ok) ok = produce<RF, SF>(a, maps, S.ring, S.full, S.empty, P, A, 1, s, pol);
      if (!ok) {
        if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
        for (int q = max(0, s - a.stages); q < s; ++q)   // the last fill of each slot lands
          (void)mbar_wait(&S.full[q % a.stages], (uint32_t)(q / a.stages) & 1u);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  int s = 0;
  bool failed = false;
  consume<true, RF, SF>(a, S, A, s, failed);
  // every h row of every CTA is written before any CTA reads one
  if (!grid_barrier(a.grid_ctr, S.misc + 32)) {
    failed = true;
    if (tid == 0 && a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
  }
  consume<false, RF, SF>(a, S, A, s, failed);
  // the shared expert's gates: token t by warp 0 of CTA t (mod the grid)
  if (a.gate_w && warp == 0)
    for (int t = blockIdx.x; t < a.M; t += gridDim.x) {
      const float g = shared_gate_warp(a.x + (size_t)t * a.H, a.gate_w, a.H);
      if (lane == 0) a.gate_vals[t] = g;
    }
  // every y row (and gate) is written before any CTA blends
  if (!grid_barrier(a.grid_ctr, S.misc + 32)) {
    failed = true;
    if (tid == 0 && a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
  }

  // ---------------- blend: this CTA's share of the M x H outputs ----------
  {
    const long long T = (long long)a.M * a.H;
    const long long o1 = T * (blockIdx.x + 1) / gridDim.x;
    for (long long o = T * blockIdx.x / gridDim.x + tid; o < o1; o += kCThreads) {
      const int tok = (int)(o / a.H), cc = (int)(o % a.H);
      const int k = a.k;
      float acc = 0.f;
      for (int j0 = 0; j0 < k; j0 += 8) {   // 8 loads in flight, then the fixed-order sum
        float yv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int jj = j0 + i;
          const int pj = jj < k ? P.pos[tok * k + jj] : -1;
          yv[i] = pj >= 0 ? __ldcg(a.y + (size_t)pj * a.H + cc) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int jj = j0 + i;
          if (jj < k && P.pos[tok * k + jj] >= 0) acc = fmaf(P.w[tok * k + jj], yv[i], acc);
        }
      }
      if (a.has_shared) {
        const float ysh = __ldcg(a.y_sh + (size_t)tok * a.H + cc);
        acc = a.gate_w ? fmaf(__ldcg(a.gate_vals + tok), ysh, acc) : acc + ysh;
      }
      a.out[(size_t)tok * a.H + cc] = float_to_bf16_rn(acc);
    }
  }
  write_tables(P, a, blockIdx.x * kCThreads + tid, gridDim.x * kCThreads);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr size_t kSmemMax = 227 * 1024;
constexpr int kStageCodeBytes = 32768;   // codes per stage

// Stage geometry of a projection with K inputs and R outputs per expert in
// format fmt, for kMats matrices per stage.
PGeo make_geo(int fmt, int K, int R, int kMats) {
  PGeo g = {};
  g.fmt = fmt;
  g.K = K;
  g.R = R;
  g.Kb = fmt == MOE_FMT_FP8_B128 ? K : K / 2;
  g.nhc = g.Kb / 64;
  // kr even (whole boxes) dividing nhc; cpw dividing kr, 1 for gate+up and
  // at most 2 for down (the item's weights stay in registers); wpt = kr / cpw
  // dividing the warp count.
  // Largest stage with at most kStageCodeBytes of codes;
  // among equals, the fewest tiles per group (a CTA's share of a projection
  // may be only a few tiles).  A function of the shapes alone: it fixes the
  // order of every sum, which must not depend on the batch.
  int best = -1, best_mt = 0;
  for (int kr = 2; kr <= g.nhc; kr += 2) {
    if (g.nhc % kr) continue;
    for (int cpw = 1; cpw <= kr && cpw <= (kMats == 2 ? 1 : 2); ++cpw) {
      if (kr % cpw) continue;
      const int wpt = kr / cpw;
      if (kCW % wpt) continue;
      const int mt = kCW / wpt;
      const int bytes = kMats * mt * kr * 1024;
      if (bytes > kStageCodeBytes || bytes < best || (bytes == best && mt >= best_mt)) continue;
      best = bytes;
      best_mt = mt;
      g.kr = kr;
      g.cpw = cpw;
    }
  }
  g.wpt = g.kr / g.cpw;
  g.mt = kCW / g.wpt;
  g.nkp = g.nhc / g.kr;
  g.code_bytes = kMats * g.mt * (g.kr / 2) * kBoxBytes;
  g.stage_bytes =
      g.code_bytes + (fmt == MOE_FMT_NVFP4_G16 ? kMats * g.mt * (g.kr / 2) * kSBoxBytes : 0);
  return g;
}

struct Shape {
  PGeo geo[2][2];
  int stages, slot_bytes, xs_row_bytes;
  size_t smem;
};

bool plan_shape(const moe_layer_desc *L, int M, int sms, Shape &sp) {
  const moe_experts &R = L->routed;
  const moe_experts *S = L->shared;
  const int n = M * L->top_k;
  if (n > kMaxN || M > kMaxM || L->top_k > 32 || sms < 1 || R.num_experts > 1024) return false;
  // one format per expert set: the nvfp4-gate-up tier runs on the staged
  // kernels, which take each projection in its own format
  if (R.fmt == MOE_FMT_NVFP4_GATE_UP || (S && S->fmt == MOE_FMT_NVFP4_GATE_UP)) return false;
  const int H = R.hidden;
  // K and R multiples of 128 in [256, 2048] (NVFP4: K of 256, so that a code
  // row is whole 128-byte boxes and a scale row whole 16-byte boxes)
  auto k_ok = [](int K, int fmt) {
    return K % 128 == 0 && K >= 256 && K <= 2048 && (fmt == MOE_FMT_FP8_B128 || K % 256 == 0);
  };
  if (!k_ok(H, R.fmt) || !k_ok(R.inter, R.fmt)) return false;
  if (S && (!k_ok(H, S->fmt) || !k_ok(S->inter, S->fmt))) return false;
  // tensor copies read 16-byte aligned tables
  auto aligned = [](const moe_experts *X) {
    if (!X) return true;
    const moe_proj *p[3] = {&X->gate, &X->up, &X->down};
    for (auto *q : p) {
      if ((uintptr_t)q->codes & 15) return false;
      if (X->fmt == MOE_FMT_NVFP4_G16 && ((uintptr_t)q->scale & 15)) return false;
    }
    return true;
  };
  if (!aligned(&R) || !aligned(S)) return false;
  const moe_experts *X[2] = {&R, S};
  int slot = 0;
  for (int seg = 0; seg < 2; ++seg) {
    if (!X[seg]) {
      sp.geo[0][seg] = sp.geo[0][0];
      sp.geo[1][seg] = sp.geo[1][0];
      continue;
    }
    sp.geo[0][seg] = make_geo(X[seg]->fmt, H, X[seg]->inter, 2);
    sp.geo[1][seg] = make_geo(X[seg]->fmt, X[seg]->inter, H, 1);
    for (int p = 0; p < 2; ++p)
      if (sp.geo[p][seg].stage_bytes > slot) slot = sp.geo[p][seg].stage_bytes;
  }
  slot = (slot + 2047) & ~2047;
  const int kd = S && S->inter > R.inter ? S->inter : R.inter;
  sp.xs_row_bytes = 2 * H > 4 * kd ? 2 * H : 4 * kd;
  const size_t fixed = fixed_smem(n, sp.xs_row_bytes) + 1024;   // + alignment slack
  if (fixed + 2 * ((size_t)slot + 16) > kSmemMax) return false;
  int ns = (int)((kSmemMax - fixed) / ((size_t)slot + 16));
  if (ns > 8) ns = 8;
  if ((size_t)ns * slot < (size_t)3 * R.num_experts * 4) return false;   // routing scratch
  sp.stages = ns;
  sp.slot_bytes = slot;
  sp.smem = (size_t)ns * slot + 16 * (size_t)ns + fixed;
  return true;
}

// cuTensorMapEncodeTiled, from the driver through the runtime (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [rows][row_bytes] u8 table seen as [row_bytes / cb][rows][cb]: column
// blocks of cb bytes (the innermost dimension), rows, column-block index; a
// box is 16 rows x nb column blocks, laid out column block after column
// block in shared memory.
int make_map(CUtensorMap *m, const void *ptr, uint64_t row_bytes, uint64_t rows, uint32_t cb,
             uint32_t nb, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return MOE_ECUDA;
  const cuuint64_t dims[3] = {cb, rows, row_bytes / cb};
  const cuuint64_t strides[2] = {row_bytes, cb};
  const cuuint32_t box[3] = {cb, 16, nb};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_EUNSUPPORTED;
}

// Tensor maps of one expert set (cached by table address and shape: encoding
// is host work that would otherwise repeat on every call).  nb[j]: column
// blocks per copy of projection j (gate, up, down).
int expert_maps(const moe_experts *X, const int (&nb)[3], CUtensorMap (&out)[3][2]) {
  struct Key {
    const void *p;
    uint64_t rb, rows;
    uint32_t cb, nb;
    bool operator==(const Key &o) const {
      return p == o.p && rb == o.rb && rows == o.rows && cb == o.cb && nb == o.nb;
    }
  };
  struct KeyHash {
    size_t operator()(const Key &k) const {
      return std::hash<const void *>()(k.p) ^ (k.rb * 0x9E3779B97F4A7C15ull) ^ (k.rows << 7) ^
             ((size_t)k.cb << 3) ^ ((size_t)k.nb << 17);
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
  const moe_proj *p[3] = {&X->gate, &X->up, &X->down};
  const int H = X->hidden, I = X->inter, E = X->num_experts;
  const bool f4 = X->fmt == MOE_FMT_NVFP4_G16;
  std::lock_guard<std::mutex> lock(mu);
  for (int j = 0; j < 3; ++j) {
    const int K = j < 2 ? H : I, R = j < 2 ? I : H;
    const Key kc = {p[j]->codes, (uint64_t)(f4 ? K / 2 : K), (uint64_t)E * R, 128,
                    (uint32_t)nb[j]};
    const Key ks = {p[j]->scale, (uint64_t)(K / 16), (uint64_t)E * R, 16, (uint32_t)nb[j]};
    for (int w = 0; w < (f4 ? 2 : 1); ++w) {
      const Key &k = w == 0 ? kc : ks;
      auto it = cache.find(k);
      if (it == cache.end()) {
        CUtensorMap m;
        const int st = make_map(&m, k.p, k.rb, k.rows, k.cb, k.nb, k.cb == 128);
        if (st) return st;
        if (cache.size() > 4096) cache.clear();
        it = cache.emplace(k, m).first;
      }
      out[j][w] = it->second;
    }
    if (!f4) out[j][1] = out[j][0];
  }
  return MOE_OK;
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
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  const int nbr[3] = {sp.geo[0][0].kr / 2, sp.geo[0][0].kr / 2, sp.geo[1][0].kr / 2};
  const int nbs[3] = {sp.geo[0][1].kr / 2, sp.geo[0][1].kr / 2, sp.geo[1][1].kr / 2};
  int st = expert_maps(&L->routed, nbr, maps.m[0]);
  if (st) return st;
  if (L->shared) {
    st = expert_maps(L->shared, nbs, maps.m[1]);
    if (st) return st;
  } else {
    memcpy(maps.m[1], maps.m[0], sizeof(maps.m[0]));
  }
  auto conv = [](const moe_experts *X) {
    Exp d = {};
    if (!X) return d;
    d.fmt = X->fmt;
    d.I = X->inter;
    const moe_proj *src[3] = {&X->gate, &X->up, &X->down};
    for (int i = 0; i < 3; ++i) {
      d.bscale[i] = reinterpret_cast<const float *>(src[i]->scale);
      d.glob[i] = src[i]->global_scale;
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
  a.gate_w = L->shared ? L->shared_gate : nullptr;
  char *base = reinterpret_cast<char *>(ws);
  a.gate_vals = reinterpret_cast<float *>(base + v.shared_gate);
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
  a.out = out;
  a.err = err;
  memcpy(a.geo, sp.geo, sizeof(a.geo));
  a.stages = sp.stages;
  a.slot_bytes = sp.slot_bytes;
  a.xs_row_bytes = sp.xs_row_bytes;
  const int rf = L->routed.fmt, sf = L->shared ? L->shared->fmt : rf;
  auto go = [&](auto kern) -> int {
    int r = ensure_max_carveout(reinterpret_cast<const void *>(kern));
    if (r) return r;
    r = ensure_smem_limit(reinterpret_cast<const void *>(kern), sp.smem);
    if (r) return r;
    // cooperative: all CTAs are co-resident, which the grid barrier needs
    return launch_pdl_coop(kern, dim3(sms), dim3(kThreads), sp.smem, stream, a, maps);
  };
  constexpr int F8 = MOE_FMT_FP8_B128, F4 = MOE_FMT_NVFP4_G16;
  if (rf == F8 && sf == F8) return go(decode_layer_kernel<F8, F8>);
  if (rf == F4 && sf == F8) return go(decode_layer_kernel<F4, F8>);
  if (rf == F8 && sf == F4) return go(decode_layer_kernel<F8, F4>);
  return go(decode_layer_kernel<F4, F4>);
}

}  // namespace moe
