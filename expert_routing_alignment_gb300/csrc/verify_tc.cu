// verify_tc.cu -- the grouped expert FFN of the decode MoE layer on the
// tensor cores (tcgen05 MMA with TMEM accumulators) for FP8 experts: decode
// batches (a token form up to 16 rows), the M = 128 verify batch and prefill
// batches up to 4096 rows.
//
// What it computes is the same as the CUDA-core kernels: for every active
// expert e and every real sorted position p of its run, token t,
//   h[p] = silu(Wg[e] . x[t]) * (Wu[e] . x[t])        (fp32)
//   y[p] = Wd[e] . h[p]                                (fp32)
// with w = e4m3(code) * scale[o/128][k/128] ("fp8_moe_grouped.rs",
// moe_expert_gate_up_act_fp8_grouped / moe_expert_down_act_fp8_grouped and
// the tensor-core twins of "metrale_model_layers/layers/ops/
// fp8_moe_grouped.rs"; the SwiGLU product of "moe_decode_vec.py").
//
// How, on sm_103a:
//  * Swap-AB.  A weight tile of 128 output rows is the MMA's M side; the
//    expert's token rows (padded to 16, at most 64 per item) are its N side,
//    so a ragged expert costs MMA work in proportion to its rows.
//  * The E4M3 codes go to the tensor cores as they are (kind::f8f6f4, no
//    dequantised copy).  The activation side is split into E4M3 terms whose
//    sum is the value: x (bf16, 8 significant bits) = t0 + t1 exactly after a
//    power-of-two row scale; h (fp32) = t0 + t1 + t2 to about 2^-12 relative
//    per element, with a power-of-two scale per (row, 128-column block).
//  * Block scales are applied exactly where they change: every 128-wide k
//    block is accumulated alone in TMEM, then read into registers and added
//    in fp32 times its scale (fp32 promotion of the per-block partial).
//  * One cooperative persistent kernel, one CTA per SM, warp-specialised:
//    warp 0 streams weight tiles (TMA, 128x128-byte boxes, 128-byte swizzle)
//    and activation terms into a byte ring of variable-size stages; warp 1
//    issues the MMAs from one thread; 16 warps promote, finish h (SiLU
//    product, the three terms of the down projection's input) or y.
//    Items are (expert row tile, 128-row gate+up tile) then (expert row
//    tile, pair of 128-row down tiles), taken in that order from a grid-wide
//    counter; a down item waits (bounded) until every gate+up item of its
//    expert has published its h terms through a per-expert counter.
//  * Token form (up to 16 rows): the gate+up MMAs take the 16 token columns
//    of a per-token x-term table that the alignment launch wrote, items are
//    16-row tiles, and one promotion group works while a second stages the
//    next item's scales, tokens and h scales.
//  * Every wait gives up after about two seconds with MOE_ERR_TIMEOUT; the
//    CTA then stops issuing, drains its copies and MMAs and frees its TMEM.
#include <mutex>
#include <unordered_map>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kEpiWarps = 16;
constexpr int kWarps = 2 + kEpiWarps;
constexpr int kThreads = kWarps * 32;          // 576
constexpr int kEpiThreads = kEpiWarps * 32;    // 512
constexpr int kRecs = 8;                       // stage records (ring slots in flight)
constexpr int kAccs = 32;                      // k-block completion barriers
constexpr int kTfree = 16;                     // per-stage TMEM release barriers
constexpr int kIQ = 32;                        // item queue (copy thread -> MMA, promotion)
constexpr int kRowTile = 64;                   // token rows per item (MMA N <= 64)
constexpr int kTokMax = 16;                    // batches up to 16 rows: token columns
constexpr int kXTerms = 2, kHTerms = 3;
constexpr int kMaxKB = 64;                     // k blocks of 128 (H <= 8192)
constexpr int kMaxKBd = 32;                    // down k blocks (I <= 4096)
constexpr uint32_t kTmemCols = 512;            // the circular accumulator range

struct TcArgs {
  int M, k, n, E, H, I, cap, max_total;
  // Token-column form (M <= 16): the gate+up MMAs take all 16 token columns
  // of a per-token x-term table instead of the item's rows, items are 16-row
  // tiles, and no grid barrier precedes the first copies.
  int tok;
  int row_tile;                              // rows per item: 16 (token form) or 64
  const uint16_t *x;
  const float *w;                            // [n] routing weight of each slot
  const int32_t *ttp, *act_count;            // the alignment's tables
  const int32_t *sti;                        // sorted_token_ids
  const int4 *items;                         // [cap] {offset, expert, slot count, 0}
  uint16_t *out;                             // [M][H] bf16
  const float *sg, *su, *sd;                 // block scales [E][R/128][K/128]
  uint8_t *xq;                               // x terms [2][max_total][H] E4M3 by sorted row,
                                             // or (token form) [H/128][2][16][128] by token
  float *xs;                                 // 2^-s of each x row [max_total] (token form: [16])
  uint8_t *hq;                               // h terms [3][max_total][I] E4M3
  float *hs;                                 // 2^-s per (row, 128-block) [max_total][I/128]
  float *h, *y;                              // [max_total][I], [max_total][H]
  int *done;                                 // [cap] finished gate+up items per active expert
  int *work;                                 // [1] next item to take (zero between calls)
  unsigned long long *grid_ctr;
  uint32_t *err;
  uint32_t ring_bytes;
};

// Weight maps: 3-D {128, E*R rows, K/128 column blocks}, box {128, 128, nb}
// for nb = 1, 2 (w[projection][nb-1]).  Term maps: 3-D {K bytes, max_total
// rows, terms}, box {128, 16 << b, terms} for b = 0..2.
struct TcMaps {
  CUtensorMap w[3][2];
  CUtensorMap xq[3], hq[3];
  CUtensorMap xt;   // token form: {128, 16 tokens, 2 * H/128}, box {128, 16, 2}
};

struct Smem {
  uint8_t *ring;
  uint64_t *full, *accf, *tfree, *iqbar, *drain;
  volatile int *iq;    // [kIQ] the CTA's items in the order it takes them
  uint32_t *rec;       // [kRecs] byte offset of each stage in the ring
  uint32_t *rlen;      // [kRecs] its size
  uint32_t *trec;      // [kRecs] its accumulators: TMEM column | count << 16
  int *twait;          // [kRecs] the stage whose TMEM release it waits for (-1: none)
  int *kend;           // [kRecs] the stage's last k block (its MMAs' completion frees the stage)
  volatile int *misc;  // [0] failed, [1] TMEM base, [2] active count, [3] row tiles
  float *sc;           // [2][kMaxKB] weight block scales of the current item
  float *cs;           // [I/128][row tile] per-row factors of the current item
  int *tokrow;         // [kRowTile] token form: each row's token
  float *xtok;         // [kTokMax] token form: 2^-s of each token's x row
  uint32_t *red;       // [4 groups][4 quadrants][16] column maxima
  int *rtp;            // [cap + 1] row-tile prefix over the active list
  int2 *info;          // [cap] {offset, expert | rows << 16}
  // token form: a second buffer of the per-item arrays above (group 1 stages
  // the next item into one while group 0 works on the other), the item of
  // each buffer, and their handover barriers
  float *sc2, *cs2;
  int *tok2;
  volatile int *slot;  // [2]
  uint64_t *staged, *consumed;   // [2] each
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

// Fixed shared memory beside the ring: barriers, records, the item queue,
// scales, the per-row factors of one item, the column maxima, the row tokens
// and the active table.  (A ring of exactly three 72 KB decode stages was
// measured slower than the two stages this leaves room for.)
__host__ __device__ inline size_t fixed_bytes(int cap, int KBd, int RT) {
  (void)KBd;
  size_t b = 0;
  if (RT == 16)   // the token form's second buffers and handover barriers
    b += al16(4 * 2 * kMaxKB) + al16(4 * kMaxKBd * 16) + al16(4 * 16) + al16(4 * 2) +
         al16(8 * 4);
  b += al16(8 * (kRecs + kAccs + kTfree + kIQ + 1));
  b += 5 * al16(4 * kRecs) + al16(4 * kIQ) + al16(4 * 16);
  b += al16(4 * 2 * kMaxKB) + al16(4 * kMaxKBd * RT) + al16(4 * 4 * 4 * 16);
  b += al16(4 * kRowTile) + al16(4 * kTokMax);
  b += al16(4 * ((size_t)cap + 1)) + al16(8 * (size_t)cap);
  return b;
}

__device__ Smem carve(uint8_t *base, const TcArgs &a) {
  Smem S;
  S.ring = base;
  uint8_t *p = base + a.ring_bytes;
  auto take = [&](size_t bytes) {
    uint8_t *r = p;
    p += al16(bytes);
    return r;
  };
  uint64_t *bars = reinterpret_cast<uint64_t *>(take(8 * (kRecs + kAccs + kTfree + kIQ + 1)));
  S.full = bars;
  S.accf = bars + kRecs;
  S.tfree = bars + kRecs + kAccs;
  S.iqbar = bars + kRecs + kAccs + kTfree;
  S.drain = bars + kRecs + kAccs + kTfree + kIQ;
  S.rec = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.rlen = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.trec = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.twait = reinterpret_cast<int *>(take(4 * kRecs));
  S.kend = reinterpret_cast<int *>(take(4 * kRecs));
  S.iq = reinterpret_cast<volatile int *>(take(4 * kIQ));
  S.misc = reinterpret_cast<volatile int *>(take(4 * 16));
  S.sc = reinterpret_cast<float *>(take(4 * 2 * kMaxKB));
  S.cs = reinterpret_cast<float *>(take(4 * (size_t)(a.I / 128) * a.row_tile));
  S.tokrow = reinterpret_cast<int *>(take(4 * kRowTile));
  S.xtok = reinterpret_cast<float *>(take(4 * kTokMax));
  S.red = reinterpret_cast<uint32_t *>(take(4 * 4 * 4 * 16));
  S.rtp = reinterpret_cast<int *>(take(4 * ((size_t)a.cap + 1)));
  S.info = reinterpret_cast<int2 *>(take(8 * (size_t)a.cap));
  if (a.tok) {
    S.sc2 = reinterpret_cast<float *>(take(4 * 2 * kMaxKB));
    S.cs2 = reinterpret_cast<float *>(take(4 * (size_t)(a.I / 128) * 16));
    S.tok2 = reinterpret_cast<int *>(take(4 * 16));
    S.slot = reinterpret_cast<volatile int *>(take(4 * 2));
    S.staged = reinterpret_cast<uint64_t *>(take(8 * 4));
    S.consumed = S.staged + 2;
  } else {
    S.sc2 = S.cs2 = nullptr;
    S.tok2 = nullptr;
    S.slot = nullptr;
    S.staged = S.consumed = nullptr;
  }
  return S;
}

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void fail(const Smem &S, const TcArgs &a) {
  if (!S.misc[0]) {
    S.misc[0] = 1;
    if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
  }
}

// Bounded waits that also give up once another role of the CTA failed.
__device__ __forceinline__ bool wait_bar(const Smem &S, uint64_t *bar, uint32_t parity) {
  return wait_phase(S.misc, bar, parity);
}
__device__ __forceinline__ bool wait_count(const Smem &S, const int *p, int target) {
  return wait_at_least(S.misc, p, target);
}

__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory");
}

// ---------------------------------------------------------------------------
// work items
// ---------------------------------------------------------------------------

struct Item {
  bool gu;       // gate+up (else down)
  int a, e;      // active-list index, expert
  int pos0;      // first sorted position of the row tile
  int rows;      // real rows in the tile (1..64)
  int n16;       // MMA N: rows rounded up to 16
  int box;       // term box: 16 << box rows
  int kps;       // k blocks per stage: 2 for up to 32 rows, else 1
  int tile;      // gate+up: 128-row tile of I; down: pair of 128-row tiles of H
};

__device__ __forceinline__ Item decode(const Smem &S, int A, int i, int TR, int FT, int FD,
                                       int RT) {
  Item it;
  int rtg;
  if (i < TR * FT) {
    it.gu = true;
    rtg = i / FT;
    it.tile = i - rtg * FT;
  } else {
    it.gu = false;
    const int j = i - TR * FT;
    rtg = j / FD;
    it.tile = j - rtg * FD;
  }
  int lo = 0, hi = A - 1;   // the last a with rtp[a] <= rtg
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.rtp[mid] <= rtg)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int2 inf = S.info[lo];
  const int rt = rtg - S.rtp[lo];
  const int rows_e = inf.y >> 16;
  it.a = lo;
  it.e = inf.y & 0xFFFF;
  it.pos0 = inf.x + rt * RT;
  it.rows = min(RT, rows_e - rt * RT);
  it.n16 = (it.rows + 15) & ~15;
  it.box = it.n16 <= 16 ? 0 : (it.n16 <= 32 ? 1 : 2);
  it.kps = it.n16 <= 32 ? 2 : 1;
  return it;
}

// TMEM columns of one k block's accumulators: the two weight tiles, each
// against the item's terms stacked along N (term t of row j in column
// t * nt + j), so one MMA per tile and 32-wide k step reads the weights once.
__device__ __forceinline__ uint32_t acc_cols(const Item &it) {
  return 2u * (uint32_t)(it.gu ? kXTerms : kHTerms) * (16u << it.box);
}

// Bytes of one stage of an item: kps k blocks of the two weight tiles and of
// the item's activation terms.
__device__ __forceinline__ uint32_t stage_bytes(const Item &it) {
  return 2u * (uint32_t)it.kps * kTileBytes +
         (uint32_t)it.kps * (uint32_t)(it.gu ? kXTerms : kHTerms) * (16u << it.box) * 128u;
}

// ---------------------------------------------------------------------------
// phase 0: x terms of every routed slot
// ---------------------------------------------------------------------------
//
// Slot i (token t = i / k) at sorted position p = token_to_perm[i]: s = shift
// putting max|x[t]| in [128, 256); xs[p] = 2^-s; t0 = e4m3(x * 2^s),
// t1 = e4m3(x * 2^s - t0).  A bf16 value has 8 significant bits and each E4M3
// term 4, so t0 + t1 equals x * 2^s exactly wherever the residual is not
// below E4M3's subnormal step (elements smaller than 2^-10 of the row maximum
// lose bits of at most 2^-18 of that maximum).  One warp per slot, its
// row's loads in flight together (16 per lane for H = 4096).
__device__ void prep_x(const TcArgs &a) {
  const int ew = (threadIdx.x >> 5) - 2, lane = threadIdx.x & 31;
  const int nw = gridDim.x * kEpiWarps;
  const size_t plane = (size_t)a.max_total * a.H;
  for (int i = blockIdx.x * kEpiWarps + ew; i < a.n; i += nw) {
    const int p = __ldcg(a.ttp + i);
    if (p < 0 || p >= a.max_total) continue;
    const uint16_t *xr = a.x + (size_t)(i / a.k) * a.H;
    uint32_t mx = 0;
    for (int c0 = 0; c0 < a.H; c0 += 16 * 256) {
      uint4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j * 256 + lane * 8;
        v[j] = c < a.H ? __ldg(reinterpret_cast<const uint4 *>(xr + c)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          mx = max(mx, (w[h] & 0x7FFFu) << 16);
          mx = max(mx, (w[h] >> 16 & 0x7FFFu) << 16);
        }
      }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    const int s = term_shift(mx);
    const float scl = pow2f(s);
    if (lane == 0) a.xs[p] = pow2f(-s);
    uint8_t *q0 = a.xq + (size_t)p * a.H;
    uint8_t *q1 = q0 + plane;
#pragma unroll 4
    for (int c = lane * 8; c < a.H; c += 256) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + c));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t t0[2] = {0, 0}, t1[2] = {0, 0};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float f0 = bf16_to_float((uint16_t)(w[h] & 0xFFFFu)) * scl;
        const float f1 = bf16_to_float((uint16_t)(w[h] >> 16)) * scl;
        const uint32_t b0 = e4m3x2(f0, f1);
        const float2 back = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)b0));
        const uint32_t b1 = e4m3x2(f0 - back.x, f1 - back.y);
        t0[h >> 1] |= b0 << (16 * (h & 1));
        t1[h >> 1] |= b1 << (16 * (h & 1));
      }
      *reinterpret_cast<uint2 *>(q0 + c) = make_uint2(t0[0], t0[1]);
      *reinterpret_cast<uint2 *>(q1 + c) = make_uint2(t1[0], t1[1]);
    }
  }
}

// Grid barrier among the promotion warps of every CTA (named barrier 1 in the
// CTA, then one thread's arrival on the monotonic count); true when all CTAs
// arrived within the wait limit.
__device__ bool epi_grid_barrier(const Smem &S, unsigned long long *ctr) {
  __threadfence();
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
  if (threadIdx.x == 64) {
    const unsigned long long G = gridDim.x;
    const unsigned long long v = atomicAdd(ctr, 1ull);
    const unsigned long long target = (v / G + 1) * G;
    bool ok = false;
    const uint64_t t0 = gtime();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
      unsigned long long c;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(c) : "l"(ctr) : "memory");
      if (c >= target) {
        ok = true;
        break;
      }
      if (gtime() - t0 > kWaitNs) break;
      __nanosleep(64);
    }
    __threadfence();
    S.misc[5] = ok;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
  return S.misc[5] != 0;
}

// Grid barrier of all threads: one thread's arrival with release semantics
// (covering every write of the CTA before the CTA barrier), its acquire of
// the full count, then the CTA barrier again.
__device__ bool grid_barrier(const Smem &S, unsigned long long *ctr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long G = gridDim.x;
    unsigned long long v;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(ctr) : "memory");
    const unsigned long long target = (v / G + 1) * G;
    bool ok = false;
    const uint64_t t0 = gtime();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
      unsigned long long c;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(c) : "l"(ctr) : "memory");
      if (c >= target) {
        ok = true;
        break;
      }
      if (gtime() - t0 > kWaitNs) break;
      __nanosleep(64);
    }
    S.misc[4] = ok;
  }
  __syncthreads();
  return S.misc[4] != 0;
}

// The active list as row tiles: info[a] = {run offset, expert | rows << 16},
// rtp = exclusive prefix of ceil(rows / 64).  The alignment launch wrote the
// active table (offset, expert and slot count of each active expert), so
// this is one coalesced load and a scan.  Returns the active count.
__device__ int build_table(const TcArgs &a, const Smem &S) {
  // the first kThreads entries are loaded together with the count (entries
  // past the count are read but not used): one round trip
  const int i0 = threadIdx.x;
  const int4 pre = i0 < a.cap ? __ldcg(a.items + i0) : make_int4(0, 0, 0, 0);
  const int A = min(max(__ldcg(a.act_count), 0), a.cap);
  for (int i = i0; i < A; i += kThreads) {
    const int4 inf = i == i0 ? pre : __ldcg(a.items + i);
    const int rows = min(inf.z, 0x7FFF);
    S.info[i] = make_int2(inf.x, (inf.y & 0xFFFF) | (rows << 16));
    S.rtp[i] = (rows + a.row_tile - 1) / a.row_tile;   // counts; scanned below
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int run = 0;
    for (int b = 0; b < A; b += 32) {
      const int v = b + lane < A ? S.rtp[b + lane] : 0;
      int inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += t;
      }
      if (b + lane < A) S.rtp[b + lane] = run + inc - v;
      run += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
    if (lane == 0) {
      S.rtp[A] = run;
      S.misc[2] = A;
      S.misc[3] = run;
    }
  }
  __syncthreads();
  return A;
}

// ---------------------------------------------------------------------------
// roles
// ---------------------------------------------------------------------------
//
// Items are taken dynamically: CTA b starts with item b; after issuing an
// item's copies its copy thread takes the next index of the grid-wide order
// (gate+up items, then down items) from a counter, and passes each index to
// the MMA thread and the promotion warps through a small queue.  Indices are taken in increasing order, so a down
// item's gate+up items have all been taken by running CTAs before it is.

// The j-th item of this CTA (total: no more items), or -1 when the wait gave up.
__device__ __forceinline__ int next_item(const Smem &S, int j) {
  if (!wait_bar(S, &S.iqbar[j % kIQ], (uint32_t)(j / kIQ) & 1)) return -1;
  return S.iq[j % kIQ];
}

__device__ void producer(const TcArgs &a, const TcMaps &m, const Smem &S, int A, int TR,
                         int total) {
  const uint64_t pol = policy_evict_first();
  const int FT = a.I / 128, FD = a.H / 256;
  uint32_t head = 0, thead = 0;   // shared-memory and TMEM ring heads
  bool x_ready = a.tok != 0;       // the grid's x terms are visible (token form: at launch)
  int s = 0, tail = 0, kq = -1;
  int ttail = 0;                   // oldest stage that may still hold TMEM
  bool ok = true;
  int jq = 0;                      // items passed to the queue
  int i = blockIdx.x;              // the first item is the CTA's own
  if (i >= total) i = total;
  while (i < total && ok) {
    S.iq[jq % kIQ] = i;
    mbar_arrive(&S.iqbar[jq % kIQ]);
    ++jq;
    const Item it = decode(S, A, i, TR, FT, FD, a.row_tile);
    if (!it.gu) {
      const int need = (S.rtp[it.a + 1] - S.rtp[it.a]) * FT;
      if (!wait_count(S, a.done + it.a, need)) {
        ok = false;
        break;
      }
      fence_proxy_async_global();
    }
    const int KB = it.gu ? a.H / 128 : a.I / 128;
    const int wrow0 = it.gu ? it.e * a.I + it.tile * 128 : it.e * a.H + it.tile * 256;
    const CUtensorMap *w0 = it.gu ? &m.w[0][it.kps - 1] : &m.w[2][it.kps - 1];
    const CUtensorMap *w1 = it.gu ? &m.w[1][it.kps - 1] : w0;
    const int wrow1 = it.gu ? wrow0 : wrow0 + 128;
    const uint32_t bterm = (uint32_t)(it.gu ? kXTerms : kHTerms) * (16u << it.box) * 128u;
    const uint32_t abytes = (uint32_t)it.kps * kTileBytes;
    const uint32_t size = stage_bytes(it);
    const uint32_t tcols = (uint32_t)it.kps * acc_cols(it);
    const CUtensorMap *bmap = it.gu ? &m.xq[it.box] : &m.hq[it.box];
    for (int kb = 0; kb < KB; kb += it.kps) {
      // Ring placement.  A stage holds a range of the shared-memory ring (its
      // copies, freed when its MMAs complete) and a range of the TMEM ring
      // (its accumulators, freed when the promotion warps have read them).
      // Ranges are placed in order and freed oldest first.  When a range does
      // not fit before the end, its ring wraps: the stages still lying in the
      // skipped end [head, end) are the oldest and go first.  Then only the
      // oldest stage can overlap the new range, so stages are retired oldest
      // first until it does not.  The copies wait here for shared memory; the
      // TMEM retirement is only computed here and waited for by the MMA
      // thread, which needs the columns (twait: the newest stage to retire).
      int need_t = -1;
      {
        const bool twrap = thead + tcols > kTmemCols;
        const uint32_t ct = twrap ? 0u : thead;
        while (ttail < s) {
          const uint32_t tr = S.trec[ttail % kRecs], cp = tr & 0xFFFFu, cl = tr >> 16;
          const bool busy = s - ttail >= kTfree / 2 || (twrap && cp >= thead) ||
                            (ct < cp + cl && cp < ct + tcols);
          if (!busy) break;
          need_t = ttail++;
        }
      }
      const bool wrap = head + size > a.ring_bytes;
      while (tail < s) {
        const int dt = tail % kRecs;
        const uint32_t tp = S.rec[dt], tl = S.rlen[dt];
        const uint32_t at = wrap ? 0u : head;
        const bool busy =
            s - tail >= kRecs || (wrap && tp >= head) || (at < tp + tl && tp < at + size);
        if (!busy) break;
        // the stage's last k block is done: so are all its MMAs
        const int ke = S.kend[dt];
        if (!wait_bar(S, &S.accf[ke % kAccs], (uint32_t)(ke / kAccs) & 1)) {
          ok = false;
          break;
        }
        ++tail;
      }
      if (!ok) break;
      const uint32_t pos = ring_place(head, size, a.ring_bytes);
      const uint32_t tpos = ring_place(thead, tcols, kTmemCols);
      const int d = s % kRecs;
      kq += it.kps;
      S.kend[d] = kq;
      S.rec[d] = pos;
      S.rlen[d] = size;
      S.trec[d] = tpos | (tcols << 16);
      S.twait[d] = need_t;
      uint64_t *fb = &S.full[d];
      mbar_expect_tx(fb, size);
      uint8_t *dst = S.ring + pos;
      tma_3d_hint(dst, w0, 0, wrow0, kb, fb, pol);
      tma_3d_hint(dst + abytes, w1, 0, wrow1, kb, fb, pol);
      if (!x_ready) {   // the weights above do not wait for the x terms
        const uint64_t t0 = gtime();
        while (!S.misc[6]) {
          if (S.misc[0] || gtime() - t0 > kWaitNs) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
        __threadfence();
        fence_proxy_async_global();
        x_ready = true;
      }
      for (int j = 0; j < it.kps; ++j) {
        if (a.tok && it.gu)   // all 16 token columns of k block kb + j
          tma_3d(dst + 2 * abytes + j * bterm, &m.xt, 0, 0, 2 * (kb + j), fb);
        else
          tma_3d(dst + 2 * abytes + j * bterm, bmap, (kb + j) * 128, it.pos0, 0, fb);
      }
      ++s;
    }
    // the next item, taken once this one's copies are all issued (taken any
    // earlier, a CTA would hold two items while another has none)
    i = (int)gridDim.x + atomicAdd(a.work, 1);
  }
  S.iq[jq % kIQ] = total;   // no more items
  mbar_arrive(&S.iqbar[jq % kIQ]);
  if (!ok) fail(S, a);
  // every copy this CTA issued has landed before it moves on
  for (int j = max(tail, s - kRecs); j < s; ++j) {
    const uint64_t t0 = gtime();
    while (!mbar_poll(&S.full[j % kRecs], (uint32_t)(j / kRecs) & 1))
      if (gtime() - t0 > kWaitNs) break;
  }
}

__device__ void mma_issuer(const TcArgs &a, const Smem &S, int A, int TR, int total,
                           uint32_t tmem) {
  const int FT = a.I / 128, FD = a.H / 256;
  const uint32_t ring = smem_addr(S.ring);
  uint32_t head = 0, thead = 0;   // the copy thread's placement, recomputed
  int s = 0;                      // stages
  int q = 0;                      // k blocks
  int tdone = -1;                 // newest stage whose TMEM release was seen
  bool ok = true;
  for (int jq = 0; ok; ++jq) {
    const int i = next_item(S, jq);
    if (i < 0) ok = false;
    if (i < 0 || i >= total) break;
    const Item it = decode(S, A, i, TR, FT, FD, a.row_tile);
    const int KB = it.gu ? a.H / 128 : a.I / 128;
    const int T = it.gu ? kXTerms : kHTerms;
    const uint32_t nt = 16u << it.box;
    const uint32_t id = idesc_e4m3(T * (int)nt);
    const uint32_t cols = acc_cols(it);
    const uint32_t abytes = (uint32_t)it.kps * kTileBytes;
    const uint32_t size = stage_bytes(it), tcols = (uint32_t)it.kps * cols;
    for (int kb = 0; kb < KB; kb += it.kps) {
      const uint32_t base = ring + ring_place(head, size, a.ring_bytes);
      const uint32_t tbase = tmem + ring_place(thead, tcols, kTmemCols);
      const int d = s % kRecs;
      if (!wait_bar(S, &S.full[d], (uint32_t)(s / kRecs) & 1)) {
        ok = false;
        break;
      }
      const int tw = S.twait[d];
      if (tw > tdone) {   // the columns are free once that stage is released
        if (!wait_bar(S, &S.tfree[tw % kTfree], (uint32_t)(tw / kTfree) & 1)) {
          ok = false;
          break;
        }
        tdone = tw;
      }
      tc_fence_after();
      for (int j = 0; j < it.kps; ++j) {
        const uint32_t a0 = base + j * kTileBytes, a1 = a0 + abytes;
        const uint32_t b0 = base + 2 * abytes + j * (uint32_t)T * nt * 128u;
        const uint32_t d0 = tbase + (uint32_t)j * cols, d1 = d0 + (uint32_t)T * nt;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = sdesc(b0 + ks * 32);
          mma_e4m3(d0, sdesc(a0 + ks * 32), bd, id, ks != 0);
          mma_e4m3(d1, sdesc(a1 + ks * 32), bd, id, ks != 0);
        }
        mma_commit(&S.accf[q % kAccs]);
        ++q;
      }
      ++s;
    }
  }
  if (!ok) fail(S, a);
  // every MMA this thread issued has completed before TMEM is freed
  mma_commit(S.drain);
  const uint64_t t0 = gtime();
  while (!mbar_poll(S.drain, 0))
    if (gtime() - t0 > kWaitNs) break;
}

// Gate+up finish of one item: h = silu(g) * u per (row, feature), written as
// three E4M3 terms with a power-of-two scale per (row, this 128-feature
// block) and returned in hv as fp32 (stored by store_h once the item is
// published).
__device__ void finish_gate_up(const TcArgs &a, const Smem &S, const Item &it, int grp, int q,
                               int lane, const float (&acc0)[16], const float (&acc1)[16],
                               const float *csb, const int *tokb, float (&hv)[16]) {
  const int c0 = grp * 16, f = q * 32 + lane, o = it.tile * 128 + f;
  const int KBd = a.I / 128;
  // only the item's real rows are finished (the condition is the same for the
  // whole warp; at decode sizes most of a warp's 16 columns are padding)
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) {
    hv[jj] = 0.f;
    if (c0 + jj < it.rows) {
      const float xi = csb[c0 + jj];
      float g = acc0[jj], u = acc1[jj];
      if (a.tok) {   // the MMA columns are tokens: take the row's own
        const int t = tokb[c0 + jj];
        g = u = 0.f;
#pragma unroll
        for (int tt = 0; tt < kTokMax; ++tt) {
          g = tt == t ? acc0[tt] : g;
          u = tt == t ? acc1[tt] : u;
        }
      }
      hv[jj] = silu_f32(g * xi) * (u * xi);
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(hv[jj])));
      if (lane == 0) S.red[(grp * 4 + q) * 16 + jj] = m;
    }
  }
  group_sync(grp);
  float scl = 1.f;
  if (lane < 16) {
    uint32_t m = 0;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) m = max(m, S.red[(grp * 4 + qq) * 16 + lane]);
    const int s = term_shift(m);
    scl = pow2f(s);
    if (q == 0 && c0 + lane < it.rows)
      a.hs[(size_t)(it.pos0 + c0 + lane) * KBd + it.tile] = pow2f(-s);
  }
  const size_t plane = (size_t)a.max_total * a.I;
#pragma unroll
  for (int jj = 0; jj < 16; jj += 2) {
    if (c0 + jj >= it.rows) break;
    const float v0 = hv[jj] * __shfl_sync(0xFFFFFFFFu, scl, jj);
    const float v1 = hv[jj + 1] * __shfl_sync(0xFFFFFFFFu, scl, jj + 1);
    const uint32_t b0 = e4m3x2(v0, v1);
    const float2 r0 = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)b0));
    const float u0 = v0 - r0.x, u1 = v1 - r0.y;
    const uint32_t b1 = e4m3x2(u0, u1);
    const float2 r1 = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)b1));
    const uint32_t b2 = e4m3x2(u0 - r1.x, u1 - r1.y);
    const uint32_t bb[3] = {b0, b1, b2};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      if (c0 + jj + h2 < it.rows) {
        uint8_t *dst = a.hq + (size_t)(it.pos0 + c0 + jj + h2) * a.I + o;
#pragma unroll
        for (int t = 0; t < kHTerms; ++t) dst[t * plane] = (uint8_t)(bb[t] >> (8 * h2));
      }
    }
  }
}

// The fp32 h of a finished gate+up tile (read by no item of the kernel, so
// written after the tile is published).
__device__ __forceinline__ void store_h(const TcArgs &a, const Item &it, int grp, int q, int lane,
                                        const float (&hv)[16]) {
  const int c0 = grp * 16, o = it.tile * 128 + q * 32 + lane;
#pragma unroll
  for (int jj = 0; jj < 16; ++jj)
    if (c0 + jj < it.rows) a.h[(size_t)(it.pos0 + c0 + jj) * a.I + o] = hv[jj];
}

// acc += scale * (sum of the T term partials of this warp's 16 columns),
// times the per-row factor hf[j] of the down projection when hf is given.
__device__ __forceinline__ void promote(uint32_t col, uint32_t nt, int T, float scale,
                                        const float *hf, float (&acc)[16]) {
  uint32_t r[16], r2[16];
  tmem_ld16(col, r);
  tmem_ld16(col + nt, r2);
  tmem_wait_ld();
  float part[16];
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) part[jj] = __uint_as_float(r[jj]) + __uint_as_float(r2[jj]);
  if (T == 3) {
    tmem_ld16(col + 2 * nt, r);
    tmem_wait_ld();
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) part[jj] += __uint_as_float(r[jj]);
  }
  if (hf == nullptr) {
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) acc[jj] = fmaf(scale, part[jj], acc[jj]);
  } else {
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) acc[jj] = fmaf(scale * hf[jj], part[jj], acc[jj]);
  }
}

// Barrier over the 16 epilogue warps that also ORs a flag across them, so
// that every warp takes the same branch after it.
__device__ __forceinline__ bool epi_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(kEpiThreads)
      : "memory");
  return r != 0;
}

// Barrier over one group of four promotion warps (named barrier 2 + g) that
// also ORs a flag across them.
__device__ __forceinline__ bool group_sync_or(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(2 + g)
      : "memory");
  return r != 0;
}

// Token form (M <= 16): every item has one 16-column block, held by group 0
// (warps 2-5).  Group 1 (warps 6-9) stages the next item into the other of
// two buffers -- its block scales, its rows' tokens and x scales, or (after
// the wait for its expert's gate+up items) a down item's h scales -- while
// group 0 promotes and finishes the current one, so no item waits for its
// own loads.  Groups 2 and 3 hold no columns and have no part here.
__device__ void epilogue_token(const TcArgs &a, const Smem &S, int A, int TR, int total,
                               uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - 2, q = warp & 3, grp = ew >> 2;
  const int lt = (threadIdx.x - 64) & 127;   // index within the group
  const int FT = a.I / 128, FD = a.H / 256, KBd = a.I / 128;
  bool bad = false;
  if (grp == 1) {
    for (int jq = 0;; ++jq) {
      const int b = jq & 1;
      int i = lane == 0 ? next_item(S, jq) : 0;
      i = __shfl_sync(0xFFFFFFFFu, i, 0);
      bool ok = i >= 0;
      // the buffer is free once group 0 is done with item jq - 2
      if (ok && jq >= 2)
        ok = __all_sync(0xFFFFFFFFu,
                        wait_bar(S, &S.consumed[b], (uint32_t)((jq - 2) >> 1) & 1));
      if (group_sync_or(1, !ok)) {
        bad = true;
        break;
      }
      if (i >= total) {   // no more items: hand over the end
        if (lt == 0) {
          S.slot[b] = total;
          mbar_arrive(&S.staged[b]);
        }
        break;
      }
      const Item it = decode(S, A, i, TR, FT, FD, a.row_tile);
      const int KB = it.gu ? a.H / 128 : KBd;
      float *sc = b ? S.sc2 : S.sc;
      float *cs = b ? S.cs2 : S.cs;
      int *tk = b ? S.tok2 : S.tokrow;
      bool dep = true;
      if (it.gu) {
        const size_t sb = ((size_t)it.e * FT + it.tile) * KB;
        for (int j = lt; j < KB; j += 128) {
          sc[j] = __ldg(a.sg + sb + j);
          sc[kMaxKB + j] = __ldg(a.su + sb + j);
        }
        if (lt < 16) {   // each row's token and that token's x scale
          const int t = lt < it.rows ? __ldcg(a.sti + it.pos0 + lt) / a.k : 0;
          tk[lt] = t;
          cs[lt] = lt < it.rows ? S.xtok[t] : 0.f;
        }
      } else {
        const size_t sb = ((size_t)it.e * (a.H / 128) + 2 * it.tile) * KB;
        for (int j = lt; j < KB; j += 128) {
          sc[j] = __ldg(a.sd + sb + j);
          sc[kMaxKB + j] = __ldg(a.sd + sb + KB + j);
        }
        if (lt == 0) dep = wait_count(S, a.done + it.a, (S.rtp[it.a + 1] - S.rtp[it.a]) * FT);
      }
      // a down item's h scales are read only after the dependency wait
      if (group_sync_or(1, !dep || S.misc[0])) {
        bad = true;
        break;
      }
      if (!it.gu) {
        for (int idx = lt; idx < KB * 16; idx += 128) {
          const int kb = idx >> 4, j = idx & 15;
          cs[idx] = j < it.rows ? __ldcg(a.hs + (size_t)(it.pos0 + j) * KBd + kb) : 0.f;
        }
        group_sync(1);
      }
      if (lt == 0) {
        S.slot[b] = i;
        mbar_arrive(&S.staged[b]);   // release: the group's stores above are visible
      }
    }
  } else if (grp == 0) {
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t arrivals = ew == 0 ? (uint32_t)(kEpiWarps - 4 + 1) : 1u;
    int s = 0, st = 0;
    uint32_t thead = 0;
    for (int jq = 0;; ++jq) {
      const int b = jq & 1;
      const bool ok = __all_sync(0xFFFFFFFFu, wait_bar(S, &S.staged[b], (uint32_t)(jq >> 1) & 1));
      if (group_sync_or(0, !ok)) {
        bad = true;
        break;
      }
      const int i = S.slot[b];
      if (i >= total) break;
      const Item it = decode(S, A, i, TR, FT, FD, a.row_tile);
      const int KB = it.gu ? a.H / 128 : KBd;
      const float *sc = b ? S.sc2 : S.sc;
      const float *cs = b ? S.cs2 : S.cs;
      const int *tk = b ? S.tok2 : S.tokrow;
      float acc0[16], acc1[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) acc0[jj] = acc1[jj] = 0.f;
      const int T = it.gu ? kXTerms : kHTerms;
      const uint32_t nt = 16u << it.box, cols = acc_cols(it), tcols = (uint32_t)it.kps * cols;
      uint32_t tbase = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int j = kb % it.kps;
        if (j == 0) tbase = ring_place(thead, tcols, kTmemCols);
        const uint32_t pos = tbase + (uint32_t)j * cols;
        const int slot = s % kAccs;
        if (!__all_sync(0xFFFFFFFFu, wait_bar(S, &S.accf[slot], (uint32_t)(s / kAccs) & 1))) {
          bad = true;
          break;
        }
        tc_fence_after();
        const uint32_t col = lane_base + pos;
        const float *hf = it.gu ? nullptr : cs + kb * 16;
        promote(col, nt, T, sc[kb], hf, acc0);
        promote(col + (uint32_t)T * nt, nt, T, sc[kMaxKB + kb], hf, acc1);
        ++s;
        if (j == it.kps - 1) {   // the stage's accumulators are free
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_n(&S.tfree[st % kTfree], arrivals);
          ++st;
        }
      }
      if (group_sync_or(0, bad)) {
        bad = true;
        break;
      }
      if (it.gu) {
        float hv[16];
        finish_gate_up(a, S, it, 0, q, lane, acc0, acc1, cs, tk, hv);
        // every h term of the tile is visible to every CTA and its tensor
        // copies before the tile is counted
        fence_proxy_async_global();
        group_sync(0);
        if (lt == 0) red_release_add(a.done + it.a, 1);
        store_h(a, it, 0, q, lane, hv);
      } else {
        const int o0 = it.tile * 256 + q * 32 + lane;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          if (jj >= it.rows) break;
          float *yr = a.y + (size_t)(it.pos0 + jj) * a.H + o0;
          yr[0] = acc0[jj];
          yr[128] = acc1[jj];
        }
        group_sync(0);
      }
      if (lt == 0) mbar_arrive(&S.consumed[b]);   // the buffer may be staged again
    }
  }
  if (bad) fail(S, a);
}

// The 16 promotion warps.  Warp w (2..17) reads TMEM lanes 32*(w%4)..+31
// (its quadrant q of the 128 weight rows) and columns 16*g..16*g+15 (its
// group g = (w-2)/4 of the item's token rows).  Every decision to leave the
// item loop is taken after a vote over all 16 warps.
__device__ void epilogue(const TcArgs &a, const Smem &S, int A, int TR, int total,
                         uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - 2, q = warp & 3, grp = ew >> 2;
  const int et = threadIdx.x - 64;
  const int FT = a.I / 128, FD = a.H / 256, KBd = a.I / 128;
  const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
  const int c0 = grp * 16;
  int s = 0;            // k blocks
  int st = 0;           // stages
  uint32_t thead = 0;   // the copy thread's TMEM placement, recomputed
  int pending = -1;   // active index of a finished gate+up item not yet published
  bool bad = false;
  if (a.tok) {
    // token form: the alignment launch wrote the x-term table and the token
    // scales; they are complete at launch
    if (et < a.M) S.xtok[et] = __ldcg(a.xs + et);
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
    epilogue_token(a, S, A, TR, total, tmem);
    return;
  } else {
    // the x terms of this CTA's share of the slots, then the grid barrier
    // that makes all of them (and the zeroed counters) visible to the copies
    prep_x(a);
    fence_proxy_async_global();
    if (!epi_grid_barrier(S, a.grid_ctr)) {
      bad = true;
      fail(S, a);
    }
  }
  if (et == 0 && !a.tok) {
    fence_proxy_async_global();
    __threadfence();
    S.misc[6] = 1;
  }
  for (int jq = 0;; ++jq) {
    // every lane of every promotion warp takes the same item
    int i = next_item(S, jq);
    i = __shfl_sync(0xFFFFFFFFu, i, 0);
    if (epi_sync_or(i < 0)) {
      bad = true;
      break;
    }
    if (i >= total) break;
    const Item it = decode(S, A, i, TR, FT, FD, a.row_tile);
    const int KB = it.gu ? a.H / 128 : KBd;
    fence_proxy_async_global();   // this thread's h terms before the publish
    if (epi_sync_or(bad || S.misc[0])) {
      bad = true;
      break;
    }
    if (et == 0) {
      if (pending >= 0) red_release_add(a.done + pending, 1);
      if (!it.gu) {
        const int need = (S.rtp[it.a + 1] - S.rtp[it.a]) * FT;
        if (!wait_count(S, a.done + it.a, need)) fail(S, a);
      }
    }
    pending = -1;
    // the item's weight block scales and per-row factors
    if (it.gu) {
      const size_t sb = ((size_t)it.e * FT + it.tile) * KB;
      for (int j = et; j < KB; j += kEpiThreads) {
        S.sc[j] = __ldg(a.sg + sb + j);
        S.sc[kMaxKB + j] = __ldg(a.su + sb + j);
      }
      if (a.tok) {   // each row's token and that token's x scale
        for (int j = et; j < a.row_tile; j += kEpiThreads) {
          const int t = j < it.rows ? __ldcg(a.sti + it.pos0 + j) / a.k : 0;
          S.tokrow[j] = t;
          S.cs[j] = j < it.rows ? S.xtok[t] : 0.f;
        }
      } else {
        for (int j = et; j < a.row_tile; j += kEpiThreads)
          S.cs[j] = j < it.rows ? __ldcg(a.xs + it.pos0 + j) : 0.f;
      }
    } else {
      const size_t sb = ((size_t)it.e * (a.H / 128) + 2 * it.tile) * KB;
      for (int j = et; j < KB; j += kEpiThreads) {
        S.sc[j] = __ldg(a.sd + sb + j);
        S.sc[kMaxKB + j] = __ldg(a.sd + sb + KB + j);
      }
    }
    // the dependency wait is over (or failed) before any h scale is read
    if (epi_sync_or(S.misc[0])) {
      bad = true;
      break;
    }
    if (!it.gu) {
      for (int idx = et; idx < KB * a.row_tile; idx += kEpiThreads) {
        const int kb = idx / a.row_tile, j = idx - kb * a.row_tile;
        S.cs[idx] = j < it.rows ? __ldcg(a.hs + (size_t)(it.pos0 + j) * KBd + kb) : 0.f;
      }
      epi_sync_or(false);
    }

    float acc0[16], acc1[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) acc0[jj] = acc1[jj] = 0.f;
    // Only the warps whose columns hold rows of the item read TMEM; the first
    // of them also arrives for the others, and the rest skip the k blocks.
    const bool mine = c0 < it.n16;
    const uint32_t arrivals = ew == 0 ? (uint32_t)(kEpiWarps - (it.n16 / 16) * 4 + 1) : 1u;
    const int T = it.gu ? kXTerms : kHTerms;
    const uint32_t nt = 16u << it.box, cols = acc_cols(it), tcols = (uint32_t)it.kps * cols;
    if (!mine) {
      for (int kb = 0; kb < KB; kb += it.kps) ring_place(thead, tcols, kTmemCols);
      s += KB;
      st += KB / it.kps;
    }
    uint32_t tbase = 0;
    for (int kb = 0; kb < KB && mine; ++kb) {
      const int j = kb % it.kps;
      if (j == 0) tbase = ring_place(thead, tcols, kTmemCols);
      const uint32_t pos = tbase + (uint32_t)j * cols;
      const int slot = s % kAccs;
      // every lane of the warp takes the same branch into the aligned TMEM loads
      if (!__all_sync(0xFFFFFFFFu, wait_bar(S, &S.accf[slot], (uint32_t)(s / kAccs) & 1))) {
        bad = true;
        break;
      }
      tc_fence_after();
      const uint32_t col = lane_base + pos + (uint32_t)c0;
      const float *hf = it.gu ? nullptr : S.cs + kb * a.row_tile + c0;
      promote(col, nt, T, S.sc[kb], hf, acc0);
      promote(col + (uint32_t)T * nt, nt, T, S.sc[kMaxKB + kb], hf, acc1);
      ++s;
      if (j == it.kps - 1) {   // the stage's accumulators are free
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_n(&S.tfree[st % kTfree], arrivals);
        ++st;
      }
    }
    // every warp finished the item's k blocks before any finishes the item
    if (epi_sync_or(bad)) {
      bad = true;
      break;
    }
    if (it.gu) {
      if (mine) {
        float hv[16];
        finish_gate_up(a, S, it, grp, q, lane, acc0, acc1, S.cs, S.tokrow, hv);
        store_h(a, it, grp, q, lane, hv);
      }
      pending = it.a;
    } else if (mine) {
      const int f = q * 32 + lane;
      const int o0 = it.tile * 256 + f;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        if (c0 + jj < it.rows) {
          float *yr = a.y + (size_t)(it.pos0 + c0 + jj) * a.H + o0;
          yr[0] = acc0[jj];
          yr[128] = acc1[jj];
        }
    }
  }
  if (bad) fail(S, a);
  // publish the last gate+up item
  fence_proxy_async_global();
  epi_sync_or(false);
  if (et == 0 && pending >= 0 && !bad) red_release_add(a.done + pending, 1);
}

__global__ void __launch_bounds__(kThreads, 1)
    verify_ffn_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ TcMaps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem S = carve(smem, a);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int j = 0; j < kRecs; ++j) mbar_init(&S.full[j], 1);
    for (int j = 0; j < kAccs; ++j) mbar_init(&S.accf[j], 1);
    for (int j = 0; j < kTfree; ++j) mbar_init(&S.tfree[j], kEpiWarps);
    for (int j = 0; j < kIQ; ++j) mbar_init(&S.iqbar[j], 1);
    if (a.tok)
      for (int j = 0; j < 4; ++j) mbar_init(&S.staged[j], 1);   // staged[2], consumed[2]
    mbar_init(S.drain, 1);
    for (int j = 0; j < 16; ++j) S.misc[j] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr((const void *)(S.misc + 1))),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)S.misc[1];
  // the swizzled operand tiles assume a 1024-byte aligned ring
  if ((smem_addr(S.ring) & 1023u) != 0) fail(S, a);

  if (threadIdx.x == 0) {   // the copy thread's descriptors, ahead of the first copies
    for (int j = 0; j < 3; ++j) prefetch_tensormap(&maps.w[j][a.tok ? 1 : 0]);
    prefetch_tensormap(a.tok ? &maps.xt : &maps.xq[0]);
  }
  pdl_wait();   // the tables of the alignment (and the token form's x terms) are final
  // The item table first (it needs only the alignment's tables); in the row
  // form the x terms are written by the promotion warps while the copy warp
  // already streams weight tiles, which do not depend on them (misc[6]: x
  // terms ready).
  const int A = build_table(a, S);
  const int TR = S.misc[3];
  const int total = S.misc[0] ? 0 : TR * (a.I / 128 + a.H / 256);

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) producer(a, maps, S, A, TR, total);
    __syncwarp();
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) mma_issuer(a, S, A, TR, total, tmem);
    __syncwarp();
  } else {
    epilogue(a, S, A, TR, total, tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }

  // ---- blend: every y row is written before any CTA blends its share ------
  //   out[t][c] = bf16_rn(sum_j w[t][j] * y[token_to_perm[t*k+j]][c]), fp32,
  //   j ascending ("fp8_moe_grouped.rs", moe_weighted_sum_blend_fp8_grouped)
  if (!grid_barrier(S, a.grid_ctr) || S.misc[0]) {
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
    return;
  }
  // every item of every CTA is done: the counters start the next call at zero
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < a.cap; i += kThreads) a.done[i] = 0;
    if (threadIdx.x == 0) {
      *a.work = 0;
    }
  }
  const long long T4 = (long long)a.M * a.H / 4;
  const long long o1 = T4 * (blockIdx.x + 1) / gridDim.x;
  for (long long o = T4 * blockIdx.x / gridDim.x + threadIdx.x; o < o1; o += kThreads) {
    const int t = (int)(o * 4 / a.H), c = (int)(o * 4 % a.H);
    const float4 acc = blend_slots(a.y, a.w, a.ttp, t, a.k, a.H, c);
    const uint32_t lo =
        (uint32_t)float_to_bf16_rn(acc.x) | ((uint32_t)float_to_bf16_rn(acc.y) << 16);
    const uint32_t hi =
        (uint32_t)float_to_bf16_rn(acc.z) | ((uint32_t)float_to_bf16_rn(acc.w) << 16);
    *reinterpret_cast<uint2 *>(a.out + (size_t)t * a.H + c) = make_uint2(lo, hi);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------

// Maps of one call, cached by (weights, workspace, shape): encoding is host
// work that would otherwise repeat on every call.
int tc_maps(const moe_experts *X, uint8_t *xq, uint8_t *hq, int max_total, TcMaps *out) {
  struct Key {
    const void *g, *u, *d, *xq, *hq;
    int E, H, I, mt;
    bool operator==(const Key &o) const {
      return g == o.g && u == o.u && d == o.d && xq == o.xq && hq == o.hq && E == o.E &&
             H == o.H && I == o.I && mt == o.mt;
    }
  };
  struct KeyHash {
    size_t operator()(const Key &k) const {
      size_t h = std::hash<const void *>()(k.g);
      for (const void *p : {k.u, k.d, k.xq, k.hq}) h = h * 1000003u ^ std::hash<const void *>()(p);
      return h ^ ((size_t)k.E << 40) ^ ((size_t)k.H << 20) ^ (size_t)k.I ^ ((size_t)k.mt << 50);
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, TcMaps, KeyHash> cache;
  const int E = X->num_experts, H = X->hidden, I = X->inter;
  const Key key = {X->gate.codes, X->up.codes, X->down.codes, xq, hq, E, H, I, max_total};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return MOE_OK;
  }
  TcMaps m;
  const void *codes[3] = {X->gate.codes, X->up.codes, X->down.codes};
  for (int j = 0; j < 3; ++j) {
    const int K = j < 2 ? H : I, R = j < 2 ? I : H;
    // [E*R][K] seen as {128 bytes, rows, K/128 column blocks}
    const cuuint64_t dims[3] = {128, (cuuint64_t)E * R, (cuuint64_t)K / 128};
    const cuuint64_t str[2] = {(cuuint64_t)K, 128};
    for (int nb = 1; nb <= 2; ++nb) {
      const cuuint32_t box[3] = {128, 128, (cuuint32_t)nb};
      const int st = encode_u8_sw128(&m.w[j][nb - 1], codes[j], 3, dims, str, box);
      if (st) return st;
    }
  }
  for (int b = 0; b < 3; ++b) {
    const cuuint32_t xbox[3] = {128, (cuuint32_t)(16 << b), (cuuint32_t)kXTerms};
    const cuuint64_t xd[3] = {(cuuint64_t)H, (cuuint64_t)max_total, (cuuint64_t)kXTerms};
    const cuuint64_t xs[2] = {(cuuint64_t)H, (cuuint64_t)H * max_total};
    int st = encode_u8_sw128(&m.xq[b], xq, 3, xd, xs, xbox);
    if (st) return st;
    const cuuint32_t hbox[3] = {128, (cuuint32_t)(16 << b), (cuuint32_t)kHTerms};
    const cuuint64_t hd[3] = {(cuuint64_t)I, (cuuint64_t)max_total, (cuuint64_t)kHTerms};
    const cuuint64_t hs[2] = {(cuuint64_t)I, (cuuint64_t)I * max_total};
    st = encode_u8_sw128(&m.hq[b], hq, 3, hd, hs, hbox);
    if (st) return st;
  }
  {   // the token-form x-term table over the same buffer (used when M <= 16)
    const cuuint32_t tbox[3] = {128, (cuuint32_t)kTokMax, 2};
    const cuuint64_t td[3] = {128, (cuuint64_t)kTokMax, (cuuint64_t)2 * (H / 128)};
    const cuuint64_t ts[2] = {128, (cuuint64_t)kTokMax * 128};
    const int st = encode_u8_sw128(&m.xt, xq, 3, td, ts, tbox);
    if (st) return st;
  }
  if (cache.size() > 1024) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return MOE_OK;
}

constexpr size_t kSmemLimit = 227 * 1024;
// the largest stage: two k blocks of two weight tiles and of 32 rows of h
// terms, or one k block with 64 rows
constexpr size_t kMaxStage = 4 * kTileBytes + 2 * kHTerms * 32 * 128;

size_t ring_bytes_for(int cap, int KBd, int RT) {
  const size_t fixed = fixed_bytes(cap, KBd, RT);
  if (fixed + 2 * kMaxStage > kSmemLimit) return 0;
  return (kSmemLimit - fixed) / 1024 * 1024;
}

}  // namespace

// Shape admission of the tensor-core path (host): FP8 routed experts, no
// shared expert, H and I multiples of 256 (H up to 8192, I up to 4096) and
// room for the ring.
bool tc_fits(const moe_layer_desc *L, int M) {
  const moe_experts &R = L->routed;
  if (R.fmt != MOE_FMT_FP8_B128 || L->shared) return false;
  if (R.hidden % 256 || R.hidden > 128 * kMaxKB || R.inter % 256 || R.inter > 128 * kMaxKBd)
    return false;
  const int n = M * L->top_k;
  const int cap = n < R.num_experts ? n : R.num_experts;
  return ring_bytes_for(cap, R.inter / 128, M <= kTokMax ? 16 : kRowTile) != 0;
}

// Workspace of the tensor-core path: the term tables, their scales and the
// active table (byte sizes, in order: x terms, x scales, h terms, h scales,
// active table).
void tc_workspace(const moe_layer_desc *L, int M, int max_total, int cap, size_t (&bytes)[5]) {
  const size_t H = L->routed.hidden, I = L->routed.inter;
  // x terms: by sorted row, or (M <= 16) the token table [H/128][2][16][128]
  const size_t rows = M <= kTokMax ? (size_t)kTokMax : (size_t)max_total;
  bytes[0] = (size_t)kXTerms * rows * H;
  bytes[1] = rows * 4;
  bytes[2] = (size_t)kHTerms * max_total * I;
  bytes[3] = (size_t)max_total * (I / 128) * 4;
  bytes[4] = (size_t)cap * 16;
}

// Counters of the tensor-core path, in ints, sized by the layer alone: one per
// active-list index (at most E) and the item counter.
size_t tc_counter_ints(const moe_layer_desc *L) { return (size_t)L->routed.num_experts + 1; }

int launch_tc(const moe_layer_desc *L, const uint16_t *x, int M, const float *w,
              const int32_t *ttp, const int32_t *act_count, uint16_t *out, void *ws,
              const moe_workspace_view &v, uint32_t *err, void *stream) {
  const moe_experts &R = L->routed;
  char *base = static_cast<char *>(ws);
  TcArgs a = {};
  a.M = M;
  a.k = L->top_k;
  a.n = M * L->top_k;
  a.E = R.num_experts;
  a.H = R.hidden;
  a.I = R.inter;
  a.cap = v.cap;
  a.max_total = v.max_total;
  a.tok = M <= kTokMax;
  a.row_tile = a.tok ? 16 : kRowTile;
  a.x = x;
  a.w = w;
  a.ttp = ttp;
  a.sti = reinterpret_cast<const int32_t *>(base + v.sorted_token_ids);
  a.act_count = act_count;
  a.items = reinterpret_cast<const int4 *>(base + v.tc_items);
  a.out = out;
  a.sg = static_cast<const float *>(R.gate.scale);
  a.su = static_cast<const float *>(R.up.scale);
  a.sd = static_cast<const float *>(R.down.scale);
  a.xq = reinterpret_cast<uint8_t *>(base + v.tc_x_terms);
  a.xs = reinterpret_cast<float *>(base + v.tc_x_scale);
  a.hq = reinterpret_cast<uint8_t *>(base + v.tc_h_terms);
  a.hs = reinterpret_cast<float *>(base + v.tc_h_scale);
  a.h = reinterpret_cast<float *>(base + v.h);
  a.y = reinterpret_cast<float *>(base + v.y);
  a.done = reinterpret_cast<int *>(base + v.tc_done);
  a.work = a.done + a.E;
  a.grid_ctr = reinterpret_cast<unsigned long long *>(base + v.blend_counters);
  a.err = err;
  const size_t ring = ring_bytes_for(v.cap, a.I / 128, a.row_tile);
  if (!ring) return MOE_EUNSUPPORTED;
  a.ring_bytes = (uint32_t)ring;
  TcMaps maps;
  int st = tc_maps(&R, a.xq, a.hq, v.max_total, &maps);
  if (st) return st;
  const size_t smem = ring + fixed_bytes(v.cap, a.I / 128, a.row_tile);
  st = ensure_smem_limit((const void *)verify_ffn_kernel, smem);
  if (st) return st;
  return launch_pdl_coop(verify_ffn_kernel, dim3(sm_count()), dim3(kThreads), smem, stream, a,
                         maps);
}

}  // namespace moe
