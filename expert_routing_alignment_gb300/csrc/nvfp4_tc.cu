// nvfp4_tc.cu -- the grouped expert FFN of the decode MoE layer on the tensor
// cores for NVFP4 experts (E2M1 codes, one E4M3 scale per 16 elements, an
// fp32 global per expert and projection), batches of up to 32 rows.
//
// What it computes is the same as the CUDA-core kernels: for every active
// expert e and every real sorted position p of its run, token t,
//   h[p] = silu(Wg[e] . x[t]) * (Wu[e] . x[t])        (fp32)
//   y[p] = Wd[e] . h[p]                                (fp32)
//   out[t] = bf16(sum_j w[t][j] * y[token_to_perm[t*k+j]] + g[t] * y_sh[t])
// with w = e2m1(code) * e4m3(scale[o][k/16]) * global ("forward_nvfp4_grouped_
// decode.rs": the NVFP4 layer and its tensor-core twins of the grouped
// kernels; the SwiGLU product and fixed-order combine of "moe_decode_vec.py").
//
// How, on sm_103a:
//  * Exact f16 operands.  E2M1 times an E4M3 scale has at most 6 significant
//    bits and lies in [2^-10, 2688], so the weight w / global is an exact f16;
//    four decoder warps turn each 128 x 128 tile of codes (copied to shared
//    memory by TMA) into f16 and write it straight into tensor memory
//    (tcgen05.st: lane = weight row, 32-bit column c = k 2c and 2c+1), where
//    the MMA reads its A operand (kind::f16, A in TMEM, B in shared memory):
//    the decoded weights never touch shared memory.  x enters as one f16
//    term under a power-of-two scale per token (bf16 has 8 significant bits),
//    h as two f16 terms (hi + lo, 22 bits) under a power-of-two scale per
//    (row, 128-column block).
//  * Token columns.  The gate+up MMAs take the batch's 16 or 32 token columns
//    of a per-token x table at once.  The table (and the shared expert's
//    gates) come from extra CTAs of the alignment launch, complete when this
//    kernel's programmatic-dependency wait returns: the first copies wait for
//    nothing else.
//  * Every 128-wide k block is accumulated alone in TMEM and added in fp32 in
//    a fixed order (times the row's h scale for down); the global scale is
//    applied once per item.  Items (expert row tile, 128-row gate+up tile),
//    then (row tile, pair of 128-row down tiles), are taken dynamically; a
//    down item waits (bounded) until its expert's gate+up tiles are counted.
//  * FP8 items.  The FP8 shared expert (its items follow the routed ones of
//    each kind) and the FP8 down projection of the nvfp4-gate-up tier run in
//    the same kernel: their E4M3 codes decode to exact f16 and the 128 x 128
//    block scale is applied when each k block is promoted.
//  * Roles: warp 0 copies, warp 1 issues MMAs, warps 2-5 decode, warps 6-13
//    promote (two groups of four: token columns 0-15 and 16-31).  After a
//    grid barrier every CTA blends its share of the outputs.  Every wait
//    gives up after about two seconds with MOE_ERR_TIMEOUT.
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kDecWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kEpi0 = 2 + kDecWarps;            // first promotion warp
constexpr int kWarps = kEpi0 + kEpiWarps;       // 14
constexpr int kThreads = kWarps * 32;           // 448
constexpr int kEpiThreads = kEpiWarps * 32;     // 256
constexpr int kRecs = 8;                        // stage records
constexpr int kKd = 32;                         // k-block completion barriers
constexpr int kTfree = 16;                      // per-stage TMEM release barriers
constexpr int kIQ = 32;                         // item queue
constexpr int kAbuf = 4;                        // TMEM A buffers (one tile k block each)
constexpr uint32_t kAcols = 64;                 // 128 k of f16 per row: 64 columns
constexpr uint32_t kAccBase = kAbuf * kAcols;   // accumulators above the A buffers
constexpr uint32_t kAccCols = 512 - kAccBase;
constexpr int kRows = 16;                       // rows per item
constexpr int kTokMax = 32;                     // token columns at most
constexpr int kMaxKBd = 32;                     // down k blocks (I <= 4096)
constexpr int kCodeTile = 128 * 128;            // codes of one tile, two k blocks
constexpr int kScaleTile = 128 * 16;            // scales of one tile, two k blocks
constexpr int kHAtom = 2 * kRows * 128;         // one 64-k atom of the h terms
constexpr int kMaxKB = 64;                      // gate+up k blocks (H <= 8192)

struct F4Args {
  int M, k, n, E, H, I, cap, max_total, NT;
  const uint16_t *x;
  const float *w;                            // [n] routing weight of each slot
  const int32_t *ttp, *sti, *act_count;      // the alignment's tables
  const int4 *items;                         // [cap] {offset, expert, slot count, 0}
  uint16_t *out;                             // [M][H] bf16
  const float *gg, *gu, *gd;                 // global scales [E] (gd NULL: FP8 down)
  // the nvfp4-gate-up tier: the routed down projection in FP8 (E4M3 codes
  // [E][H][I], block scales [E][H/128][I/128])
  int down_fp8;
  const float *sdown;
  const uint8_t *xt;                         // f16 x table [H/128][2 atoms][NT][128 B]
  const float *xs;                           // [32] 2^-s of each token
  uint16_t *hq;                              // f16 h terms [2][max_total][I]
  float *hs;                                 // [max_total][I/128] 2^-s per (row, block)
  float *h, *y;                              // [max_total][I], [max_total][H]
  // the FP8 shared expert (Is = its inter; 0 without one): rows are tokens
  int Is;
  const float *ssg, *ssu, *ssd;              // its block scales [Is/128][H/128], [H/128][Is/128]
  uint16_t *hq_sh;                           // f16 h terms [2][32][Is]
  float *hs_sh;                              // [32][Is/128]
  float *h_sh, *y_sh;                        // [M][Is], [M][H]
  int gated;                                 // the shared term is gated
  const float *gate_vals;                    // [M] the gates (written with the x table)
  int *done, *work;
  unsigned long long *grid_ctr;
  uint32_t *err;
  uint32_t ring_bytes;
};

// Codes {K/2 bytes, E*R rows} box {128, 128} (two k blocks, 128-byte swizzle);
// scales {K/16 bytes, E*R rows} box {16, 128}; the x table {128, NT, 2 KB}
// box {128, NT, 4}; the h terms {2 I bytes, max_total, 2} box {128, 16, 2};
// the shared expert's E4M3 codes {K bytes, R rows} box {128, 128} (one k
// block) and its h terms {2 Is bytes, 32, 2} box {128, 16, 2}.
struct F4Maps {
  CUtensorMap codes[3], scales[3];
  CUtensorMap xt, hq;
  CUtensorMap scodes[3], hq_sh;
};

struct Smem {
  uint8_t *ring;
  uint64_t *full, *kdone, *tfree, *iqbar, *afull, *drain;
  volatile int *iq;
  uint32_t *rec, *rlen, *trec;
  int *twait, *kend;    // [kRecs] the stage's TMEM wait, its last k block
  volatile int *misc;   // [0] failed, [1] TMEM base, [3] row tiles, [4] grid barrier passed
  float *cs;            // [kMaxKBd][kRows] down: per-row h factors of the current item
  float *xinv;          // [kRows] gate+up: 2^-s of each row's token
  int *tokrow;          // [kRows] each row's token
  float *xtok;          // [kTokMax] 2^-s of each token
  float *glob;          // [2] the item's global scales
  float *fs;            // [2][kMaxKB] shared items: each tile's block scale per k block
  uint32_t *red;        // [2 groups][4 quadrants][16] column maxima
  int *rtp;             // [cap + 1]
  int2 *info;           // [cap] {offset, expert | rows << 16}
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) & ~size_t(15); }
constexpr int kBars = kRecs + kKd + kTfree + kIQ + kAbuf + 1;

__host__ __device__ inline size_t fixed_bytes(int cap) {
  size_t b = al16(8 * kBars);
  b += 5 * al16(4 * kRecs) + al16(4 * kIQ) + al16(4 * 16);
  b += al16(4 * kMaxKBd * kRows) + al16(4 * kRows) + al16(4 * kRows) + al16(4 * kTokMax) +
       al16(4 * 2) + al16(4 * 2 * kMaxKB) + al16(4 * 2 * 4 * 16);
  b += al16(4 * ((size_t)cap + 1)) + al16(8 * (size_t)cap);
  return b;
}

__device__ Smem carve(uint8_t *base, const F4Args &a) {
  Smem S;
  S.ring = base;
  uint8_t *p = base + a.ring_bytes;
  auto take = [&](size_t bytes) {
    uint8_t *r = p;
    p += al16(bytes);
    return r;
  };
  uint64_t *b = reinterpret_cast<uint64_t *>(take(8 * kBars));
  S.full = b;
  S.kdone = S.full + kRecs;
  S.tfree = S.kdone + kKd;
  S.iqbar = S.tfree + kTfree;
  S.afull = S.iqbar + kIQ;
  S.drain = S.afull + kAbuf;
  S.rec = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.rlen = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.trec = reinterpret_cast<uint32_t *>(take(4 * kRecs));
  S.twait = reinterpret_cast<int *>(take(4 * kRecs));
  S.kend = reinterpret_cast<int *>(take(4 * kRecs));
  S.iq = reinterpret_cast<volatile int *>(take(4 * kIQ));
  S.misc = reinterpret_cast<volatile int *>(take(4 * 16));
  S.cs = reinterpret_cast<float *>(take(4 * kMaxKBd * kRows));
  S.xinv = reinterpret_cast<float *>(take(4 * kRows));
  S.tokrow = reinterpret_cast<int *>(take(4 * kRows));
  S.xtok = reinterpret_cast<float *>(take(4 * kTokMax));
  S.glob = reinterpret_cast<float *>(take(4 * 2));
  S.fs = reinterpret_cast<float *>(take(4 * 2 * kMaxKB));
  S.red = reinterpret_cast<uint32_t *>(take(4 * 2 * 4 * 16));
  S.rtp = reinterpret_cast<int *>(take(4 * ((size_t)a.cap + 1)));
  S.info = reinterpret_cast<int2 *>(take(8 * (size_t)a.cap));
  return S;
}

__device__ __forceinline__ void fail(const Smem &S, const F4Args &a) {
  if (!S.misc[0]) {
    S.misc[0] = 1;
    if (a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
  }
}
__device__ __forceinline__ bool wait_bar(const Smem &S, uint64_t *bar, uint32_t parity) {
  return wait_phase(S.misc, bar, parity);
}
__device__ __forceinline__ int next_item(const Smem &S, int j) {
  if (!wait_bar(S, &S.iqbar[j % kIQ], (uint32_t)(j / kIQ) & 1)) return -1;
  return S.iq[j % kIQ];
}
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}
// Barrier over the promotion warps that also ORs a flag across them.
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
__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory");
}

// ---------------------------------------------------------------------------
// items
// ---------------------------------------------------------------------------

// An item: a 128-row gate+up tile (or a pair of 128-row down tiles) of one
// 16-row tile of an expert's rows.  Shared-expert items (sh) have the tokens
// as rows (pos0 = first token) and stream one E4M3 k block per stage; the
// routed NVFP4 items two.  Item order: routed gate+up, shared gate+up, routed
// down, shared down (every gate+up item is taken before any down item).
struct Item {
  bool gu, sh;
  bool f8;   // E4M3 codes (the shared expert; the tier's routed down): one k block per stage
  int a, e, pos0, rows, tile;
};

struct Counts {
  int TR, FT, FD, TRs, FTs;   // routed row tiles, tiles; shared row tiles, tiles
};

__device__ __forceinline__ Item decode(const Smem &S, const F4Args &a, int A, int i,
                                       const Counts &c) {
  Item it;
  const int G = c.TR * c.FT, Gs = c.TRs * c.FTs, D = c.TR * c.FD;
  if ((i >= G && i < G + Gs) || i >= G + Gs + D) {   // the shared expert
    const bool gu = i < G + Gs;
    const int j = gu ? i - G : i - G - Gs - D, per = gu ? c.FTs : c.FD;
    const int rt = j / per;
    it.gu = gu;
    it.sh = true;
    it.f8 = true;
    it.tile = j - rt * per;
    it.a = A;
    it.e = 0;
    it.pos0 = rt * kRows;
    it.rows = min(kRows, a.M - rt * kRows);
    return it;
  }
  it.sh = false;
  int rtg;
  if (i < G) {
    it.gu = true;
    rtg = i / c.FT;
    it.tile = i - rtg * c.FT;
  } else {
    it.gu = false;
    const int j = i - G - Gs;
    rtg = j / c.FD;
    it.tile = j - rtg * c.FD;
  }
  it.f8 = !it.gu && a.down_fp8;
  int lo = 0, hi = A - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.rtp[mid] <= rtg)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int2 inf = S.info[lo];
  const int rt = rtg - S.rtp[lo];
  it.a = lo;
  it.e = inf.y & 0xFFFF;
  it.pos0 = inf.x + rt * kRows;
  it.rows = min(kRows, (inf.y >> 16) - rt * kRows);
  return it;
}

// The MMA's N (gate+up: the token columns; down: two terms of 16 rows), the
// bytes of a stage's B operand (two k blocks = four 64-k atoms), of a whole
// stage (B, then the codes and scales of two weight tiles), and the TMEM
// columns of one k block's accumulators (two tiles).
__device__ __forceinline__ int item_n(const Item &it, int NT) { return it.gu ? NT : 2 * kRows; }
__device__ __forceinline__ uint32_t b_bytes(const Item &it, int NT) {
  return it.gu ? 4u * (uint32_t)NT * 128u : 4u * kHAtom;
}
__device__ __forceinline__ uint32_t stage_bytes(const Item &it, int NT) {
  return b_bytes(it, NT) + 2u * kCodeTile + (it.f8 ? 0u : 2u * kScaleTile);
}
__device__ __forceinline__ uint32_t acc_cols(const Item &it, int NT) {
  return 2u * (uint32_t)item_n(it, NT);
}
// k blocks of the item, and per stage
__device__ __forceinline__ int item_kb(const Item &it, const F4Args &a) {
  return it.gu ? a.H / 128 : (it.sh ? a.Is : a.I) / 128;
}
__device__ __forceinline__ int stage_kbs(const Item &it) { return it.f8 ? 1 : 2; }

// ---------------------------------------------------------------------------
// roles
// ---------------------------------------------------------------------------

// The gate+up tiles an expert's down items wait for (routed: its row tiles
// times I/128; the shared expert: its row tiles times Is/128).
__device__ __forceinline__ int gu_tiles(const Smem &S, const Item &it, const Counts &c) {
  return it.sh ? c.TRs * c.FTs : (S.rtp[it.a + 1] - S.rtp[it.a]) * c.FT;
}

__device__ void producer(const F4Args &a, const F4Maps &m, const Smem &S, int A,
                         const Counts &c, int total) {
  const uint64_t pol = policy_evict_first();
  const int NT = a.NT;
  uint32_t head = 0, thead = 0;
  int s = 0, tail = 0, ttail = 0, jq = 0, kq = -1;
  bool ok = true;
  int i = (int)blockIdx.x < total ? (int)blockIdx.x : total;
  while (i < total && ok) {
    S.iq[jq % kIQ] = i;
    mbar_arrive(&S.iqbar[jq % kIQ]);
    ++jq;
    const Item it = decode(S, a, A, i, c);
    if (!it.gu) {
      if (!wait_at_least(S.misc, a.done + it.a, gu_tiles(S, it, c))) {
        ok = false;
        break;
      }
      fence_proxy_async_global();
    }
    const int KB = item_kb(it, a), kbs = stage_kbs(it);
    const uint32_t size = stage_bytes(it, NT), bb = b_bytes(it, NT);
    const uint32_t tcols = (uint32_t)kbs * acc_cols(it, NT);
    const int p0 = it.gu ? 0 : 2, p1 = it.gu ? 1 : 2;
    const int R = it.gu ? (it.sh ? a.Is : a.I) : a.H;
    const int row0 = it.e * R + it.tile * (it.gu ? 128 : 256);
    const int row1 = it.gu ? row0 : row0 + 128;
    for (int kb = 0; kb < KB; kb += kbs) {
      int need_t = -1;
      {
        const bool twrap = thead + tcols > kAccCols;
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
        const int ke = S.kend[dt];   // the stage's last k block: all its MMAs are done
        if (!wait_bar(S, &S.kdone[ke % kKd], (uint32_t)(ke / kKd) & 1)) {
          ok = false;
          break;
        }
        ++tail;
      }
      if (!ok) break;
      const uint32_t pos = ring_place(head, size, a.ring_bytes);
      const uint32_t tpos = ring_place(thead, tcols, kAccCols);
      const int d = s % kRecs;
      kq += kbs;
      S.rec[d] = pos;
      S.rlen[d] = size;
      S.trec[d] = tpos | (tcols << 16);
      S.twait[d] = need_t;
      S.kend[d] = kq;
      uint64_t *fb = &S.full[d];
      mbar_expect_tx(fb, size);
      uint8_t *dst = S.ring + pos;
      if (it.f8) {   // one E4M3 k block of each tile
        const CUtensorMap *cm = it.sh ? m.scodes : m.codes;
        tma_2d_hint(dst + bb, &cm[p0], kb * 128, row0, fb, pol);
        tma_2d_hint(dst + bb + kCodeTile, &cm[p1], kb * 128, row1, fb, pol);
      } else {       // two k blocks of E2M1 codes and their scales
        tma_2d_hint(dst + bb, &m.codes[p0], kb * 64, row0, fb, pol);
        tma_2d_hint(dst + bb + kCodeTile, &m.codes[p1], kb * 64, row1, fb, pol);
        tma_2d_hint(dst + bb + 2 * kCodeTile, &m.scales[p0], kb * 8, row0, fb, pol);
        tma_2d_hint(dst + bb + 2 * kCodeTile + kScaleTile, &m.scales[p1], kb * 8, row1, fb, pol);
      }
      // the B operand: 4 atoms of 64 k (a shared stage uses the first two;
      // atoms past the end read as zeros)
      if (it.gu) {
        tma_3d(dst, &m.xt, 0, 0, 2 * kb, fb);   // x 4 atoms x NT tokens
      } else {
        const CUtensorMap *hm = it.sh ? &m.hq_sh : &m.hq;
        for (int at4 = 0; at4 < 4; ++at4)         // 4 atoms x (2 terms x 16 rows)
          tma_3d(dst + at4 * kHAtom, hm, kb * 256 + at4 * 128, it.pos0, 0, fb);
      }
      ++s;
    }
    i = (int)gridDim.x + atomicAdd(a.work, 1);
  }
  S.iq[jq % kIQ] = total;
  mbar_arrive(&S.iqbar[jq % kIQ]);
  if (!ok) fail(S, a);
  for (int j = max(tail, s - kRecs); j < s; ++j) {
    const uint64_t t0 = gtime();
    while (!mbar_poll(&S.full[j % kRecs], (uint32_t)(j / kRecs) & 1))
      if (gtime() - t0 > kWaitNs) break;
  }
}

// One weight row's 128 k of a routed tile (k block kbl of the two in the
// 128-byte row): w / global = e2m1 * e4m3 scale, exact in f16, as 64 packed
// pairs (column c = k 2c, 2c + 1).  The row's bytes sit in 16-byte chunks
// permuted by the 128-byte swizzle (chunk j at j ^ (row % 8)).
__device__ __forceinline__ void decode_e2m1(const uint8_t *crow, const uint8_t *srow, int r,
                                            int kbl, uint32_t (&v)[64]) {
  const uint2 sv = *reinterpret_cast<const uint2 *>(srow + kbl * 8);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int chunk = kbl * 4 + c;   // 16 bytes: 32 codes, groups 2c and 2c + 1
    const uint4 cv = *reinterpret_cast<const uint4 *>(crow + ((chunk ^ (r & 7)) << 4));
    const uint32_t words[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
      const int g = 2 * c + g2;
      const uint32_t sbyte = (g < 4 ? sv.x >> (8 * g) : sv.y >> (8 * (g - 4))) & 0xFFu;
      const uint32_t s2 = e4m3x2_to_f16x2((uint16_t)(sbyte | (sbyte << 8)));
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t byte = (words[g2 * 2 + b / 4] >> (8 * (b % 4))) & 0xFFu;
        uint32_t f = e2m1x2_to_f16x2(byte);
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(f) : "r"(s2));
        v[c * 16 + g2 * 8 + b] = f;
      }
    }
  }
}

// One weight row's 128 k of a shared-expert tile: the E4M3 codes as f16
// (exact); the block scale is applied when the k block is promoted.
__device__ __forceinline__ void decode_e4m3(const uint8_t *crow, int r, uint32_t (&v)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 cv = *reinterpret_cast<const uint4 *>(crow + ((c ^ (r & 7)) << 4));
    const uint32_t words[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
    for (int p = 0; p < 8; ++p)
      v[c * 8 + p] = e4m3x2_to_f16x2((uint16_t)((words[p / 2] >> (16 * (p % 2))) & 0xFFFFu));
  }
}

// Warps 2-5: each thread decodes one weight row (warp w: rows 32 (w % 4) ..)
// of a tile's k block into an A buffer of tensor memory.
__device__ void decoder(const F4Args &a, const Smem &S, int A, const Counts &cn, int total,
                        uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
  const int r = q * 32 + lane;
  const int NT = a.NT;
  const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
  uint32_t head = 0;
  int s = 0, abn = 0;
  bool ok = true;
  for (int jq = 0; ok; ++jq) {
    int i = next_item(S, jq);
    i = __shfl_sync(0xFFFFFFFFu, i, 0);
    if (i < 0) {
      ok = false;
      break;
    }
    if (i >= total) break;
    const Item it = decode(S, a, A, i, cn);
    const int KB = item_kb(it, a), kbs = stage_kbs(it);
    const uint32_t size = stage_bytes(it, NT), bb = b_bytes(it, NT);
    for (int kb = 0; kb < KB && ok; kb += kbs) {
      const uint32_t pos = ring_place(head, size, a.ring_bytes);
      const int d = s % kRecs;
      if (!__all_sync(0xFFFFFFFFu, wait_bar(S, &S.full[d], (uint32_t)(s / kRecs) & 1))) {
        ok = false;
        break;
      }
      const uint8_t *codes = S.ring + pos + bb;
      const uint8_t *scales = codes + 2 * kCodeTile;
      for (int kbl = 0; kbl < kbs && ok; ++kbl)
        for (int t = 0; t < 2; ++t) {
          const int ab = abn % kAbuf;
          if (abn >= kAbuf) {   // the k block that read this buffer (two buffers per k block)
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar(S, &S.kdone[(abn / 2 - 2) % kKd],
                                     (uint32_t)((abn / 2 - 2) / kKd) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();   // the MMAs that read the buffer are complete
          }
          const uint8_t *crow = codes + t * kCodeTile + r * 128;
          uint32_t v[64];
          if (it.f8)
            decode_e4m3(crow, r, v);
          else
            decode_e2m1(crow, scales + t * kScaleTile + r * 16, r, kbl, v);
          tmem_st64(lane_base + (uint32_t)ab * kAcols, v);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.afull[ab]);
          ++abn;
        }
      ++s;
    }
  }
  if (!ok) fail(S, a);
}

__device__ void mma_issuer(const F4Args &a, const Smem &S, int A, const Counts &cn, int total,
                           uint32_t tmem) {
  const int NT = a.NT;
  const uint32_t ring = smem_addr(S.ring);
  uint32_t head = 0, thead = 0;
  int s = 0, q = 0, abn = 0, tdone = -1;
  bool ok = true;
  for (int jq = 0; ok; ++jq) {
    const int i = next_item(S, jq);
    if (i < 0) ok = false;
    if (i < 0 || i >= total) break;
    const Item it = decode(S, a, A, i, cn);
    const int KB = item_kb(it, a), kbs = stage_kbs(it);
    const int N = item_n(it, NT);
    const uint32_t id = idesc_f16(N), cols = acc_cols(it, NT);
    const uint32_t size = stage_bytes(it, NT), tcols = (uint32_t)kbs * cols;
    const uint32_t atom_bytes = it.gu ? (uint32_t)NT * 128u : (uint32_t)kHAtom;
    for (int kb = 0; kb < KB; kb += kbs) {
      const uint32_t base = ring + ring_place(head, size, a.ring_bytes);
      const uint32_t tbase = tmem + kAccBase + ring_place(thead, tcols, kAccCols);
      const int d = s % kRecs;
      if (!wait_bar(S, &S.full[d], (uint32_t)(s / kRecs) & 1)) {
        ok = false;
        break;
      }
      const int tw = S.twait[d];
      while (tdone < tw && ok) {
        ++tdone;
        if (!wait_bar(S, &S.tfree[tdone % kTfree], (uint32_t)(tdone / kTfree) & 1)) ok = false;
      }
      if (!ok) break;
      // the stage's B operand: a descriptor moves by (bytes / 16)
      const uint64_t bd0 = sdesc(base);
      const uint32_t astep = atom_bytes >> 4;
      for (int kbl = 0; kbl < kbs && ok; ++kbl) {
        for (int t = 0; t < 2; ++t) {
          const int ab = abn % kAbuf;
          if (!wait_bar(S, &S.afull[ab], (uint32_t)(abn / kAbuf) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dcol = tbase + (uint32_t)kbl * cols + (uint32_t)t * (uint32_t)N;
          const uint32_t acol = tmem + (uint32_t)ab * kAcols;
          const uint64_t bk = bd0 + (uint64_t)(2u * (uint32_t)kbl * astep);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ta(dcol, acol + (uint32_t)ks * 8u,
                       bk + (uint64_t)((uint32_t)(ks >> 2) * astep + (uint32_t)(ks & 3) * 2u), id,
                       ks != 0);
          ++abn;
        }
        if (!ok) break;
        // One commit per k block (each commit costs the tensor pipe about as
        // much as two MMAs): it frees the k block's two A buffers, hands its
        // accumulators to the promotion, and after the stage's last k block
        // frees the ring stage.
        mma_commit(&S.kdone[q % kKd]);
        ++q;
      }
      if (!ok) break;
      ++s;
    }
  }
  if (!ok) fail(S, a);
  mma_commit(S.drain);
  const uint64_t t0 = gtime();
  while (!mbar_poll(S.drain, 0))
    if (gtime() - t0 > kWaitNs) break;
}

// Gate+up finish by promotion group g: the rows whose token is one of the
// group's 16 columns; h = silu(g) * u as fp32 and as two f16 terms
// (hi = f16(h 2^s), lo = f16(h 2^s - hi)) with s putting the (row, tile)
// maximum in [2^14, 2^15).
__device__ void finish_gate_up(const F4Args &a, const Smem &S, const Item &it, int grp, int q,
                               int lane, const float (&acc0)[16], const float (&acc1)[16]) {
  const int f = q * 32 + lane, o = it.tile * 128 + f;
  // routed rows by sorted position, the shared expert's by token
  const int Iw = it.sh ? a.Is : a.I, KBd = Iw / 128;
  float *const hb = it.sh ? a.h_sh : a.h;
  uint16_t *const hqb = it.sh ? a.hq_sh : a.hq;
  float *const hsb = it.sh ? a.hs_sh : a.hs;
  const size_t plane = it.sh ? (size_t)kTokMax * a.Is : (size_t)a.max_total * a.I;
  const float g0 = S.glob[0], g1 = S.glob[1];
  float hv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) hv[j] = 0.f;
  // only the item's rows (a uniform bound: the unrolled rows keep their registers)
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= it.rows) break;
    const int t = S.tokrow[j] - 16 * grp;
    const bool mine = t >= 0 && t < 16;
    uint32_t mx = 0;
    if (mine) {
      float gv = 0.f, uv = 0.f;
#pragma unroll
      for (int tt = 0; tt < 16; ++tt) {
        gv = tt == t ? acc0[tt] : gv;
        uv = tt == t ? acc1[tt] : uv;
      }
      const float xi = S.xinv[j];
      hv[j] = silu_f32(gv * g0 * xi) * (uv * g1 * xi);
      hb[(size_t)(it.pos0 + j) * Iw + o] = hv[j];
      mx = __float_as_uint(fabsf(hv[j]));
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) S.red[(grp * 4 + q) * 16 + j] = mx;
  }
  group_sync(grp);
  float scl = 1.f;
  if (lane < 16) {
    uint32_t mx = 0;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) mx = max(mx, S.red[(grp * 4 + qq) * 16 + lane]);
    int sh = 0;
    if (mx) {
      const int e = (int)(mx >> 23) - 127;
      sh = 14 - e;
      sh = sh < -126 ? -126 : (sh > 126 ? 126 : sh);
    }
    scl = pow2f(sh);
    const int t = S.tokrow[lane] - 16 * grp;
    if (q == 0 && lane < it.rows && t >= 0 && t < 16)
      hsb[(size_t)(it.pos0 + lane) * KBd + it.tile] = pow2f(-sh);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j >= it.rows) break;
    const float sj = __shfl_sync(0xFFFFFFFFu, scl, j);
    const int t = S.tokrow[j] - 16 * grp;
    if (t >= 0 && t < 16) {
      const float v = hv[j] * sj;
      const uint16_t hi = f16_rn(v);
      const uint16_t lo = f16_rn(v - f16_to_f32(hi));
      uint16_t *dst = hqb + (size_t)(it.pos0 + j) * Iw + o;
      dst[0] = hi;
      dst[plane] = lo;
    }
  }
}

// acc[j] += f * (column value) (gate+up), or acc[j] += hf[j] f (term 0 +
// term 1) (down), for 16 columns of this warp's lanes; f is the k block's
// block scale for E4M3 items (1 for the NVFP4 items, whose scales are in the
// decoded weights).
__device__ __forceinline__ void promote_gu(uint32_t col, float f, float (&acc)[16]) {
  uint32_t r[16];
  tmem_ld16(col, r);
  tmem_wait_ld();
#pragma unroll
  for (int jj = 0; jj < 16; ++jj) acc[jj] = fmaf(f, __uint_as_float(r[jj]), acc[jj]);
}
__device__ __forceinline__ void promote_dn(uint32_t col, const float *hf, float f,
                                           float (&acc)[16]) {
  uint32_t r[16], r2[16];
  tmem_ld16(col, r);
  tmem_ld16(col + kRows, r2);
  tmem_wait_ld();
#pragma unroll
  for (int jj = 0; jj < 16; ++jj)
    acc[jj] = fmaf(hf[jj] * f, __uint_as_float(r[jj]) + __uint_as_float(r2[jj]), acc[jj]);
}

// Warps 6-13: group g = (w - 6) / 4 holds token columns 16 g .. 16 g + 15 of a
// gate+up item; group 0 the 16 rows of a down item.  Warp w reads TMEM lanes
// 32 (w % 4) ..
__device__ void epilogue(const F4Args &a, const Smem &S, int A, const Counts &cn, int total,
                         uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = (warp - kEpi0) >> 2, q = warp & 3;
  const int et = threadIdx.x - kEpi0 * 32;
  const int NT = a.NT, KBh = a.H / 128;
  const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
  int s = 0, st = 0;
  uint32_t thead = 0;
  bool bad = false;
  if (et < a.M) S.xtok[et] = __ldcg(a.xs + et);   // the x table is complete at launch
  epi_sync();
  for (int jq = 0;; ++jq) {
    int i = next_item(S, jq);
    i = __shfl_sync(0xFFFFFFFFu, i, 0);
    if (epi_sync_or(i < 0 || bad)) {
      bad = true;
      break;
    }
    if (i >= total) break;
    const Item it = decode(S, a, A, i, cn);
    const int KB = item_kb(it, a), kbs = stage_kbs(it);
    const int KBd = (it.sh ? a.Is : a.I) / 128;
    // the item's rows, scales and (down) its dependency
    if (et == 0 && !it.gu && !wait_at_least(S.misc, a.done + it.a, gu_tiles(S, it, cn)))
      fail(S, a);
    if (et < kRows) {
      int t = 0;
      if (et < it.rows) t = it.sh ? it.pos0 + et : __ldcg(a.sti + it.pos0 + et) / a.k;
      S.tokrow[et] = et < it.rows ? t : -1;
      S.xinv[et] = et < it.rows ? S.xtok[t] : 0.f;
    }
    if (et == 0) {
      S.glob[0] = it.sh || it.f8 ? 1.f : (it.gu ? __ldg(a.gg + it.e) : __ldg(a.gd + it.e));
      S.glob[1] = it.sh ? 1.f : (it.gu ? __ldg(a.gu + it.e) : 0.f);
    }
    // (the down item's h scales are read only after the dependency wait)
    if (epi_sync_or(S.misc[0])) {
      bad = true;
      break;
    }
    if (it.f8) {   // each tile's block scale per k block
      const float *sd = it.sh ? a.ssd : a.sdown + (size_t)it.e * KBh * KBd;
      for (int idx = et; idx < 2 * KB; idx += kEpiThreads) {
        const int t = idx / KB, kb = idx - t * KB;
        S.fs[t * kMaxKB + kb] = it.gu ? __ldg((t ? a.ssu : a.ssg) + it.tile * KBh + kb)
                                      : __ldg(sd + (2 * it.tile + t) * KBd + kb);
      }
    }
    if (!it.gu) {
      const float *hsb = it.sh ? a.hs_sh : a.hs;
      for (int idx = et; idx < KB * kRows; idx += kEpiThreads) {
        const int kb = idx / kRows, j = idx - kb * kRows;
        S.cs[idx] = j < it.rows ? __ldcg(hsb + (size_t)(it.pos0 + j) * KBd + kb) : 0.f;
      }
    }
    if (it.f8 || !it.gu) epi_sync();
    float acc0[16], acc1[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) acc0[jj] = acc1[jj] = 0.f;
    const int N = item_n(it, NT);
    const uint32_t cols = acc_cols(it, NT), tcols = (uint32_t)kbs * cols;
    // Only the groups that hold columns of the item read TMEM; the first
    // warp also arrives for the warps of the other group, which skip the
    // k blocks.
    const bool mine = it.gu ? 16 * grp < NT : grp == 0;
    const int nmine = it.gu && NT > 16 ? kEpiWarps : 4;
    const uint32_t arrivals = warp == kEpi0 ? (uint32_t)(kEpiWarps - nmine + 1) : 1u;
    if (!mine) {
      for (int kb = 0; kb < KB; kb += kbs) ring_place(thead, tcols, kAccCols);
      s += KB;
      st += KB / kbs;
    }
    uint32_t tbase = 0;
    for (int kb = 0; kb < KB && mine; ++kb) {
      const int j = kb % kbs;
      if (j == 0) tbase = ring_place(thead, tcols, kAccCols);
      // every lane of the warp takes the same branch into the aligned TMEM loads
      if (!__all_sync(0xFFFFFFFFu, wait_bar(S, &S.kdone[s % kKd], (uint32_t)(s / kKd) & 1))) {
        bad = true;
        break;
      }
      tc_fence_after();
      const uint32_t col = lane_base + kAccBase + tbase + (uint32_t)j * cols;
      const float f0 = it.f8 ? S.fs[kb] : 1.f, f1 = it.f8 ? S.fs[kMaxKB + kb] : 1.f;
      if (it.gu) {
        promote_gu(col + 16u * (uint32_t)grp, f0, acc0);
        promote_gu(col + (uint32_t)N + 16u * (uint32_t)grp, f1, acc1);
      } else {
        promote_dn(col, S.cs + kb * kRows, f0, acc0);
        promote_dn(col + (uint32_t)N, S.cs + kb * kRows, f1, acc1);
      }
      ++s;
      if (j == kbs - 1) {   // the stage's accumulators are free
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_n(&S.tfree[st % kTfree], arrivals);
        ++st;
      }
    }
    if (epi_sync_or(bad)) {
      bad = true;
      break;
    }
    if (it.gu) {
      if (mine) finish_gate_up(a, S, it, grp, q, lane, acc0, acc1);
      // every h of the tile is visible to every CTA and its tensor copies
      // before the tile is counted
      fence_proxy_async_global();
      epi_sync();
      if (et == 0) red_release_add(a.done + it.a, 1);
    } else if (mine) {
      const float gd = S.glob[0];
      const int c0 = it.tile * 256 + q * 32 + lane;
      float *const yb = it.sh ? a.y_sh : a.y;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        if (jj >= it.rows) break;
        float *yr = yb + (size_t)(it.pos0 + jj) * a.H + c0;
        yr[0] = acc0[jj] * gd;
        yr[128] = acc1[jj] * gd;
      }
    }
  }
  if (bad) fail(S, a);
}

__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_ffn_kernel(const __grid_constant__ F4Args a, const __grid_constant__ F4Maps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Smem S = carve(smem, a);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int j = 0; j < kRecs; ++j) mbar_init(&S.full[j], 1);
    for (int j = 0; j < kKd; ++j) mbar_init(&S.kdone[j], 1);
    for (int j = 0; j < kTfree; ++j) mbar_init(&S.tfree[j], kEpiWarps);
    for (int j = 0; j < kIQ; ++j) mbar_init(&S.iqbar[j], 1);
    for (int j = 0; j < kAbuf; ++j) mbar_init(&S.afull[j], kDecWarps);
    mbar_init(S.drain, 1);
    for (int j = 0; j < 16; ++j) S.misc[j] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr((const void *)(S.misc + 1))),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)S.misc[1];
  if ((smem_addr(S.ring) & 1023u) != 0) fail(S, a);

  pdl_wait();
  // the active table as 16-row tiles: info[a] = {offset, expert | rows << 16}
  // (the first kThreads entries are loaded together with the count; entries
  // past the count are read but not used)
  const int j0 = threadIdx.x;
  const int4 pre = j0 < a.cap ? __ldcg(a.items + j0) : make_int4(0, 0, 0, 0);
  const int A = min(max(__ldcg(a.act_count), 0), a.cap);
  for (int j = j0; j < A; j += kThreads) {
    const int4 inf = j == j0 ? pre : __ldcg(a.items + j);
    const int rows = min(inf.z, 0x7FFF);
    S.info[j] = make_int2(inf.x, (inf.y & 0xFFFF) | (rows << 16));
    S.rtp[j] = (rows + kRows - 1) / kRows;
  }
  __syncthreads();
  if (warp == 0) {
    const int lane = threadIdx.x & 31;
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
      S.misc[3] = run;
    }
  }
  __syncthreads();
  Counts cn;
  cn.TR = S.misc[3];
  cn.FT = a.I / 128;
  cn.FD = a.H / 256;
  cn.TRs = a.Is ? (a.M + kRows - 1) / kRows : 0;
  cn.FTs = a.Is / 128;
  const int total = S.misc[0] ? 0 : cn.TR * (cn.FT + cn.FD) + cn.TRs * (cn.FTs + cn.FD);

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) producer(a, maps, S, A, cn, total);
    __syncwarp();
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) mma_issuer(a, S, A, cn, total, tmem);
    __syncwarp();
  } else if (warp < kEpi0) {
    decoder(a, S, A, cn, total, tmem);
  } else {
    epilogue(a, S, A, cn, total, tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }

  // ---- blend: every y row is written before any CTA blends its share ------
  //   out[t][c] = bf16_rn(sum_j w[t][j] * y[token_to_perm[t*k+j]][c]
  //                       + g[t] * y_sh[t][c]), fp32, j ascending
  // (one thread's arrival with release semantics covers every write of the
  // CTA before the CTA barrier; its acquire of the full count, every write of
  // the grid)
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long G = gridDim.x;
    unsigned long long v;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(a.grid_ctr)
                 : "memory");
    const unsigned long long target = (v / G + 1) * G;
    bool ok = false;
    const uint64_t t0 = gtime();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
      unsigned long long c;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(c) : "l"(a.grid_ctr) : "memory");
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
  if (!S.misc[4] || S.misc[0]) {
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, MOE_ERR_TIMEOUT);
    return;
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= a.cap; i += kThreads) a.done[i] = 0;
    if (threadIdx.x == 0) {
      *a.work = 0;
    }
  }
  const long long T4 = (long long)a.M * a.H / 4;
  const long long o1 = T4 * (blockIdx.x + 1) / gridDim.x;
  for (long long o = T4 * blockIdx.x / gridDim.x + threadIdx.x; o < o1; o += kThreads) {
    const int t = (int)(o * 4 / a.H), c = (int)(o * 4 % a.H);
    float4 acc = blend_slots(a.y, a.w, a.ttp, t, a.k, a.H, c);
    if (a.y_sh) {
      const float gt = a.gated ? __ldcg(a.gate_vals + t) : 1.f;
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.y_sh + (size_t)t * a.H + c));
      acc.x = fmaf(gt, v.x, acc.x);
      acc.y = fmaf(gt, v.y, acc.y);
      acc.z = fmaf(gt, v.z, acc.z);
      acc.w = fmaf(gt, v.w, acc.w);
    }
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

int f4_maps(const moe_experts *X, const moe_experts *Sx, const uint8_t *xt, uint16_t *hq,
            uint16_t *hq_sh, int max_total, int NT, F4Maps *out) {
  // every address a map holds is part of the key (codes and scales of the
  // three projections, the shared expert's codes, the workspace tables)
  struct Key {
    const void *p[11];
    int E, H, I, Is, mt, nt;
    bool operator==(const Key &o) const {
      for (int j = 0; j < 11; ++j)
        if (p[j] != o.p[j]) return false;
      return E == o.E && H == o.H && I == o.I && Is == o.Is && mt == o.mt && nt == o.nt;
    }
  };
  struct KeyHash {
    size_t operator()(const Key &k) const {
      size_t h = 0;
      for (int j = 0; j < 11; ++j) h = h * 1000003u ^ std::hash<const void *>()(k.p[j]);
      return h ^ ((size_t)k.E << 40) ^ ((size_t)k.H << 20) ^ (size_t)k.I ^ ((size_t)k.mt << 50) ^
             ((size_t)k.nt << 58) ^ ((size_t)k.Is << 30);
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, F4Maps, KeyHash> cache;
  const int E = X->num_experts, H = X->hidden, I = X->inter, Is = Sx ? Sx->inter : 0;
  const Key key = {{X->gate.codes, X->up.codes, X->down.codes, X->gate.scale, X->up.scale,
                    X->down.scale, xt, hq, Sx ? Sx->gate.codes : nullptr,
                    Sx ? Sx->up.codes : nullptr, Sx ? Sx->down.codes : nullptr},
                   E * 8 + X->fmt, H, I, Is, max_total, NT};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return MOE_OK;
  }
  F4Maps m;
  memset(&m, 0, sizeof(m));
  const moe_proj *P[3] = {&X->gate, &X->up, &X->down};
  for (int j = 0; j < 3; ++j) {
    const int K = j < 2 ? H : I, R = j < 2 ? I : H;
    const cuuint32_t cbox[2] = {128, 128};
    if (proj_fmt(X->fmt, j) == MOE_FMT_FP8_B128) {   // E4M3 codes [E][R][K], one k block per box
      const cuuint64_t cd[2] = {(cuuint64_t)K, (cuuint64_t)E * R};
      const cuuint64_t cs[1] = {(cuuint64_t)K};
      const int st = encode_u8_sw128(&m.codes[j], P[j]->codes, 2, cd, cs, cbox);
      if (st) return st;
      continue;
    }
    const cuuint64_t cd[2] = {(cuuint64_t)K / 2, (cuuint64_t)E * R};
    const cuuint64_t cs[1] = {(cuuint64_t)K / 2};
    int st = encode_u8_sw128(&m.codes[j], P[j]->codes, 2, cd, cs, cbox);
    if (st) return st;
    const cuuint64_t sd[2] = {(cuuint64_t)K / 16, (cuuint64_t)E * R};
    const cuuint64_t ss[1] = {(cuuint64_t)K / 16};
    const cuuint32_t sbox[2] = {16, 128};
    st = encode_u8_plain(&m.scales[j], P[j]->scale, 2, sd, ss, sbox);
    if (st) return st;
  }
  {
    const cuuint64_t d[3] = {128, (cuuint64_t)NT, (cuuint64_t)2 * (H / 128)};
    const cuuint64_t s[2] = {128, (cuuint64_t)NT * 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)NT, 4};
    const int st = encode_u8_sw128(&m.xt, xt, 3, d, s, box);
    if (st) return st;
  }
  {
    const cuuint64_t d[3] = {(cuuint64_t)2 * I, (cuuint64_t)max_total, 2};
    const cuuint64_t s[2] = {(cuuint64_t)2 * I, (cuuint64_t)2 * I * max_total};
    const cuuint32_t box[3] = {128, (cuuint32_t)kRows, 2};
    const int st = encode_u8_sw128(&m.hq, hq, 3, d, s, box);
    if (st) return st;
  }
  if (Sx) {   // the shared expert: E4M3 codes [R][K], its h terms [2][32][Is]
    const moe_proj *Q[3] = {&Sx->gate, &Sx->up, &Sx->down};
    for (int j = 0; j < 3; ++j) {
      const int K = j < 2 ? H : Is, R = j < 2 ? Is : H;
      const cuuint64_t cd[2] = {(cuuint64_t)K, (cuuint64_t)R};
      const cuuint64_t cs[1] = {(cuuint64_t)K};
      const cuuint32_t cbox[2] = {128, 128};
      const int st = encode_u8_sw128(&m.scodes[j], Q[j]->codes, 2, cd, cs, cbox);
      if (st) return st;
    }
    const cuuint64_t d[3] = {(cuuint64_t)2 * Is, (cuuint64_t)kTokMax, 2};
    const cuuint64_t s[2] = {(cuuint64_t)2 * Is, (cuuint64_t)2 * Is * kTokMax};
    const cuuint32_t box[3] = {128, (cuuint32_t)kRows, 2};
    const int st = encode_u8_sw128(&m.hq_sh, hq_sh, 3, d, s, box);
    if (st) return st;
  }
  if (cache.size() > 1024) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return MOE_OK;
}

constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kMaxStage = 4 * kHAtom + 2 * kCodeTile + 2 * kScaleTile;

size_t ring_bytes_for(int cap) {
  const size_t fixed = fixed_bytes(cap);
  if (fixed + 2 * kMaxStage > kSmemLimit) return 0;
  return (kSmemLimit - fixed) / 1024 * 1024;
}

}  // namespace

// Shape admission (host): NVFP4 routed experts (or the nvfp4-gate-up tier:
// NVFP4 gate and up, FP8 down), M <= 32, H and I multiples of 256 (H up to
// 8192, I up to 4096), a shared expert (if any) in FP8 with its inter a
// multiple of 128 up to 4096, room for the ring.
bool f4_fits(const moe_layer_desc *L, int M) {
  const moe_experts &R = L->routed;
  if ((R.fmt != MOE_FMT_NVFP4_G16 && R.fmt != MOE_FMT_NVFP4_GATE_UP) || M > kTokMax) return false;
  if (R.hidden % 256 || R.hidden > 128 * kMaxKB || R.inter % 256 || R.inter > 128 * kMaxKBd)
    return false;
  if (L->shared && (L->shared->fmt != MOE_FMT_FP8_B128 || L->shared->inter % 128 ||
                    L->shared->inter > 128 * kMaxKBd))
    return false;
  const int n = M * L->top_k;
  const int cap = n < R.num_experts ? n : R.num_experts;
  return ring_bytes_for(cap) != 0;
}

// Workspace of this path (byte sizes, in order): the x table, the token
// scales, the h terms (routed [2][max_total][I], then the shared expert's
// [2][32][Is]), their scales (routed, then shared) and the active table.
void f4_workspace(const moe_layer_desc *L, int max_total, int cap, size_t (&bytes)[5]) {
  const size_t H = L->routed.hidden, I = L->routed.inter;
  const size_t Is = L->shared ? L->shared->inter : 0;
  bytes[0] = 2 * (size_t)kTokMax * H;
  bytes[1] = (size_t)kTokMax * 4;
  bytes[2] = 2 * 2 * ((size_t)max_total * I + (size_t)kTokMax * Is);
  bytes[3] = ((size_t)max_total * (I / 128) + (size_t)kTokMax * (Is / 128)) * 4;
  bytes[4] = (size_t)cap * 16;
}

// Counters, in ints (sized by the layer alone): done [E + 1] (the last one
// can be the shared expert's), the item counter.
size_t f4_counter_ints(const moe_layer_desc *L) { return (size_t)L->routed.num_experts + 2; }

int launch_f4(const moe_layer_desc *L, const uint16_t *x, int M, const float *w,
              const int32_t *ttp, const int32_t *act_count, uint16_t *out, void *ws,
              const moe_workspace_view &v, uint32_t *err, void *stream) {
  const moe_experts &R = L->routed;
  const moe_experts *Sx = L->shared;
  char *base = static_cast<char *>(ws);
  F4Args a = {};
  a.M = M;
  a.k = L->top_k;
  a.n = M * L->top_k;
  a.E = R.num_experts;
  a.H = R.hidden;
  a.I = R.inter;
  a.cap = v.cap;
  a.max_total = v.max_total;
  a.NT = M <= 16 ? 16 : 32;
  a.x = x;
  a.w = w;
  a.ttp = ttp;
  a.sti = reinterpret_cast<const int32_t *>(base + v.sorted_token_ids);
  a.act_count = act_count;
  a.items = reinterpret_cast<const int4 *>(base + v.tc_items);
  a.out = out;
  a.gg = R.gate.global_scale;
  a.gu = R.up.global_scale;
  a.down_fp8 = R.fmt == MOE_FMT_NVFP4_GATE_UP ? 1 : 0;
  a.gd = a.down_fp8 ? nullptr : R.down.global_scale;
  a.sdown = a.down_fp8 ? static_cast<const float *>(R.down.scale) : nullptr;
  a.xt = reinterpret_cast<uint8_t *>(base + v.tc_x_terms);
  a.xs = reinterpret_cast<float *>(base + v.tc_x_scale);
  a.hq = reinterpret_cast<uint16_t *>(base + v.tc_h_terms);
  a.hs = reinterpret_cast<float *>(base + v.tc_h_scale);
  a.h = reinterpret_cast<float *>(base + v.h);
  a.y = reinterpret_cast<float *>(base + v.y);
  if (Sx) {
    a.Is = Sx->inter;
    a.ssg = static_cast<const float *>(Sx->gate.scale);
    a.ssu = static_cast<const float *>(Sx->up.scale);
    a.ssd = static_cast<const float *>(Sx->down.scale);
    a.hq_sh = a.hq + (size_t)2 * v.max_total * a.I;
    a.hs_sh = a.hs + (size_t)v.max_total * (a.I / 128);
    a.h_sh = reinterpret_cast<float *>(base + v.h_shared);
    a.y_sh = reinterpret_cast<float *>(base + v.y_shared);
    a.gated = L->shared_gate ? 1 : 0;
  }
  a.gate_vals = reinterpret_cast<float *>(base + v.shared_gate);
  a.done = reinterpret_cast<int *>(base + v.tc_done);
  a.work = a.done + a.E + 1;
  a.grid_ctr = reinterpret_cast<unsigned long long *>(base + v.blend_counters);
  a.err = err;
  const size_t ring = ring_bytes_for(v.cap);
  if (!ring) return MOE_EUNSUPPORTED;
  a.ring_bytes = (uint32_t)ring;
  F4Maps maps;
  int st = f4_maps(&R, Sx, a.xt, a.hq, a.hq_sh, v.max_total, a.NT, &maps);
  if (st) return st;
  const size_t smem = ring + fixed_bytes(v.cap);
  st = ensure_smem_limit((const void *)nvfp4_ffn_kernel, smem);
  if (st) return st;
  return launch_pdl_coop(nvfp4_ffn_kernel, dim3(sm_count()), dim3(kThreads), smem, stream, a,
                         maps);
}

}  // namespace moe
