// align.cu -- deterministic device-side token alignment (moe_align).
//
// What it computes is the three-stage alignment of "nbxtensor/ops/moe_align.py"
// (stage 1: per-expert counts, block padding, exclusive offsets and the total;
// stage 2: sentinel fill and the block -> expert map; stage 3: rank = number of
// earlier slots routed to the same expert, scatter) together with the
// token_to_perm map and the ascending active-expert list of
// moe_fp8_grouped_sort ("metrale_model_layers/layers/ops/fp8_moe_grouped.rs").
//
// How: one CTA, no atomics on any table.  Each warp owns a contiguous chunk of
// slots.  Pass 1 counts its chunk into a private shared-memory histogram row:
// __match_any_sync groups the lanes holding the same expert and the lowest
// lane of each group adds the group's popcount, so no two lanes ever write the
// same counter.  A column scan over the warps turns the rows into per-warp
// exclusive bases and the per-expert totals; one block-wide scan gives the
// padded offsets and the active-list positions.  Pass 2 recomputes each slot's
// group and writes it to offsets[e] + base[warp][e] + (earlier equal lanes in
// its 32-slot step) + (earlier steps of the warp): exactly the count of
// earlier equal slots, so the order equals a stable sort and is bit-identical
// run to run.  The pages' pairwise O(n^2) rank is replaced by this O(n) form,
// which computes the same integers.
#include "common.cuh"
#include "xprep.cuh"

namespace moe {
namespace {

struct AlignArgs {
  const void *ids;
  int is64;
  int n, E, BS, max_total, max_blocks, cap;
  int32_t *sti, *sei, *off, *ttp, *act, *act_count, *ntpp;
  uint32_t *err;
  // optional (the layer's tensor-core kernels): per active-list index,
  // {run offset, expert, slot count, 0}
  int4 *items;
  // optional: the per-token x table, one extra CTA per token
  XPrep xp;
};

// Expert id of slot i, or -1 when it lies outside [0, E).
__device__ __forceinline__ int read_id(const AlignArgs &a, int i) {
  long long v;
  if (a.is64)
    v = __ldcg(reinterpret_cast<const long long *>(a.ids) + i);
  else
    v = __ldcg(reinterpret_cast<const int *>(a.ids) + i);
  return (v >= 0 && v < a.E) ? (int)v : -1;
}

constexpr int kUnroll = 8;            // ids in flight per lane in pass 1
constexpr int kCacheIdsMax = 32768;   // slots whose ids are kept in shared memory

template <int NT>
__global__ void __launch_bounds__(NT) align_kernel(AlignArgs a) {
  constexpr int NW = NT / 32;
  extern __shared__ int smem[];
  const int E = a.E;
  int *cnt = smem;                  // [NW][E] per-warp counts, then bases
  int *count = cnt + NW * E;        // [E]
  int *offs = count + E;            // [E+1]
  int *apos = offs + E + 1;         // [E]
  int *scan = apos + E;             // [2 * 32] block-scan scratch
  short *idc = reinterpret_cast<short *>(scan + 64);  // [n] cached ids (n <= kCacheIdsMax)
  const bool cache_ids = a.n <= kCacheIdsMax;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  pdl_wait();      // topk_ids (and x) may come from the previous kernel on the stream
  pdl_trigger();
  if (blockIdx.x > 0) {   // the extra CTAs: token blockIdx.x - 1 of the x table
    __shared__ int red[8];
    xprep_token(a.xp, (int)blockIdx.x - 1, red);
    return;
  }

  for (int i = tid; i < NW * E; i += NT) cnt[i] = 0;
  __syncthreads();

  // ---- pass 1: per-warp histograms of contiguous chunks --------------------
  const int chunk = (((a.n + NW - 1) / NW) + 31) & ~31;
  const int beg = min(a.n, w * chunk);
  const int end = min(a.n, beg + chunk);
  int *mine = cnt + w * E;
  bool bad = false;
  for (int base = beg; base < end; base += 32 * kUnroll) {
    int ev[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      int i = base + 32 * j + lane;
      ev[j] = -2;                                   // past the chunk
      if (i < end) {
        ev[j] = read_id(a, i);
        if (ev[j] < 0) bad = true;
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      int i = base + 32 * j + lane;
      if (cache_ids && i < end) idc[i] = (short)ev[j];
      unsigned m = __match_any_sync(0xffffffffu, ev[j]);
      if (ev[j] >= 0 && lane == __ffs(m) - 1) mine[ev[j]] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();

  // ---- column scan over warps: per-warp exclusive bases, per-expert counts --
  for (int e = tid; e < E; e += NT) {
    int run = 0;
#pragma unroll 4
    for (int ww = 0; ww < NW; ++ww) {
      int c = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += c;
    }
    count[e] = run;
  }
  __syncthreads();

  // ---- block-wide exclusive scan of padded counts and active flags ----------
  const int ept = (E + NT - 1) / NT;   // consecutive experts per thread
  const int e0 = tid * ept;
  int ps = 0, as = 0;
  for (int j = 0; j < ept; ++j) {
    int e = e0 + j;
    if (e < E) {
      int c = count[e];
      ps += (c + a.BS - 1) / a.BS * a.BS;
      as += c > 0;
    }
  }
  int pin = ps, ain = as;              // inclusive warp scan
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int pv = __shfl_up_sync(0xffffffffu, pin, d);
    int av = __shfl_up_sync(0xffffffffu, ain, d);
    if (lane >= d) {
      pin += pv;
      ain += av;
    }
  }
  if (lane == 31) {
    scan[w] = pin;
    scan[32 + w] = ain;
  }
  __syncthreads();
  if (w == 0) {
    int pv = lane < NW ? scan[lane] : 0;
    int av = lane < NW ? scan[32 + lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int p2 = __shfl_up_sync(0xffffffffu, pv, d);
      int a2 = __shfl_up_sync(0xffffffffu, av, d);
      if (lane >= d) {
        pv += p2;
        av += a2;
      }
    }
    if (lane < NW) {               // inclusive -> exclusive warp offsets
      scan[lane] = pv;
      scan[32 + lane] = av;
    }
  }
  __syncthreads();
  int pex = (w > 0 ? scan[w - 1] : 0) + pin - ps;
  int aex = (w > 0 ? scan[32 + w - 1] : 0) + ain - as;
  const int total = scan[NW - 1];
  const int nact = scan[32 + NW - 1];
  for (int j = 0; j < ept; ++j) {
    int e = e0 + j;
    if (e < E) {
      int c = count[e];
      offs[e] = pex;
      apos[e] = aex;
      pex += (c + a.BS - 1) / a.BS * a.BS;
      aex += c > 0;
    }
  }
  if (tid == 0) offs[E] = total;
  __syncthreads();

  // ---- stage-2 outputs: offsets, active list, block map, sentinels ---------
  for (int e = tid; e <= E; e += NT) a.off[e] = offs[e];
  for (int e = tid; e < E; e += NT)
    if (count[e] > 0) {
      a.act[apos[e]] = e;
      if (a.items) a.items[apos[e]] = make_int4(offs[e], e, count[e], 0);
    }
  for (int x = nact + tid; x < a.cap; x += NT) a.act[x] = -1;
  if (tid == 0) {
    *a.act_count = nact;
    *a.ntpp = total;
  }
  for (int b = tid; b < a.max_blocks; b += NT) {
    const int start = b * a.BS;
    int owner = -1;
    if (start < total) {             // last expert whose offset <= start
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= start) lo = mid; else hi = mid - 1;
      }
      owner = lo;
    }
    a.sei[b] = owner;
  }
  for (int e = tid; e < E; e += NT)     // padding inside each run
    for (int p = offs[e] + count[e]; p < offs[e + 1]; ++p) a.sti[p] = a.n;
  for (int p = total + tid; p < a.max_total; p += NT) a.sti[p] = a.n;   // tail

  // ---- pass 2: scatter each slot to offsets[e] + rank ----------------------
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    int e = -2;
    if (i < end) e = cache_ids ? (int)idc[i] : read_id(a, i);
    unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = offs[e] + mine[e] + __popc(m & lanemask_lt());
      a.sti[pos] = i;
      a.ttp[i] = pos;
    } else if (i < end) {
      a.ttp[i] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(m) - 1) mine[e] += __popc(m);
    __syncwarp();
  }

  if (__syncthreads_or(bad) && tid == 0 && a.err) atomicOr(a.err, MOE_ERR_BAD_ID);
}

template <int NT>
size_t align_smem_bytes(int n, int E) {
  size_t ints = (size_t)(NT / 32) * E + E + (E + 1) + E + 64;
  size_t bytes = ints * 4;
  if (n <= kCacheIdsMax) bytes += (size_t)n * 2;
  return (bytes + 15) & ~(size_t)15;
}

template <int NT>
int launch_align(const AlignArgs &a, void *stream) {
  const size_t smem = align_smem_bytes<NT>(a.n, a.E);
  const int st = ensure_smem_limit(reinterpret_cast<const void *>(align_kernel<NT>),
                                   align_smem_bytes<NT>(kCacheIdsMax, MOE_MAX_EXPERTS));
  if (st) return st;
  const int grid = 1 + (a.xp.mode != kXPrepNone ? a.xp.M : 0);
  return launch_pdl(align_kernel<NT>, dim3(grid), dim3(NT), smem, stream, a);
}

__global__ void __launch_bounds__(kXPrepThreads) xprep_kernel(XPrep p) {
  __shared__ int red[8];
  pdl_wait();   // x may come from the previous kernel on the stream
  pdl_trigger();
  xprep_token(p, (int)blockIdx.x, red);
}

}  // namespace
}  // namespace moe

extern "C" int moe_align_sizes(int n, int num_experts, int block_size, int *max_total,
                               int *max_blocks, int *cap) {
  if (!max_total || !max_blocks || !cap || n < 0 || num_experts < 1 || block_size < 1)
    return MOE_EINVAL;
  if (n > MOE_MAX_SLOTS) return MOE_EUNSUPPORTED;
  const int64_t a = (int64_t)n * block_size;
  const int64_t b = (int64_t)n + (int64_t)num_experts * (block_size - 1);
  const int64_t m = a < b ? a : b;
  const int64_t mt = moe::ceil_div64(m, block_size) * block_size;
  if (mt > INT32_MAX) return MOE_EUNSUPPORTED;
  *max_total = (int)mt;
  *max_blocks = (int)(mt / block_size);
  *cap = n < num_experts ? n : num_experts;
  return MOE_OK;
}

namespace moe {

// moe_align, plus (when items is not NULL) the active table of the layer's
// tensor-core kernels: items[a] = {expert_offsets[e], e, count[e], 0} for the
// a-th active expert e; and (when xp is not NULL and names a format) the
// per-token x table of those kernels, by M extra CTAs of the same launch.
int align_launch(const void *topk_ids, int ids_is_int64, int n, int num_experts, int block_size,
                 int32_t *sorted_token_ids, int32_t *sorted_expert_ids, int32_t *expert_offsets,
                 int32_t *token_to_perm, int32_t *active_experts, int32_t *active_count,
                 int32_t *num_tokens_post_padded, uint32_t *err_word, int4 *items,
                 const XPrep *xp, void *stream) {
  int max_total, max_blocks, cap;
  int st = moe_align_sizes(n, num_experts, block_size, &max_total, &max_blocks, &cap);
  if (st != MOE_OK) return st;
  if (num_experts > MOE_MAX_EXPERTS) return MOE_EUNSUPPORTED;
  if (!expert_offsets || !active_count || !num_tokens_post_padded) return MOE_EINVAL;
  if (n > 0 && (!topk_ids || !sorted_token_ids || !sorted_expert_ids || !token_to_perm ||
                !active_experts))
    return MOE_EINVAL;
  AlignArgs a;
  a.ids = topk_ids;
  a.is64 = ids_is_int64 ? 1 : 0;
  a.n = n;
  a.E = num_experts;
  a.BS = block_size;
  a.max_total = max_total;
  a.max_blocks = max_blocks;
  a.cap = cap;
  a.sti = sorted_token_ids;
  a.sei = sorted_expert_ids;
  a.off = expert_offsets;
  a.ttp = token_to_perm;
  a.act = active_experts;
  a.act_count = active_count;
  a.ntpp = num_tokens_post_padded;
  a.err = err_word;
  a.items = items;
  a.xp = xp ? *xp : XPrep{};
  if (a.xp.mode != kXPrepNone && (a.xp.M < 1 || a.xp.M > 32 || !a.xp.x || !a.xp.table ||
                                  !a.xp.scale || a.xp.H % 128))
    return MOE_EINVAL;
  // One CTA (plus the x-table CTAs); its width grows with n (a launch tuple
  // fixed per shape class).
  if (n <= 512) return launch_align<128>(a, stream);
  if (n <= 4096) return launch_align<256>(a, stream);
  if (n <= 16384) return launch_align<512>(a, stream);
  return launch_align<1024>(a, stream);
}

}  // namespace moe

extern "C" int moe_align(const void *topk_ids, int ids_is_int64, int n, int num_experts,
                         int block_size, int32_t *sorted_token_ids, int32_t *sorted_expert_ids,
                         int32_t *expert_offsets, int32_t *token_to_perm,
                         int32_t *active_experts, int32_t *active_count,
                         int32_t *num_tokens_post_padded, uint32_t *err_word, void *stream) {
  return moe::align_launch(topk_ids, ids_is_int64, n, num_experts, block_size, sorted_token_ids,
                           sorted_expert_ids, expert_offsets, token_to_perm, active_experts,
                           active_count, num_tokens_post_padded, err_word, nullptr, nullptr,
                           stream);
}

namespace moe {

// The per-token x table alone (moe_decode_experts on a new x): M CTAs.
int xprep_launch(const XPrep &p, void *stream) {
  if (p.mode == kXPrepNone) return MOE_OK;
  if (p.M < 1 || p.M > 32 || !p.x || !p.table || !p.scale || p.H % 128) return MOE_EINVAL;
  return launch_pdl(xprep_kernel, dim3(p.M), dim3(kXPrepThreads), 0, stream, p);
}

}  // namespace moe
