// tc_common.cuh -- pieces shared by the tensor-core expert kernels of the
// decode MoE layer (sm_103a): bounded mbarrier and counter waits, the E4M3
// term split of activations, tcgen05 MMA / TMEM access, 3-D tensor copies,
// the ring placement rule, and the host-side tensor-map encoding.
#pragma once

#include <cudaTypedefs.h>

#include "async.cuh"
#include "common.cuh"

namespace moe {
namespace tc {

constexpr uint64_t kWaitNs = 2000000000ull;   // a wait gives up after ~2 s
constexpr int kTileBytes = 128 * 128;          // one 128-row x 128-byte weight box

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One potentially blocking test of an mbarrier phase: the hardware may park
// the thread until the phase completes or a short time limit passes, so
// waiting warps leave the issue slots to the MMA and copy threads.
__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` of an mbarrier; false when *failed is set
// meanwhile (another role of the CTA gave up) or after about two seconds.
__device__ __forceinline__ bool wait_phase(const volatile int *failed, uint64_t *bar,
                                           uint32_t parity) {
  if (mbar_poll(bar, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 1; i < (1u << 28); ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 15) == 0 && (*failed || gtime() - t0 > kWaitNs)) return false;
  }
  return false;
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n)
               : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until *p >= target (written by other CTAs with release); bounded, and
// false as soon as *failed is set.
__device__ __forceinline__ bool wait_at_least(const volatile int *failed, const int *p,
                                              int target) {
  const uint64_t t0 = gtime();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (ld_acquire(p) >= target) return true;
    if (*failed || gtime() - t0 > kWaitNs) return false;
    __nanosleep(64);
  }
  return false;
}

// Add v to *p at gpu scope with release semantics, without waiting for the
// result (every write ordered before it -- this thread's, and those of the
// threads it synchronised with at a CTA barrier -- is visible to a thread
// that acquires the new value).
__device__ __forceinline__ void red_release_add(int *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// The same with acquire-release semantics, returning the previous value.
__device__ __forceinline__ int atom_acq_rel_add(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// sum_j w[t][j] * y[token_to_perm[t*k + j]][c .. c+3] in fp32, j ascending,
// slots with a negative position skipped: the blend's weighted sum.  The
// loads of 8 slots go out together (one round trip for the positions and
// weights, one for the rows) before the sums, which keep the slot order.
__device__ __forceinline__ float4 blend_slots(const float *y, const float *w, const int32_t *ttp,
                                              int t, int k, int H, int c) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {
    int p[8];
    float wv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = j0 + jj;
      p[jj] = j < k ? __ldcg(ttp + (size_t)t * k + j) : -1;
      wv[jj] = j < k ? __ldcg(w + (size_t)t * k + j) : 0.f;
    }
    float4 v[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      v[jj] = p[jj] >= 0 ? __ldcg(reinterpret_cast<const float4 *>(y + (size_t)p[jj] * H + c))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (p[jj] < 0) continue;
      acc.x = fmaf(wv[jj], v[jj].x, acc.x);
      acc.y = fmaf(wv[jj], v[jj].y, acc.y);
      acc.z = fmaf(wv[jj], v[jj].z, acc.z);
      acc.w = fmaf(wv[jj], v[jj].w, acc.w);
    }
  }
  return acc;
}

// A tensor map's descriptor fetched ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const void *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy writes to global memory made visible to later tensor copies
// (async proxy) of any CTA.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Generic-proxy writes to this CTA's shared memory made visible to the
// tensor cores' operand reads (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// f16 conversions (round to nearest even) and back (exact).
__device__ __forceinline__ uint16_t f16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Power-of-two exponent s such that amax * 2^s lies in [128, 256) (0 for a
// zero maximum), kept where 2^s and 2^-s are normal floats.
__device__ __forceinline__ int term_shift(uint32_t amax_bits) {
  if (amax_bits == 0) return 0;
  const int e = (int)(amax_bits >> 23) - 127;
  const int s = 7 - e;
  return s < -126 ? -126 : (s > 126 ? 126 : s);
}

// Two floats -> two E4M3 bytes (first in the low byte), nearest-even,
// saturating at 448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two values already scaled into E4M3 range -> their two E4M3 terms t0, t1
// (t0 + t1 = the value exactly for a bf16 input, see the split rule in the
// kernels): two bytes each, first element in the low byte.
__device__ __forceinline__ void e4m3_split2(float v0, float v1, uint32_t &t0, uint32_t &t1) {
  t0 = e4m3x2(v0, v1);
  const float2 back = f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)t0));
  t1 = e4m3x2(v0 - back.x, v1 - back.y);
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major operand tile written with the
// 128-byte swizzle (rows of 128 bytes, groups of 8 rows 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: E4M3 x E4M3 -> f32, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_e4m3(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 64 consecutive 32-bit columns of this warp's 32 TMEM lanes, from registers.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,"
      "%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,"
      "%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]),
      "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]),
      "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]),
      "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]),
      "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor: f16 x f16 -> f32, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D (+)= A x B with A (128 rows, 16 f16 of k per row) in TMEM at column
// a_col and B from shared memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t d, uint32_t a_col, uint64_t bd, uint32_t id,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_col), "l"(bd), "r"(id), "r"(acc));
}

// 8 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tensor copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_3d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                            int z, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_2d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                       uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Placement of the next range of `len` units in a ring of `cap` units: at
// the head, or at 0 when it does not fit before the end.  Ranges depend only
// on the sequence of lengths, so every role computes the same positions.
__device__ __forceinline__ uint32_t ring_place(uint32_t &head, uint32_t len, uint32_t cap) {
  const uint32_t pos = head + len <= cap ? head : 0u;
  head = pos + len;
  return pos;
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------

// A tiled u8 tensor map with the 128-byte swizzle (the operand layout of the
// MMAs); MOE_OK, or MOE_ECUDA / MOE_EUNSUPPORTED when encoding fails.
int encode_u8_sw128(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box);
// The same without swizzle (tiles read by threads, not by the tensor cores).
int encode_u8_plain(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box);

}  // namespace tc
}  // namespace moe
