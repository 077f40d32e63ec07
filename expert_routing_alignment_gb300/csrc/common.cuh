// common.cuh -- device helpers and launch plumbing shared by the CUDA sources
// of the decode MoE layer (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace moe {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Records a failing cudaError_t for moe_last_cuda_error() (thread-local).
void set_last_cuda_error(cudaError_t e);

// Checks the launch that was just enqueued; MOE_OK or MOE_ECUDA.
int check_launch();

// Raises a kernel's dynamic shared-memory limit to `bytes` (once per kernel
// and device; never again afterwards, so launches inside a stream capture
// make no attribute calls).
int ensure_smem_limit(const void *func, size_t bytes);

// Prefers the largest shared-memory carveout for a kernel (once per kernel
// and device), so that kernels meant to share an SM fit together.
int ensure_max_carveout(const void *func);

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Launch with programmatic dependent launch enabled: the kernel may be
// scheduled while its predecessor on the stream is finishing.  Every kernel
// of this library calls pdl_wait() before it reads anything a predecessor
// wrote or writes anything at all, so this only hides launch latency.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
               void *stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ((KArgs)args)...);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  return MOE_OK;
}

// launch_pdl for a grid whose CTAs wait on one another: also cooperative, so
// the launch fails unless every CTA can be resident at once.
template <typename... KArgs, typename... Args>
int launch_pdl_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                    void *stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, ((KArgs)args)...);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  return MOE_OK;
}

inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The format of one projection of an expert set (0 gate, 1 up, 2 down): the
// set's format, except under the nvfp4-gate-up tier (NVFP4 gate and up, FP8
// down).
inline int proj_fmt(int set_fmt, int proj) {
  if (set_fmt == MOE_FMT_NVFP4_GATE_UP) return proj == 2 ? MOE_FMT_FP8_B128 : MOE_FMT_NVFP4_G16;
  return set_fmt;
}

// ---------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------

// Programmatic dependent launch: wait until the predecessor grid on the
// stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the successor grid on the stream to be scheduled.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// bf16 bit pattern -> float (exact).
__device__ __forceinline__ float bf16_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// float -> bf16 bit pattern, round to nearest even (hardware cvt).
__device__ __forceinline__ uint16_t float_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Two E4M3 bytes (low byte = first element) -> two f16 in one register
// (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

// One byte holding two E2M1 codes (low nibble = first element) -> two f16.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t.reg .b16 s;\n\t"
      "cvt.u16.u32 s, %1;\n\t"
      "cvt.u8.u16 t, s;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte_in_low_bits));
  return r;
}

// The two halves of an f16x2 register as floats (exact).
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h2) {
  float2 f;
  asm("{\n\t.reg .f16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\t"
      "cvt.f32.f16 %1, hi;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(h2));
  return f;
}

// One E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  return f16x2_to_float2(e4m3x2_to_f16x2((uint16_t)(byte & 0xFFu))).x;
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Loads that bypass L1 for data written by an earlier kernel of the stream.
__device__ __forceinline__ int ld_cg(const int32_t *p) { return __ldcg(p); }

// 16-byte streaming load of read-only weights (not kept in L1).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace moe
