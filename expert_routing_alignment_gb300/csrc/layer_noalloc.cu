// layer_noalloc.cu -- moe_decode_layer for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// code that runs inside another framework's captured CUDA graph or stream
// callback, plugins whose host forbids device allocation after start-up, and
// embedded runtimes with a fixed device-memory budget decided at load time.
// moe_decode_layer_noalloc serves them: it runs the same layer with its
// workspace taken from a file-scope device array of fixed size instead of a
// caller buffer, and allocates nothing.
//
// The array costs MOE_NOALLOC_SCRATCH_BYTES of device memory on every GPU that
// loads the library, for as long as the library stays loaded.  Every call on a
// device uses the same array, so calls that overlap on the GPU (on different
// streams, or from different host threads without ordering) race on it: order
// them on one stream.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
int check_layer_call(const moe_layer_desc *layer, const uint16_t *x, int M,
                     const float *router_logits, const int32_t *topk_ids, const float *topk_w,
                     const uint16_t *out, moe_workspace_view *v);
size_t tc_counter_bytes(const moe_layer_desc *L);
}

namespace {

// The workspace of moe_decode_layer_noalloc (zero at module load).
static __device__ __align__(256) unsigned char g_layer_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Slot {
  unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
  void *addr;                  // device address of g_layer_scratch in it
};
Slot g_scratch[kMaxDevices];

// The unique id of the calling thread's current context (0 if it cannot be
// read): a context created after cudaDeviceReset gets a new id, and the
// module, with the array, may then sit at a new address.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
      get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// The array's device address on the current device.  It is looked up with
// cudaGetSymbolAddress the first time a device (more precisely, a context of
// it) calls, and cached: that first call should come before any stream
// capture that contains the entry point.  A call from a new context of the
// device (after cudaDeviceReset) looks the address up again.
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    moe::set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  // 0 when no context is current yet: the lookup below then makes the
  // device's primary context current
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  Slot &slot = g_scratch[dev];
  if (!slot.addr || ctx == 0 || slot.ctx_id != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layer_scratch);
    if (e != cudaSuccess || !p) {
      moe::set_last_cuda_error(e);
      return MOE_ECUDA;
    }
    slot.addr = p;
    slot.ctx_id = ctx;
  }
  *out = slot.addr;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_layer_noalloc(const moe_layer_desc *layer, const uint16_t *x, int M,
                                        const float *router_logits, const int32_t *topk_ids,
                                        const float *topk_w, uint16_t *out, uint32_t *err_word,
                                        void *stream) {
  // every host check first: a rejected call enqueues nothing
  moe_workspace_view v;
  int st = moe::check_layer_call(layer, x, M, router_logits, topk_ids, topk_w, out, &v);
  if (st) return st;
  if (v.total_bytes > MOE_NOALLOC_SCRATCH_BYTES) return MOE_EUNSUPPORTED;   // too large for it
  void *ws = nullptr;
  st = scratch_address(&ws);
  if (st) return st;
  // The layer's grid-barrier count and the tensor-core path's counters must
  // start the call consistent: clear them (the rest of the workspace is fully
  // written before it is read).
  cudaError_t e = cudaMemsetAsync(static_cast<char *>(ws) + v.blend_counters, 0, 8,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess && v.tc_done)
    e = cudaMemsetAsync(static_cast<char *>(ws) + v.tc_done, 0, moe::tc_counter_bytes(layer),
                        (cudaStream_t)stream);
  if (e != cudaSuccess) {
    moe::set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  return moe_decode_layer(layer, x, M, router_logits, topk_ids, topk_w, out, ws,
                          MOE_NOALLOC_SCRATCH_BYTES, err_word, stream);
}
