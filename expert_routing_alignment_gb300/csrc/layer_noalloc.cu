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
#include <mutex>

#include "common.cuh"

namespace {

// The workspace of moe_decode_layer_noalloc (zero at module load).
static __device__ __align__(256) unsigned char g_layer_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch[kMaxDevices];   // device address of g_layer_scratch, per device

// The array's device address on the current device, looked up once per device
// (the first call on a device does this, so it should come before any stream
// capture that contains the call).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    moe::set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layer_scratch);
    if (e != cudaSuccess || !p) {
      moe::set_last_cuda_error(e);
      return MOE_ECUDA;
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_layer_noalloc(const moe_layer_desc *layer, const uint16_t *x, int M,
                                        const float *router_logits, const int32_t *topk_ids,
                                        const float *topk_w, uint16_t *out, uint32_t *err_word,
                                        void *stream) {
  moe_workspace_view v;
  int st = moe_decode_layer_workspace_view(layer, M, &v);
  if (st) return st;
  if (v.total_bytes > MOE_NOALLOC_SCRATCH_BYTES) return MOE_EUNSUPPORTED;   // too large for it
  void *ws = nullptr;
  st = scratch_address(&ws);
  if (st) return st;
  // The layer's grid-barrier count and the tensor-core path's item counters
  // must start the call consistent: clear them (the rest of the workspace is
  // fully written before it is read).
  cudaError_t e = cudaMemsetAsync(static_cast<char *>(ws) + v.blend_counters, 0, 8,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess && v.tc_done)
    e = cudaMemsetAsync(static_cast<char *>(ws) + v.tc_done, 0, ((size_t)v.cap + 1) * 4,
                        (cudaStream_t)stream);
  if (e != cudaSuccess) {
    moe::set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  return moe_decode_layer(layer, x, M, router_logits, topk_ids, topk_w, out, ws,
                          MOE_NOALLOC_SCRATCH_BYTES, err_word, stream);
}
