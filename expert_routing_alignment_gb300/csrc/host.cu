// host.cu -- library information, error bookkeeping and device attributes.
#include <mutex>
#include <unordered_map>

#include "common.cuh"

namespace moe {

static thread_local int g_last_cuda_error = 0;

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

int check_launch() {
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    (void)cudaGetLastError();
    return MOE_ECUDA;
  }
  return MOE_OK;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int ensure_smem_limit(const void *func, size_t bytes) {
  if (bytes <= 48 * 1024) return MOE_OK;
  static std::mutex mu;
  static std::unordered_map<uint64_t, size_t> done;   // (func, device) -> bytes set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
  const uint64_t key = (uint64_t)(uintptr_t)func * 64u + (uint64_t)(dev & 63);
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return MOE_OK;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  done[key] = bytes;
  return MOE_OK;
}

int ensure_max_carveout(const void *func) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, bool> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
  const uint64_t key = (uint64_t)(uintptr_t)func * 64u + (uint64_t)(dev & 63);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return MOE_OK;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ECUDA;
  }
  done[key] = true;
  return MOE_OK;
}

}  // namespace moe

extern "C" const char *moe_version(void) { return "moe_gb300 0.1 sm_103a"; }

extern "C" const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_EUNSUPPORTED: return "shape or option not supported";
    case MOE_ECUDA: return "CUDA error";
    default: return "unknown status";
  }
}

extern "C" int moe_last_cuda_error(void) { return moe::g_last_cuda_error; }
