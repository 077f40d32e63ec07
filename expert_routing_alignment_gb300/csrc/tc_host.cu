// tc_host.cu -- host side shared by the tensor-core expert kernels: the
// tensor-map encoder, taken from the driver through the runtime (no -lcuda).
#include <mutex>

#include "tc_common.cuh"

namespace moe {
namespace tc {

namespace {
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
}  // namespace

namespace {
int encode_u8(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
              const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return MOE_ECUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_EUNSUPPORTED;
}
}  // namespace

int encode_u8_sw128(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box) {
  return encode_u8(m, ptr, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

int encode_u8_plain(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box) {
  return encode_u8(m, ptr, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace tc
}  // namespace moe
