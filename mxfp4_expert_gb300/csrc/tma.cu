// Host-side tensor-map encoder (see tma.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "host_util.h"
#include "tma.cuh"

namespace moe {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
    (void)cudaGetLastError();
  });
  return fn;
}

}  // namespace

bool tma_available() { return encode_fn() != nullptr; }

int tma_encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  const EncodeTiled fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  if (rank < 1 || rank > 5) return MOE_ERR_INVALID_ARG;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = cuuint64_t(dims[i]);
    b[i] = cuuint32_t(box[i]);
    e[i] = 1;
    if (i + 1 < rank) s[i] = cuuint64_t(strides[i]);
  }
  const CUresult r = fn(map, type, cuuint32_t(rank), const_cast<void*>(base), d, s, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace moe
