// Tensor memory accelerator (TMA): tiled copies global -> shared memory
// described by tensor maps (inline PTX), and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// 2-D tiled load of the box at (x = innermost element, y) into shared memory
// at dst, completion counted in bytes on `bar`. x times the element size is
// a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
// 4-D tiled load of the box at (x, y, z, w); as above.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Host: a tiled tensor map (cuTensorMapEncodeTiled, looked up once through
// the runtime, so the library has no link-time dependence on the driver
// library). dims[0] is the innermost (contiguous) dimension; strides are the
// byte strides of dims 1 .. rank-1; box the box extent per dimension; element
// strides 1, no interleave, 256-byte L2 promotion, zero fill outside the
// tensor. Returns MOE_OK, MOE_ERR_CUDA (no encoder) or
// MOE_ERR_UNSUPPORTED_SHAPE (rejected by the encoder).
int tma_encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle);
bool tma_available();

}  // namespace moe
