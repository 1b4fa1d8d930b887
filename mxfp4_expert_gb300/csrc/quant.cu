// Activation rows -> E4M3 elements with one E8M0 scale per 32 (the B operand
// of the block-scaled tcgen05 expert GEMMs).
//
// Two forms, both "value = sum of the terms x 2^(s - 127)" per 32-element block:
//   kQuantMxfp8 (1 term): MXFP8 as defined by OCP MX v1.0 (§5.3, §6.3):
//     s = floor(log2 amax) - 8 + 127 clamped to [0, 254] (amax = 0: s = 0),
//     element = RNE(v * 2^(127 - s)) to E4M3, saturating at +-448. This is
//     the 8-bit activation format of the W4A8 configuration (page "3 ways to
//     speed up MoE inference on NVIDIA DGX Spark", §2).
//   kQuantSplit2 (2 terms): s = floor(log2 amax) - 7 + 127, t0 = E4M3(v 2^(127-s)),
//     t1 = E4M3(v 2^(127-s) - t0): about 8 significant bits per element,
//     the precision of bf16, for the bf16-activation layer.
// One thread per (row, 32-block); the 32 values are read as 8 x 16 bytes (bf16)
// or 8 x 32 bytes (fp32).
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "mma_tile.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return uint32_t(f32x2_to_e4m3x2(a, b)) | (uint32_t(f32x2_to_e4m3x2(c, d)) << 16);
}

template <bool kBf16>
__global__ void __launch_bounds__(256) act_quant_kernel(const void* src, int rows, int K, int mode, uint8_t* q,
                                                        uint8_t* scales) {
  const int KB = K / kMxBlock;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)rows * KB) return;
  const int r = int(i / KB), kb = int(i - (long long)r * KB);
  float v[kMxBlock];
  if (kBf16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + (size_t)r * K + kb * kMxBlock);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = p[j];
      v[8 * j + 0] = bf16_lo(w.x);
      v[8 * j + 1] = bf16_hi(w.x);
      v[8 * j + 2] = bf16_lo(w.y);
      v[8 * j + 3] = bf16_hi(w.y);
      v[8 * j + 4] = bf16_lo(w.z);
      v[8 * j + 5] = bf16_hi(w.z);
      v[8 * j + 6] = bf16_lo(w.w);
      v[8 * j + 7] = bf16_hi(w.w);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + (size_t)r * K + kb * kMxBlock);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 w = p[j];
      v[4 * j + 0] = w.x;
      v[4 * j + 1] = w.y;
      v[4 * j + 2] = w.z;
      v[4 * j + 3] = w.w;
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < kMxBlock; ++j) amax = fmaxf(amax, fabsf(v[j]));
  // E8M0 byte s; elements are v * 2^(127 - s)
  int s = 0;
  if (amax > 0.0f) {
    s = floor_log2(amax) - (mode == kQuantMxfp8 ? 8 : 7) + 127;
    s = s < 0 ? 0 : (s > 254 ? 254 : s);
  }
  const int nterms = mode == kQuantMxfp8 ? 1 : 2;
  uint8_t* q0 = q + ((size_t)r * nterms) * K + kb * kMxBlock;
  uint32_t t0[8], t1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) a[m] = scale2(v[4 * j + m], 127 - s);
    t0[j] = e4m3x4(a[0], a[1], a[2], a[3]);
    if (mode != kQuantMxfp8) {
      float b[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) b[m] = a[m] - e4m3_to_f32_hw((t0[j] >> (8 * m)) & 0xFFu);
      t1[j] = e4m3x4(b[0], b[1], b[2], b[3]);
    }
  }
  uint4* o0 = reinterpret_cast<uint4*>(q0);
  o0[0] = make_uint4(t0[0], t0[1], t0[2], t0[3]);
  o0[1] = make_uint4(t0[4], t0[5], t0[6], t0[7]);
  if (mode != kQuantMxfp8) {
    uint4* o1 = reinterpret_cast<uint4*>(q0 + K);
    o1[0] = make_uint4(t1[0], t1[1], t1[2], t1[3]);
    o1[1] = make_uint4(t1[4], t1[5], t1[6], t1[7]);
  }
  scales[(size_t)r * KB + kb] = uint8_t(s);
}

}  // namespace

int launch_act_quant(const void* src, bool src_bf16, int rows, int K, int mode, uint8_t* q, uint8_t* scales,
                     cudaStream_t s) {
  if (rows <= 0) return MOE_OK;
  if (K % kMxBlock) return MOE_ERR_UNSUPPORTED_SHAPE;
  const long long n = (long long)rows * (K / kMxBlock);
  const int threads = 256;
  const unsigned blocks = unsigned((n + threads - 1) / threads);
  if (src_bf16)
    act_quant_kernel<true><<<blocks, threads, 0, s>>>(src, rows, K, mode, q, scales);
  else
    act_quant_kernel<false><<<blocks, threads, 0, s>>>(src, rows, K, mode, q, scales);
  return launch_status();
}

}  // namespace moe
