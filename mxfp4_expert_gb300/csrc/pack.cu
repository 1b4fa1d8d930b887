// MXFP4 packing: fp32 weights -> E2M1 codes + E8M0 scales in the TILE16
// layout (include/moe_mxfp4.h), and the inverse permutation to the canonical
// layout for tests.
//
// Quantisation rule: OCP Microscaling Formats (MX) v1.0, §6.3 — per block of
// 32 along K, X = 2^(floor(log2 amax) - 2); elements v/X rounded to the
// nearest E2M1 value, ties to even mantissa, saturating at 6.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

// Source row of packed row r (0..15) of tile `tile`.
__device__ __forceinline__ int source_row(int layout, int tile, int r, int N) {
  if (layout == MOE_LAYOUT_TILE16_GATEUP) {
    const int I = N / 2;
    return r < 8 ? tile * 8 + r : I + tile * 8 + (r - 8);
  }
  return tile * kTileRows + r;
}

// Nearest E2M1 magnitude code for |q| < 8, ties to even (codes 0, 2, 4, 6
// have mantissa bit 0): the decision points are the midpoints of the grid.
__device__ __forceinline__ uint32_t e2m1_magnitude(float a) {
  return uint32_t(a > 0.25f) + uint32_t(a >= 0.75f) + uint32_t(a > 1.25f) + uint32_t(a >= 1.75f) +
         uint32_t(a > 2.5f) + uint32_t(a >= 3.5f) + uint32_t(a > 5.0f);
}

constexpr int kPackWarps = 8;

__global__ void __launch_bounds__(kPackWarps * 32)
pack_kernel(const float* __restrict__ w, uint8_t* __restrict__ packed, int n_mat, int N, int K,
            int layout, int* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KB = K / kMxBlock, NT = N / kTileRows;
  const long long units = (long long)n_mat * NT * KB;
  // lane = 2 r + hh: row r of the unit, elements 16 hh .. 16 hh + 15 of its K-block
  const int r = lane >> 1, hh = lane & 1;
  for (long long u = (long long)blockIdx.x * kPackWarps + warp; u < units;
       u += (long long)gridDim.x * kPackWarps) {
    const int kb = int(u % KB);
    const long long mt = u / KB;
    const int tile = int(mt % NT);
    const int mat = int(mt / NT);
    const int srow = source_row(layout, tile, r, N);
    const float4* src = reinterpret_cast<const float4*>(
        w + ((long long)mat * N + srow) * K + (long long)kb * kMxBlock + hh * 16);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 t = __ldg(src + i);
      v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float amax = 0.0f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const bool fin = isfinite(v[i]);
      bad |= !fin;
      amax = fin ? fmaxf(amax, fabsf(v[i])) : amax;
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    bad = __shfl_xor_sync(0xffffffffu, int(bad), 1) | int(bad);
    // s = floor(log2 amax) - 2 + 127, clamped to [0, 254]; subnormal amax -> 0.
    const uint32_t ebits = __float_as_uint(amax) >> 23;
    int s = amax == 0.0f ? 0 : max(int(ebits) - 2, 0);
    const float inv_x = exp2i(127 - s);   // exact power of two
    uint32_t wd[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const bool fin = isfinite(v[i]);
      const float q = fin ? v[i] * inv_x : 0.0f;
      uint32_t c = e2m1_magnitude(fabsf(q));
      c |= (fin && signbit(v[i])) ? 8u : 0u;
      wd[i >> 3] |= c << (4 * (i & 7));   // element 2j in the low nibble of byte j
    }
    if (bad && hh == 0 && status) atomicOr(status, MOE_DEV_NONFINITE_INPUT);
    if (!bad && s > 248 && hh == 0 && status) atomicOr(status, MOE_DEV_SCALE_RANGE);
    uint8_t* unit = packed + ((long long)mat * NT * KB + (long long)tile * KB + kb) * kUnitBytes;
    *reinterpret_cast<uint2*>(unit + r * 16 + hh * 8) = make_uint2(wd[0], wd[1]);
    if (hh == 0) {
      const int pos = r < 8 ? 2 * r : 2 * (r - 8) + 1;
      unit[kUnitCodeBytes + pos] = bad ? uint8_t(255) : uint8_t(s);
    }
  }
}

__global__ void __launch_bounds__(kPackWarps * 32)
unpack_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ codes,
              uint8_t* __restrict__ scales, int n_mat, int N, int K, int layout) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KB = K / kMxBlock, NT = N / kTileRows;
  const long long units = (long long)n_mat * NT * KB;
  const int r = lane >> 1, half = lane & 1;
  for (long long u = (long long)blockIdx.x * kPackWarps + warp; u < units;
       u += (long long)gridDim.x * kPackWarps) {
    const int kb = int(u % KB);
    const long long mt = u / KB;
    const int tile = int(mt % NT);
    const int mat = int(mt / NT);
    const uint8_t* unit = packed + ((long long)mat * NT * KB + (long long)tile * KB + kb) * kUnitBytes;
    // a unit row is the canonical row's 16 bytes of this K-block
    const int srow = source_row(layout, tile, r, N);
    const uint2 v = *reinterpret_cast<const uint2*>(unit + r * 16 + half * 8);
    uint8_t* dst = codes + ((long long)mat * N + srow) * (K / 2) + (long long)kb * 16 + half * 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      dst[j] = uint8_t(v.x >> (8 * j));
      dst[4 + j] = uint8_t(v.y >> (8 * j));
    }
    if (half == 0) {
      const int pos = r < 8 ? 2 * r : 2 * (r - 8) + 1;
      scales[((long long)mat * N + srow) * KB + kb] = unit[kUnitCodeBytes + pos];
    }
  }
}

bool shape_ok(int n_mat, int N, int K, int layout) {
  if (n_mat < 1 || N < kTileRows || K < kMxBlock) return false;
  if (N % kTileRows || K % kMxBlock) return false;
  if (layout != MOE_LAYOUT_TILE16 && layout != MOE_LAYOUT_TILE16_GATEUP) return false;
  return true;
}

int unit_grid(long long units, const DeviceInfo& di) {
  long long blocks = (units + kPackWarps - 1) / kPackWarps;
  long long cap = (long long)di.sm_count * 8;
  return int(blocks < cap ? blocks : cap);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_packed_bytes(int n_mat, int N, int K, int layout) {
  if (!shape_ok(n_mat, N, K, layout)) return 0;
  return (size_t)n_mat * (size_t)N * (size_t)K / 2 + (size_t)n_mat * (size_t)N * (size_t)K / 32;
}

extern "C" int moe_describe_packed(int n_mat, int N, int K, int layout, moe_packed_desc* out) {
  MOE_CHECK_ARG(out != nullptr, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(shape_ok(n_mat, N, K, layout), MOE_ERR_UNSUPPORTED_SHAPE);
  out->magic = MOE_PACK_MAGIC;
  out->version = MOE_PACK_VERSION;
  out->layout = layout;
  out->n_mat = n_mat;
  out->N = N;
  out->K = K;
  out->bytes_per_mat = (uint64_t)N * K / 2 + (uint64_t)N * K / 32;
  out->total_bytes = out->bytes_per_mat * (uint64_t)n_mat;
  return MOE_OK;
}

extern "C" int moe_pack_mxfp4(const float* w_dev, int n_mat, int N, int K, int layout,
                              void* packed_dev, size_t packed_bytes, moe_packed_desc* desc_out,
                              int* dev_status, moe_stream_t stream) {
  MOE_CHECK_ARG(w_dev && packed_dev, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(layout == MOE_LAYOUT_TILE16 || layout == MOE_LAYOUT_TILE16_GATEUP, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(shape_ok(n_mat, N, K, layout), MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK_ARG(aligned(w_dev, 16) && aligned(packed_dev, 16), MOE_ERR_INVALID_ARG);
  moe_packed_desc d;
  moe_describe_packed(n_mat, N, K, layout, &d);
  MOE_CHECK_ARG(packed_bytes >= d.total_bytes, MOE_ERR_BUFFER_TOO_SMALL);
  DeviceInfo di;
  int st = current_device(&di);
  if (st != MOE_OK) return st;
  const long long units = (long long)n_mat * (N / kTileRows) * (K / kMxBlock);
  pack_kernel<<<unit_grid(units, di), kPackWarps * 32, 0, (cudaStream_t)stream>>>(
      w_dev, static_cast<uint8_t*>(packed_dev), n_mat, N, K, layout, dev_status);
  st = launch_status();
  if (st == MOE_OK && desc_out) *desc_out = d;
  return st;
}

extern "C" int moe_unpack_mxfp4(const void* packed_dev, const moe_packed_desc* desc,
                                uint8_t* codes_dev, uint8_t* scales_dev, moe_stream_t stream) {
  MOE_CHECK_ARG(packed_dev && desc && codes_dev && scales_dev, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(desc->magic == MOE_PACK_MAGIC && desc->version == MOE_PACK_VERSION,
                MOE_ERR_BAD_DESCRIPTOR);
  MOE_CHECK_ARG(shape_ok(desc->n_mat, desc->N, desc->K, desc->layout), MOE_ERR_BAD_DESCRIPTOR);
  MOE_CHECK_ARG(aligned(packed_dev, 16), MOE_ERR_INVALID_ARG);
  DeviceInfo di;
  int st = current_device(&di);
  if (st != MOE_OK) return st;
  const long long units = (long long)desc->n_mat * (desc->N / kTileRows) * (desc->K / kMxBlock);
  unpack_kernel<<<unit_grid(units, di), kPackWarps * 32, 0, (cudaStream_t)stream>>>(
      static_cast<const uint8_t*>(packed_dev), codes_dev, scales_dev, desc->n_mat, desc->N,
      desc->K, desc->layout);
  return launch_status();
}
