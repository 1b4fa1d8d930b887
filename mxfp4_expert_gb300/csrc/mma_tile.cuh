// The 3-term e4m3 split of one 32-element activation block (B operand of the
// e4m3 warp MMA), and floor(log2). Shared by the per-stage expert kernels and
// the single-launch decode kernel.
#pragma once

#include "common.cuh"

namespace moe {

// floor(log2(a)) for finite a > 0 (fp32, including subnormals).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = int(b >> 23);
  if (e > 0) return e - 127;
  return (31 - __clz(int(b & 0x7FFFFFu))) - 149;
}

// Whole warp: lane j holds element j of a 32-element block. Writes the three
// e4m3 terms in B-fragment byte order to dst[0..96) and returns the block
// exponent e (value = (t0 + t1 + t2) * 2^e), or kActZeroExp. Within a term's
// 32 bytes, element j sits at bfrag_pos(j): lane q of a quad reads bytes
// [8q, 8q+8) = elements 8q + {0, 2, 4, 6} then 8q + {1, 3, 5, 7}, the K order
// of the A fragments (load_afrag).
__device__ __forceinline__ int split_block(float v, int lane, uint8_t* dst) {
  const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
  uint32_t t0 = 0, t1 = 0, t2 = 0;
  int e = kActZeroExp;
  if (amax > 0.0f) {
    e = floor_log2(amax) - 7;
    const float sv = scale2(v, -e);
    t0 = f32x2_to_e4m3x2(sv, 0.0f) & 0xFFu;
    const float r1 = sv - e4m3_to_f32_hw(t0);
    t1 = f32x2_to_e4m3x2(r1, 0.0f) & 0xFFu;
    const float r2 = r1 - e4m3_to_f32_hw(t1);
    t2 = f32x2_to_e4m3x2(r2, 0.0f) & 0xFFu;
  }
  const int pos = bfrag_pos(lane);
  dst[pos] = uint8_t(t0);
  dst[32 + pos] = uint8_t(t1);
  dst[64 + pos] = uint8_t(t2);
  return e;
}

}  // namespace moe
