// One packed MXFP4 unit (16 rows x 32 K) times activation B-fragments on the
// e4m3 warp MMA, and the 3-term e4m3 split of one 32-element activation block.
// Shared by the per-stage expert kernels and the single-launch decode kernel.
#pragma once

#include "common.cuh"

namespace moe {

// A-fragments (4 x e4m3x4) and the two row scales of one 272-byte unit, for
// this lane (g = lane/4 owns rows g and g+8).
struct UnitFrag {
  uint32_t a0, a1, a2, a3;
  uint32_t s_lo, s_hi;
};

__device__ __forceinline__ UnitFrag load_unit(const uint8_t* unit, int lane) {
  const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
  const uint32_t sc = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * (lane >> 2));
  UnitFrag f;
  f.a0 = decode_rowlo(wv.x);
  f.a1 = decode_rowhi(wv.x);
  f.a2 = decode_rowlo(wv.y);
  f.a3 = decode_rowhi(wv.y);
  f.s_lo = sc & 0xFFu;
  f.s_hi = sc >> 8;
  return f;
}

// acc_lo (row g) and acc_hi (row g+8) += block dot products for the token
// whose C-fragment columns this lane holds (exponent ex of its block).
__device__ __forceinline__ void unit_mma(const UnitFrag& f, uint2 b, int ex, float& acc_lo, float& acc_hi) {
  float d[4];
  mma_e4m3(d, f.a0, f.a1, f.a2, f.a3, b.x, b.y);
  acc_lo = fmaf(d[0] + d[1], block_factor(f.s_lo, ex), acc_lo);
  acc_hi = fmaf(d[2] + d[3], block_factor(f.s_hi, ex), acc_hi);
}

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
// 32 bytes, lane q of a quad reads bytes [8q, 8q+8) = k {4q..4q+3, 16+4q..16+4q+3}.
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
  const int pos = ((lane & 15) >> 2) * 8 + (lane >> 4) * 4 + (lane & 3);
  dst[pos] = uint8_t(t0);
  dst[32 + pos] = uint8_t(t1);
  dst[64 + pos] = uint8_t(t2);
  return e;
}

// B-fragment of one (activation row, K-block) for this lane: column g&3 is
// term g&3 (column 3 is zero), rows k {4q..4q+3} and {16+4q..16+4q+3}.
__device__ __forceinline__ uint2 load_bfrag_smem(const uint8_t* blk, int lane) {
  const int col = (lane >> 2) & 3, q = lane & 3;
  if (col == 3) return make_uint2(0u, 0u);
  return *reinterpret_cast<const uint2*>(blk + col * 32 + q * 8);
}

}  // namespace moe
