// Warp-wide top-k with renormalised softmax weights over one row of fp32
// logits (E <= 1024, k <= 32). Each lane keeps up to 32 candidate keys in
// registers; every round takes the warp maximum with redux.sync, breaks ties
// to the lowest expert index with a second redux, and retires the winner.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving map fp32 -> uint32: a larger key is a larger value. -0
// ranks as +0 and NaN as -inf; 0 is reserved for "no candidate".
__device__ __forceinline__ uint32_t rank_key(float v) {
  if (isnan(v)) return 0x007FFFFFu;
  if (v == 0.0f) v = 0.0f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float rank_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Candidate key of expert e: logit (+ bias, fp32 round-to-nearest) or 0 if e >= E.
template <bool kCoherent>
__device__ __forceinline__ uint32_t candidate(const float* row, const float* brow, int e, int E) {
  if (e >= E) return 0u;
  float v = kCoherent ? __ldcg(row + e) : row[e];
  if (brow) v = __fadd_rn(v, brow[e]);
  return rank_key(v);
}

// Selects k experts for one token. Lane j < k returns the j-th selected expert
// (descending key, ties to the lower index) in *e_out and its weight in *w_out.
// kPL = per-lane capacity (E <= 32 * kPL). kCoherent: read logits through L2
// (they were written by other CTAs of the same kernel).
template <int kPL, bool kCoherent>
__device__ __forceinline__ void warp_topk(const float* row, const float* brow, int E, int k, int lane,
                                          int* e_out, float* w_out) {
  uint32_t key[kPL];
#pragma unroll
  for (int i = 0; i < kPL; ++i) key[i] = candidate<kCoherent>(row, brow, i * 32 + lane, E);
  uint32_t bk = 0u, be = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < kPL; ++i)
    if (key[i] > bk) { bk = key[i]; be = uint32_t(i * 32 + lane); }
  uint32_t my_e = 0, my_key = 0;
  for (int r = 0; r < k; ++r) {
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, bk == wmax ? be : 0xFFFFFFFFu);
    if (lane == r) { my_e = emin; my_key = wmax; }
    if (lane == int(emin & 31u)) {
      const int slot = int(emin >> 5);
      bk = 0u;
      be = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < kPL; ++i) {
        if (i == slot) key[i] = 0u;
        if (key[i] > bk) { bk = key[i]; be = uint32_t(i * 32 + lane); }
      }
    }
  }
  const float v = rank_value(my_key);
  const float v0 = __shfl_sync(0xFFFFFFFFu, v, 0);
  const float ex = lane < k ? expf(v - v0) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  *e_out = int(my_e);
  *w_out = ex / sum;
}

}  // namespace moe
