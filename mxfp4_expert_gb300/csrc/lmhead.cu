// FP8 LM head: logits[t][v] = s_v * sum_j x[t][j] * W8[v][j] for a vocabulary
// of V rows (page "3 ways to speed up MoE inference on NVIDIA DGX Spark", §4:
// the LM head quantised online from BF16 to FP8 halves the bytes read per
// decode step). W8 is E4M3 row-major [V][d] with one fp32 scale per row.
//
// Decode is bound by reading W8 once (d bytes per row). A warp owns items of
// 16 rows x half of K and multiplies them on the e4m3 warp MMA (m16n8k32)
// against x split into 3 e4m3 terms per 32-element block (exact for bf16 x).
// Lane (g, q) loads bytes [8q, 8q + 8) of rows g and g + 8 of each 32-wide
// K-block: the MMA reads those 8 bytes as its K positions {4q..4q+3,
// 16+4q..16+4q+3}, and the B fragment is taken from the same 8 bytes of the
// x terms, so both operands agree on the order without any shuffling and the
// weights keep their plain row-major layout. The two K halves of a row are
// added with float atomics into logits zeroed beforehand; with exactly two
// addends the sum does not depend on their order, so results are
// deterministic.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "mma_tile.cuh"

namespace moe {
namespace {

constexpr int kLWarps = 16;
constexpr int kLThreads = kLWarps * 32;
constexpr int kLBatch = 8;     // K-blocks a lane loads together (16 bytes each)

// per-row fp32 scale and E4M3 codes (quantisation of one bf16 row per block)
__global__ void __launch_bounds__(256) lm_pack_kernel(const __nv_bfloat16* w, int d, uint8_t* codes, float* scales) {
  const int v = blockIdx.x, tid = threadIdx.x;
  const __nv_bfloat16* row = w + (size_t)v * d;
  float am = 0.0f;
  for (int j = tid; j < d; j += blockDim.x) am = fmaxf(am, fabsf(__bfloat162float(row[j])));
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
  if ((tid & 31) == 0) red[tid >> 5] = am;
  __syncthreads();
  am = red[0];
  for (int i = 1; i < int(blockDim.x >> 5); ++i) am = fmaxf(am, red[i]);
  const float s = am == 0.0f ? 1.0f : __fdiv_rn(am, 448.0f);
  if (tid == 0) scales[v] = s;
  for (int j = 2 * tid; j < d; j += 2 * blockDim.x) {
    const float a = __fdiv_rn(__bfloat162float(row[j]), s);
    const float b = __fdiv_rn(__bfloat162float(row[j + 1]), s);
    *reinterpret_cast<uint16_t*>(codes + (size_t)v * d + j) = f32x2_to_e4m3x2(a, b);
  }
}

// x [T][d] bf16 -> 3 e4m3 terms per 32-block, natural K order:
// xt[t][kb][term][32], factor xf[t][kb] = 2^e (0 for a zero block)
template <int T>
__global__ void __launch_bounds__(kLThreads, 2) lm_gemv_kernel(const uint8_t* __restrict__ codes,
                                                             const float* __restrict__ scales, int V, int d,
                                                             const __nv_bfloat16* __restrict__ x,
                                                             float* __restrict__ logits) {
  extern __shared__ __align__(16) uint8_t lsm[];
  constexpr int kPairs = (T + 1) / 2;
  const int KB = d / kMxBlock, KBh = KB / 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
  uint8_t* xt = lsm;                                                     // [T][KB][3][32]
  float* xf = reinterpret_cast<float*>(lsm + (size_t)T * KB * 96);      // [T][KB]
  for (int u = warp; u < T * KB; u += kLWarps) {
    const float v = __bfloat162float(x[(size_t)u * kMxBlock + lane]);
    // split_block writes B-fragment order; the natural order is wanted here
    const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
    uint32_t t0 = 0, t1 = 0, t2 = 0;
    int e = kActZeroExp;
    if (amax > 0.0f) {
      e = floor_log2(amax) - 7;
      const float sv = scale2(v, -e);
      t0 = f32x2_to_e4m3x2(sv, 0.0f) & 0xFFu;
      const float r1 = sv - e4m3_to_f32_hw(t0);
      t1 = f32x2_to_e4m3x2(r1, 0.0f) & 0xFFu;
      t2 = f32x2_to_e4m3x2(r1 - e4m3_to_f32_hw(t1), 0.0f) & 0xFFu;
    }
    uint8_t* dst = xt + (size_t)u * 96;
    dst[lane] = uint8_t(t0);
    dst[32 + lane] = uint8_t(t1);
    dst[64 + lane] = uint8_t(t2);
    if (lane == 0) xf[u] = e == kActZeroExp ? 0.0f : scale2(1.0f, e);
  }
  __syncthreads();
  // B offsets per token pair: column g of the MMA is token 2p + g/4, term g%4
  int boff[kPairs];
  bool bok[kPairs];
#pragma unroll
  for (int p = 0; p < kPairs; ++p) {
    const int t = 2 * p + (g >> 2), term = g & 3;
    bok[p] = t < T && term < 3;
    boff[p] = (t < T ? t : 0) * KB * 96 + (term < 3 ? term : 0) * 32 + 8 * q;
  }
  const int n_items = (V / kTileRows) * 2;
  const int gw = blockIdx.x * kLWarps + warp, nw = gridDim.x * kLWarps;
#pragma unroll 1
  for (int it = gw; it < n_items; it += nw) {
    const int tile = it >> 1, half = it & 1;
    const int kb0 = half * KBh, kb1 = half ? KB : KBh;
    const uint8_t* r0 = codes + (size_t)(tile * kTileRows + g) * d + 8 * q;
    const uint8_t* r1 = r0 + (size_t)8 * d;
    float acc[kPairs][2];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) acc[p][0] = acc[p][1] = 0.0f;
#pragma unroll 1
    for (int kb = kb0; kb < kb1; kb += kLBatch) {
      uint2 wa[kLBatch], wb[kLBatch];
#pragma unroll
      for (int u = 0; u < kLBatch; ++u) {
        const int k = min(kb + u, kb1 - 1) * kMxBlock;
        wa[u] = ldg_nc_u2(r0 + k);
        wb[u] = ldg_nc_u2(r1 + k);
      }
#pragma unroll
      for (int u = 0; u < kLBatch; ++u) {
        if (kb + u < kb1) {
#pragma unroll
          for (int p = 0; p < kPairs; ++p) {
            const uint2 bv = bok[p] ? *reinterpret_cast<const uint2*>(xt + boff[p] + (kb + u) * 96) : make_uint2(0u, 0u);
            const int tq = 2 * p + (q >> 1);
            const float fa = tq < T ? xf[tq * KB + kb + u] : 0.0f;
            float dd[4];
            mma_e4m3(dd, wa[u].x, wb[u].x, wa[u].y, wb[u].y, bv.x, bv.y);
            acc[p][0] = fmaf(dd[0] + dd[1], fa, acc[p][0]);
            acc[p][1] = fmaf(dd[2] + dd[3], fa, acc[p][1]);
          }
        }
      }
    }
    // terms of a token sit in lanes q and q^1
    const int v0 = tile * kTileRows + g;
    const float s0 = scales[v0], s1 = scales[v0 + 8];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      const float lo = acc[p][0] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][0], 1);
      const float hi = acc[p][1] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][1], 1);
      const int t = 2 * p + (q >> 1);
      if ((q & 1) == 0 && t < T) {
        atomicAdd(logits + (size_t)t * V + v0, lo * s0);
        atomicAdd(logits + (size_t)t * V + v0 + 8, hi * s1);
      }
    }
  }
}

template <int T>
int launch_lm(const uint8_t* codes, const float* scales, int V, int d, const __nv_bfloat16* x, float* logits,
              const DeviceInfo& di, cudaStream_t s) {
  const size_t smem = (size_t)T * (d / kMxBlock) * (96 + 4);
  if (smem + 1024 > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  MOE_CUDA_TRY(cudaFuncSetAttribute(lm_gemv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  int per_sm = 0;
  MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lm_gemv_kernel<T>, kLThreads, smem));
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  lm_gemv_kernel<T><<<di.sm_count * per_sm, kLThreads, smem, s>>>(codes, scales, V, d, x, logits);
  return launch_status();
}

}  // namespace

int launch_lm_pack(const void* w, int V, int d, uint8_t* codes, float* scales, cudaStream_t s) {
  lm_pack_kernel<<<V, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w), d, codes, scales);
  return launch_status();
}

int launch_lm_gemv(const uint8_t* codes, const float* scales, int V, int d, const void* x, int T, float* logits,
                   const DeviceInfo& di, cudaStream_t s) {
  MOE_CUDA_TRY(cudaMemsetAsync(logits, 0, sizeof(float) * (size_t)T * V, s));
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  switch (T) {
    case 1: return launch_lm<1>(codes, scales, V, d, xb, logits, di, s);
    case 2: return launch_lm<2>(codes, scales, V, d, xb, logits, di, s);
    case 3: return launch_lm<3>(codes, scales, V, d, xb, logits, di, s);
    case 4: return launch_lm<4>(codes, scales, V, d, xb, logits, di, s);
    case 5: return launch_lm<5>(codes, scales, V, d, xb, logits, di, s);
    case 6: return launch_lm<6>(codes, scales, V, d, xb, logits, di, s);
    case 7: return launch_lm<7>(codes, scales, V, d, xb, logits, di, s);
    default: return launch_lm<8>(codes, scales, V, d, xb, logits, di, s);
  }
}

}  // namespace moe
