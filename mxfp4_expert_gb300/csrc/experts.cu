// Routed-expert GEMVs over MXFP4 weights (gate/up with SwiGLU, and down).
//
// Each work item is one 16-row tile of one active expert's matrix over the
// whole K. The tile (K/32 units of 272 bytes) is fetched with one 1-D bulk
// copy into a ring of shared-memory stages; all items of a CTA are requested
// up front as far as the ring allows, so the HBM queue stays full. Eight warps
// split the K-blocks; per K-block a lane loads its 8 code bytes, turns them
// into four e4m3x4 registers with mask/shift operations (the packed format
// places every code where an E4M3 byte worth 2^-6 times the E2M1 value has
// its bits), and one m16n8k32 e4m3 MMA multiplies 16 rows by two activation
// rows (4 columns each: the activation split into e4m3 terms, see
// act_split_kernel). The E8M0 scale of the weight block and the exponent of
// the activation block are applied to the MMA result in fp32, so the sum over
// K-blocks is an fp32 accumulation of exact block dot products of the split
// terms.
//
// Why MMA: decoding E2M1 to fp32 costs at least two integer operations per
// element and an FMA after it; at HBM speed that is most of the SM's issue
// slots for T = 1 and more than all of them for T = 4 .. 64. Decoding to e4m3
// costs 10 operations per 16 elements and the MMA takes the multiply-adds.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "mma_tile.cuh"

namespace moe {
namespace {

// One warp per (row, K-block): 32 values -> e4m3 terms hi, lo, lo2 with
// value = (hi + lo + lo2) * 2^e, e chosen so the block maximum scaled by 2^-e
// lies in [128, 256). The remainder after each term is exact in fp32, so three
// terms carry 12 significant bits; bf16 inputs (8 bits) are reproduced exactly
// except for elements more than 2^10 below their block maximum.
__global__ void __launch_bounds__(256)
act_split_kernel(const void* __restrict__ src, int src_bf16, int rows, int K,
                 uint8_t* __restrict__ act_b, int16_t* __restrict__ act_e) {
  const int lane = threadIdx.x & 31;
  const int KB = K / kMxBlock;
  const long long units = (long long)rows * KB;
  for (long long u = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); u < units;
       u += (long long)gridDim.x * 8) {
    const long long row = u / KB;
    const int kb = int(u % KB);
    const long long off = row * K + (long long)kb * kMxBlock + lane;
    const float v = src_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(src)[off])
                             : static_cast<const float*>(src)[off];
    const int e = split_block(v, lane, act_b + u * kActRowKbBytes);
    if (lane == 0) act_e[u] = int16_t(e);
  }
}

constexpr int kRoutedWarps = 8;
constexpr int kPairs = 4;   // activation-row pairs per pass (one MMA each)

template <int MODE>
__global__ void __launch_bounds__(kRoutedWarps * 32, 1)
routed_kernel(RoutedArgs a, int stages, uint32_t item_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)stages * item_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kRoutedWarps * kPairs * 32 * 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n_items = *a.n_active * a.n_tiles;
  const int lo = int((long long)blockIdx.x * n_items / gridDim.x);
  const int hi = int((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  if (lo >= hi) return;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](int item, int s) {
    const int ai = item / a.n_tiles, tile = item % a.n_tiles;
    const int e = a.active[ai];
    const uint8_t* src = a.w + (uint64_t)e * a.mat_bytes + (uint64_t)tile * a.KB * kUnitBytes;
    mbar_arrive_expect_tx(&full[s], item_bytes);
    bulk_g2s(ring + (size_t)s * item_bytes, src, item_bytes, &full[s]);
  };
  if (tid == 0)
    for (int s = 0; s < stages && lo + s < hi; ++s) issue(lo + s, s);

  for (int it = lo; it < hi; ++it) {
    const int rel = it - lo, s = rel % stages;
    // block-uniform, so every __syncthreads below is reached by all threads
    const bool ok = __syncthreads_and(mbar_wait(&full[s], uint32_t(rel / stages) & 1u, a.status));
    const uint8_t* st = ring + (size_t)s * item_bytes;
    const int ai = it / a.n_tiles, tile = it % a.n_tiles;
    const int e = a.active[ai];
    const int pos0 = a.offsets[e];
    const int n = ok ? a.offsets[e + 1] - pos0 : 0;
    for (int c0 = 0; c0 < n; c0 += 2 * kPairs) {
      int brow[kPairs], crow[kPairs];
#pragma unroll
      for (int pr = 0; pr < kPairs; ++pr) {
        const int sb = c0 + 2 * pr + (g >> 2), sc = c0 + 2 * pr + (q >> 1);
        brow[pr] = sb < n ? (a.act_by_token ? a.perm[pos0 + sb] / a.k : pos0 + sb) : -1;
        crow[pr] = sc < n ? (a.act_by_token ? a.perm[pos0 + sc] / a.k : pos0 + sc) : -1;
      }
      float acc[kPairs][2];
#pragma unroll
      for (int pr = 0; pr < kPairs; ++pr) acc[pr][0] = acc[pr][1] = 0.0f;
      for (int kb = warp; kb < a.KB; kb += kRoutedWarps) {
        const uint8_t* unit = st + (size_t)kb * kUnitBytes;
        const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
        const uint32_t a0 = decode_rowlo(wv.x), a1 = decode_rowhi(wv.x);
        const uint32_t a2 = decode_rowlo(wv.y), a3 = decode_rowhi(wv.y);
        const uint32_t sc = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
        const uint32_t s_lo = sc & 0xFFu, s_hi = sc >> 8;
#pragma unroll
        for (int pr = 0; pr < kPairs; ++pr) {
          if (c0 + 2 * pr >= n) break;
          uint2 bv = make_uint2(0u, 0u);
          if (brow[pr] >= 0 && (g & 3) < kActTerms)
            bv = ldg_nc_u2(a.act_b + ((size_t)brow[pr] * a.KB + kb) * kActRowKbBytes + (g & 3) * 32 + q * 8);
          const int ex = crow[pr] >= 0 ? int(__ldg(a.act_e + (size_t)crow[pr] * a.KB + kb)) : int(kActZeroExp);
          float d[4];
          mma_e4m3(d, a0, a1, a2, a3, bv.x, bv.y);
          acc[pr][0] = fmaf(d[0] + d[1], block_factor(s_lo, ex), acc[pr][0]);
          acc[pr][1] = fmaf(d[2] + d[3], block_factor(s_hi, ex), acc[pr][1]);
        }
      }
#pragma unroll
      for (int pr = 0; pr < kPairs; ++pr) {
        red[((warp * kPairs + pr) * 32 + lane) * 2 + 0] = acc[pr][0];
        red[((warp * kPairs + pr) * 32 + lane) * 2 + 1] = acc[pr][1];
      }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int pr = 0; pr < kPairs; ++pr) {
          if (c0 + 2 * pr >= n) break;
          float v0 = 0.0f, v1 = 0.0f;
#pragma unroll
          for (int w = 0; w < kRoutedWarps; ++w) {
            v0 += red[((w * kPairs + pr) * 32 + lane) * 2 + 0];
            v1 += red[((w * kPairs + pr) * 32 + lane) * 2 + 1];
          }
          v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);   // terms 0,1 + terms 2,3
          v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
          const int sc = c0 + 2 * pr + (q >> 1);
          if ((q & 1) == 0 && sc < n) {
            float* o = a.out + (size_t)(pos0 + sc) * a.out_ld;
            if (MODE == kModeGateUp) {
              o[tile * 8 + g] = silu_f(v0) * v1;         // row g = gate, row g+8 = up
            } else {
              o[tile * kTileRows + g] = v0;
              o[tile * kTileRows + g + 8] = v1;
            }
          }
        }
      }
      __syncthreads();
    }
    __syncthreads();
    if (tid == 0 && it + stages < hi) issue(it + stages, s);
  }
}

}  // namespace

int launch_act_split(const void* src, bool src_bf16, int rows, int K, uint8_t* act_b,
                     int16_t* act_e, const DeviceInfo& di, cudaStream_t s) {
  const long long units = (long long)rows * (K / kMxBlock);
  long long blocks = (units + 7) / 8;
  const long long cap = (long long)di.sm_count * 8;
  if (blocks > cap) blocks = cap;
  act_split_kernel<<<int(blocks), 256, 0, s>>>(src, src_bf16 ? 1 : 0, rows, K, act_b, act_e);
  return launch_status();
}

int launch_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s) {
  const uint32_t item_bytes = uint32_t(a.KB) * kUnitBytes;
  const size_t fixed = sizeof(float) * kRoutedWarps * kPairs * 32 * 2;
  const size_t budget = (di.smem_optin > fixed + 4096 ? di.smem_optin - fixed - 4096 : 0);
  int stages = int(budget / (item_bytes + 8));
  if (stages > 16) stages = 16;
  if (stages < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  const size_t smem = (size_t)stages * item_bytes + fixed + (size_t)stages * 8;
  int grid = di.sm_count;
  if (a.max_items < grid) grid = a.max_items > 0 ? a.max_items : 1;
  if (mode == kModeGateUp) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(routed_kernel<kModeGateUp>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    routed_kernel<kModeGateUp><<<grid, kRoutedWarps * 32, smem, s>>>(a, stages, item_bytes);
  } else {
    MOE_CUDA_TRY(cudaFuncSetAttribute(routed_kernel<kModeDown>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    routed_kernel<kModeDown><<<grid, kRoutedWarps * 32, smem, s>>>(a, stages, item_bytes);
  }
  return launch_status();
}

}  // namespace moe
