// bf16 GEMVs on CUDA cores: the router (E rows) and the shared expert's gate
// and up projections (routing-independent, one kernel), and the final
// combine: shared down projection plus the routing-weighted sum of the routed
// experts' outputs, rounded to bf16.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kTokChunk = 8;    // activation rows held in shared memory per pass
constexpr int kDenseWarps = 8;

// sum over 8 bf16 weights (one uint4) times 8 fp32 activations
__device__ __forceinline__ float dot8(uint4 w, const float* x) {
  const float4 xa = *reinterpret_cast<const float4*>(x);
  const float4 xb = *reinterpret_cast<const float4*>(x + 4);
  float s = bf16_lo(w.x) * xa.x;
  s = fmaf(bf16_hi(w.x), xa.y, s);
  s = fmaf(bf16_lo(w.y), xa.z, s);
  s = fmaf(bf16_hi(w.y), xa.w, s);
  s = fmaf(bf16_lo(w.z), xb.x, s);
  s = fmaf(bf16_hi(w.z), xb.y, s);
  s = fmaf(bf16_lo(w.w), xb.z, s);
  s = fmaf(bf16_hi(w.w), xb.w, s);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Items: router rows e in [0, E), then shared features i in [0, I) (gate row i
// and up row i together). One warp per item; lanes stride K by 8 elements.
__global__ void __launch_bounds__(kDenseWarps * 32)
front_kernel(FrontArgs a) {
  extern __shared__ __align__(16) float xs[];   // [kTokChunk][d]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_items = a.E + (a.sh_gate ? a.I : 0);
  for (int t0 = 0; t0 < a.T; t0 += kTokChunk) {
    const int tn = min(kTokChunk, a.T - t0);
    __syncthreads();
    for (int i = threadIdx.x; i < tn * a.d; i += blockDim.x)
      xs[i] = __bfloat162float(a.x[(size_t)t0 * a.d + i]);
    __syncthreads();
    for (int item = blockIdx.x * kDenseWarps + warp; item < n_items; item += gridDim.x * kDenseWarps) {
      const bool router = item < a.E;
      const __nv_bfloat16* r0 = router ? a.router_w + (size_t)item * a.d
                                       : a.sh_gate + (size_t)(item - a.E) * a.d;
      const __nv_bfloat16* r1 = router ? nullptr : a.sh_up + (size_t)(item - a.E) * a.d;
      float acc0[kTokChunk], acc1[kTokChunk];
#pragma unroll
      for (int tt = 0; tt < kTokChunk; ++tt) acc0[tt] = acc1[tt] = 0.0f;
#pragma unroll 4
      for (int j = lane * 8; j < a.d; j += 256) {
        const uint4 w0 = ldg_nc_stream_u4(r0 + j);
        uint4 w1 = make_uint4(0, 0, 0, 0);
        if (!router) w1 = ldg_nc_stream_u4(r1 + j);
#pragma unroll
        for (int tt = 0; tt < kTokChunk; ++tt) {
          if (tt < tn) {
            acc0[tt] += dot8(w0, xs + tt * a.d + j);
            if (!router) acc1[tt] += dot8(w1, xs + tt * a.d + j);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTokChunk; ++tt) {
        if (tt < tn) {
          const float g = warp_sum(acc0[tt]);
          const float u = router ? 0.0f : warp_sum(acc1[tt]);
          if (lane == 0) {
            if (router) a.logits[(size_t)(t0 + tt) * a.E + item] = g;
            else a.h_sh[(size_t)(t0 + tt) * a.I + (item - a.E)] = silu_f(g) * u;
          }
        }
      }
    }
  }
}

// One block per 16 output rows. Phase 1: shared down rows dot h_sh (warps
// split rows, lanes split I). Phase 2: y = shared + sum_j w[t][j] * part[slot][r].
__global__ void __launch_bounds__(kDenseWarps * 32)
combine_kernel(CombineArgs a) {
  extern __shared__ __align__(16) float sm[];    // h_sh chunk [kTokChunk][I], then sh_out[kTokChunk][16]
  float* hs = sm;
  float* sh_out = sm + kTokChunk * a.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = blockIdx.x * 16;
  for (int t0 = 0; t0 < a.T; t0 += kTokChunk) {
    const int tn = min(kTokChunk, a.T - t0);
    __syncthreads();
    if (a.sh_down) {
      for (int i = threadIdx.x; i < tn * a.I; i += blockDim.x) hs[i] = a.h_sh[(size_t)t0 * a.I + i];
    }
    __syncthreads();
    for (int rr = warp; rr < 16; rr += kDenseWarps) {
      float acc[kTokChunk];
#pragma unroll
      for (int tt = 0; tt < kTokChunk; ++tt) acc[tt] = 0.0f;
      if (a.sh_down) {
        const __nv_bfloat16* wr = a.sh_down + (size_t)(r0 + rr) * a.I;
        for (int j = lane * 8; j < a.I; j += 256) {
          const uint4 w = ldg_nc_stream_u4(wr + j);
#pragma unroll
          for (int tt = 0; tt < kTokChunk; ++tt)
            if (tt < tn) acc[tt] += dot8(w, hs + tt * a.I + j);
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTokChunk; ++tt) {
        const float v = warp_sum(acc[tt]);
        if (lane == 0 && tt < tn) sh_out[tt * 16 + rr] = v;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < tn * 16; i += blockDim.x) {
      const int tt = i >> 4, r = i & 15, t = t0 + tt;
      float y = sh_out[tt * 16 + r];
      for (int j = 0; j < a.k; ++j) {
        const int slot = a.inv[(size_t)t * a.k + j];
        if (slot >= 0) y = fmaf(a.w[(size_t)t * a.k + j], a.part[(size_t)slot * a.d + r0 + r], y);
      }
      a.y[(size_t)t * a.d + r0 + r] = __float2bfloat16_rn(y);
    }
  }
}

}  // namespace

int launch_front(const FrontArgs& a, const DeviceInfo& di, cudaStream_t s) {
  const size_t smem = sizeof(float) * kTokChunk * a.d;
  MOE_CUDA_TRY(cudaFuncSetAttribute(front_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  const int n_items = a.E + (a.sh_gate ? a.I : 0);
  int grid = (n_items + kDenseWarps - 1) / kDenseWarps;
  if (grid > di.sm_count * 2) grid = di.sm_count * 2;
  front_kernel<<<grid, kDenseWarps * 32, smem, s>>>(a);
  return launch_status();
}

int launch_combine(const CombineArgs& a, const DeviceInfo& di, cudaStream_t s) {
  (void)di;
  const size_t smem = sizeof(float) * (kTokChunk * a.I + kTokChunk * 16);
  MOE_CUDA_TRY(cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  combine_kernel<<<a.d / 16, kDenseWarps * 32, smem, s>>>(a);
  return launch_status();
}

}  // namespace moe
