// bf16 GEMMs on the warp-level tensor-core MMA (m16n8k16, fp32 accumulate)
// for the routing-independent dense parts of the per-stage path. The router
// and the shared expert stay in bf16 (page "MoE-SpeQ ...", §2.1-§2.2: routing
// is sensitive to quantisation, and the shared expert acts on every token):
//   * the router and the shared expert's gate/up projections in one kernel
//     (SwiGLU in the epilogue), and
//   * the combine: the shared down projection plus the routing-weighted sum of
//     the routed experts' outputs, rounded to bf16.
//
// C[weight row][token] = sum_k W[row][k] * X[token][k]: the weight rows are
// the MMA's M dimension (16 per warp), the tokens its N dimension (8 per MMA),
// both operands K-contiguous in memory. A block computes 16 * WM weight rows x
// 64 tokens with its 4 warps arranged WM along the rows and 4 / WM along the
// tokens: 64 rows when there are many tokens (the weight tile is reused by
// 64 tokens), 16 rows for at most 64 tokens (4x more blocks, so the weight
// bytes are spread over every SM). K goes in steps of 32 through padded
// shared-memory tiles (80-byte rows, so the ldmatrix row reads hit distinct
// banks), with the next step's tiles loaded into registers while the current
// one is multiplied.
//
// In the first kernel the shared gate and up rows are interleaved 8 + 8 per
// 16-row tile (as the TILE16_GATEUP weight layout does), so one lane holds gate and up of the
// same feature for the SwiGLU; h_sh goes out as fp32, or as the two bf16
// terms the tcgen05 combine reads. The shared down projection reads h_sh (fp32)
// as two bf16 terms, hi = bf16(h) and lo = bf16(h - hi), about 16 significant
// bits, with one MMA per term.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBN = 64;            // tokens per block
constexpr int kDWarps = 4;
constexpr int kDThreads = kDWarps * 32;
constexpr int kSmallT = 64;        // up to this many tokens: 16-row blocks

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Weight row n of the first kernel: router rows [0, Ep) (rows >= E are zero),
// then the shared expert's rows in 16-row tiles of 8 gate + 8 up rows.
__device__ __forceinline__ const __nv_bfloat16* front_row(const FrontArgs& a, int Ep, int n) {
  if (n < Ep) return n < a.E ? a.router_w + (size_t)n * a.d : nullptr;
  const int s = n - Ep;
  if (!a.sh_gate || s >= 2 * a.I) return nullptr;
  const int f = (s >> 4) * 8 + (s & 7);
  return ((s & 8) ? a.sh_up : a.sh_gate) + (size_t)f * a.d;
}

// MODE 0: router + shared gate/up (FrontArgs). MODE 1: shared down + combine
// (CombineArgs). Both share the tiling; P carries the mode's arguments.
// BK: K per step (128 for 16-row blocks and 64 for the router + shared
// gate/up with 64-row blocks when K allows, else 32: fewer and larger steps
// hide more of the load latency). K % BK == 0.
template <int MODE, int WM, int BK, typename P>
__global__ void __launch_bounds__(kDThreads)
dense_kernel(P a, int Ep, int N, int K) {
  constexpr int kBM = 16 * WM;              // weight rows per block
  constexpr int kBK = BK;
  constexpr int kLd = kBK + 8;              // shared-memory row, bf16 elements
  constexpr int kCPR = kBK / 8;             // 16-byte chunks per tile row
  constexpr int kRPP = kDThreads / kCPR;    // tile rows per pass of the block
  constexpr int kNT = kBN / 8 / (kDWarps / WM);   // 8-token MMA tiles per warp
  constexpr int kWH = (kBM + kRPP - 1) / kRPP;    // weight-tile passes
  constexpr int kXH = kBN / kRPP;                 // token-tile passes
  __shared__ __align__(16) __nv_bfloat16 Ws[kBM * kLd];
  __shared__ __align__(16) __nv_bfloat16 Xh[kBN * kLd];
  __shared__ __align__(16) __nv_bfloat16 Xl[MODE == 1 ? kBN * kLd : 8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp % WM, wn = warp / WM;   // the warp's 16 rows and kNT token tiles
  const int n0 = blockIdx.x * kBM, t0 = blockIdx.y * kBN;
  const int T = a.T;
  bool have_w = true;
  if constexpr (MODE == 1) have_w = a.sh_down != nullptr;

  // per thread: 16-byte chunk column cc = (tid % kCPR) * 8 of the weight-tile
  // rows cr + kRPP h (only rows < kBM) and of the token-tile rows cr + kRPP h
  // (8 fp32 of h_sh in MODE 1), cr = tid / kCPR
  const __nv_bfloat16* wrow[kWH];
  const void* xrow[kXH];
  const int cr = tid / kCPR, cc = (tid % kCPR) * 8;
#pragma unroll
  for (int h = 0; h < kWH; ++h) {
    const int r = cr + kRPP * h;
    if constexpr (MODE == 0)
      wrow[h] = r < kBM ? front_row(a, Ep, n0 + r) : nullptr;
    else
      wrow[h] = (r < kBM && have_w && n0 + r < N) ? a.sh_down + (size_t)(n0 + r) * K : nullptr;
  }
#pragma unroll
  for (int h = 0; h < kXH; ++h) {
    const int r = cr + kRPP * h;
    if constexpr (MODE == 0)
      xrow[h] = t0 + r < T ? static_cast<const void*>(a.x + (size_t)(t0 + r) * K) : nullptr;
    else
      xrow[h] = t0 + r < T ? static_cast<const void*>(a.h_sh + (size_t)(t0 + r) * K) : nullptr;
  }
  uint4 wreg[kWH], xh[kXH], xl[MODE == 1 ? kXH : 1];
  auto load = [&](int k0) {
#pragma unroll
    for (int h = 0; h < kWH; ++h)
      wreg[h] = wrow[h] ? ldg_nc_stream_u4(wrow[h] + k0 + cc) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int h = 0; h < kXH; ++h) {
      if constexpr (MODE == 0) {
        xh[h] = xrow[h] ? __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(xrow[h]) + k0 + cc))
                        : make_uint4(0u, 0u, 0u, 0u);
      } else {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (xrow[h]) {
          const float4 u0 = *reinterpret_cast<const float4*>(static_cast<const float*>(xrow[h]) + k0 + cc);
          const float4 u1 = *reinterpret_cast<const float4*>(static_cast<const float*>(xrow[h]) + k0 + cc + 4);
          v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
          v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = __bfloat162float(__float2bfloat16_rn(v[2 * e]));
          const float a1 = __bfloat162float(__float2bfloat16_rn(v[2 * e + 1]));
          hi[e] = pack_bf16(a0, a1);
          lo[e] = pack_bf16(v[2 * e] - a0, v[2 * e + 1] - a1);
        }
        xh[h] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        xl[h] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int h = 0; h < kWH; ++h)
      if (cr + kRPP * h < kBM) *reinterpret_cast<uint4*>(Ws + (cr + kRPP * h) * kLd + cc) = wreg[h];
#pragma unroll
    for (int h = 0; h < kXH; ++h) {
      const int r = cr + kRPP * h;
      *reinterpret_cast<uint4*>(Xh + r * kLd + cc) = xh[h];
      if constexpr (MODE == 1) *reinterpret_cast<uint4*>(Xl + r * kLd + cc) = xl[h];
    }
  };

  float acc[kNT][4];
#pragma unroll
  for (int j = 0; j < kNT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

  if (have_w) {
    load(0);
    for (int k0 = 0; k0 < K; k0 += kBK) {
      __syncthreads();   // the previous step's tiles are no longer read
      store();
      __syncthreads();
      if (k0 + kBK < K) load(k0 + kBK);   // next step's tiles in flight during the MMAs
#pragma unroll
      for (int ks = 0; ks < kBK; ks += 16) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, Ws + (wm * 16 + (lane & 15)) * kLd + ks + (lane >> 4) * 8);
#pragma unroll
        for (int j = 0; j < kNT; j += 2) {
          const int xr = (wn * kNT + j) * 8 + (lane & 7) + ((lane >> 4) << 3), xc = ks + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, Xh + xr * kLd + xc);
          mma_bf16(acc[j], a0, a1, a2, a3, b0, b1);
          mma_bf16(acc[j + 1], a0, a1, a2, a3, b2, b3);
          if constexpr (MODE == 1) {
            ldsm_x4(b0, b1, b2, b3, Xl + xr * kLd + xc);
            mma_bf16(acc[j], a0, a1, a2, a3, b0, b1);
            mma_bf16(acc[j + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
    }
  }

  // lane (g, q): rows m = n0 + 16 wm + g (c[0], c[1]) and m + 8 (c[2], c[3]),
  // tokens t0 + 8 (wn kNT + j) + 2 q + {0, 1}
  const int g = lane >> 2, q = lane & 3;
  const int m = n0 + wm * 16 + g;
#pragma unroll
  for (int j = 0; j < kNT; ++j) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int t = t0 + (wn * kNT + j) * 8 + 2 * q + u;
      if (t >= T) continue;
      if constexpr (MODE == 0) {
        if (n0 + wm * 16 < Ep) {
          if (m < a.E) a.logits[(size_t)t * a.E + m] = acc[j][u];
          if (m + 8 < a.E) a.logits[(size_t)t * a.E + m + 8] = acc[j][2 + u];
        } else if (a.sh_gate) {
          const int s = m - Ep;   // gate row of feature f in c[u], its up row in c[2 + u]
          const int f = (s >> 4) * 8 + (s & 7);
          if (f < a.I) {
            const float h = silu_f(acc[j][u]) * acc[j][2 + u];
            if (a.h_hi) {
              const __nv_bfloat16 hi = __float2bfloat16_rn(h);
              a.h_hi[(size_t)t * a.I + f] = hi;
              a.h_lo[(size_t)t * a.I + f] = __float2bfloat16_rn(h - __bfloat162float(hi));
            } else {
              a.h_sh[(size_t)t * a.I + f] = h;
            }
          }
        }
      } else {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = m + 8 * hh;
          if (r >= N) continue;
          float y = acc[j][2 * hh + u];
          for (int jj = 0; jj < a.k; ++jj) {
            const int slot = a.inv[(size_t)t * a.k + jj];
            if (slot >= 0) y = fmaf(a.w[(size_t)t * a.k + jj], a.part[(size_t)slot * a.d + r], y);
          }
          a.y[(size_t)t * a.d + r] = __float2bfloat16_rn(y);
        }
      }
    }
  }
}

}  // namespace

int launch_front(const FrontArgs& a, const DeviceInfo& di, cudaStream_t s) {
  (void)di;
  const int Ep = (a.E + 15) / 16 * 16;
  const int N = Ep + (a.sh_gate ? 2 * a.I : 0);
  if (a.T <= kSmallT && a.d % 128 == 0)
    dense_kernel<0, 1, 128, FrontArgs><<<dim3((N + 15) / 16, 1), kDThreads, 0, s>>>(a, Ep, N, a.d);
  else if (a.T <= kSmallT)
    dense_kernel<0, 1, 32, FrontArgs><<<dim3((N + 15) / 16, 1), kDThreads, 0, s>>>(a, Ep, N, a.d);
  else if (a.d % 64 == 0)
    dense_kernel<0, 4, 64, FrontArgs><<<dim3((N + 63) / 64, (a.T + kBN - 1) / kBN), kDThreads, 0, s>>>(a, Ep, N, a.d);
  else
    dense_kernel<0, 4, 32, FrontArgs><<<dim3((N + 63) / 64, (a.T + kBN - 1) / kBN), kDThreads, 0, s>>>(a, Ep, N, a.d);
  return launch_status();
}

int launch_combine(const CombineArgs& a, const DeviceInfo& di, cudaStream_t s) {
  (void)di;
  if (a.T <= kSmallT && a.I % 128 == 0)
    dense_kernel<1, 1, 128, CombineArgs><<<dim3((a.d + 15) / 16, 1), kDThreads, 0, s>>>(a, 0, a.d, a.I);
  else if (a.T <= kSmallT)
    dense_kernel<1, 1, 32, CombineArgs><<<dim3((a.d + 15) / 16, 1), kDThreads, 0, s>>>(a, 0, a.d, a.I);
  else   // (64-wide steps are slower here: the h_sh hi/lo split doubles the staged registers)
    dense_kernel<1, 4, 32, CombineArgs><<<dim3((a.d + 63) / 64, (a.T + kBN - 1) / kBN), kDThreads, 0, s>>>(a, 0, a.d,
                                                                                                       a.I);
  return launch_status();
}

}  // namespace moe
