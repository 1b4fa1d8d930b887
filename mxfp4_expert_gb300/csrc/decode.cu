// Single-launch decode path (T <= 4 tokens): one cooperative persistent kernel,
// one CTA per SM, so a layer call is a single launch with no host round trips
// and no idle HBM between stages.
//
// Every CTA walks a private sequence of "loads". Each load fills one slot of a
// shared-memory ring through 1-D bulk copies, and the CTA consumes the loads in
// order:
//
//   R   its slice of router rows             -> logits (global)     phase A
//   F   its slice of shared gate/up rows     -> h_sh (global)       phase A
//   SD  shared-down rows of its output tiles -> y accumulators      needs all h_sh
//   GU  its routed gate/up items             -> h blocks (global)   needs routing
//   DN  routed-down units of its output tiles -> y accumulators     needs all h blocks
//
// R, F and SD do not depend on routing and are requested at kernel start, so
// HBM is busy from the first cycle. After its R loads a CTA arrives at a
// counter barrier; it computes its F loads while the others catch up, then
// reads all logits and runs the top-k itself (every CTA derives the same
// routing, so no second exchange is needed), and requests its phase-B loads.
//
// A routed gate/up item is one 32-feature block of one active expert (four
// 16-row tiles, 87 KB for the Ling shape). The CTA that computes it holds the
// block's 32 values of h per token and writes them directly as e4m3 terms with
// one block exponent (the B operand of the down MMA), so no other CTA has to
// touch h. After its last item a CTA publishes with one release increment;
// before its down units it waits for all CTAs, then pulls every token's h
// terms into shared memory with one bulk copy. Down units accumulate in
// registers across experts and K-blocks; the cross-warp sum is taken once per
// output tile at the end. Each CTA owns whole 16-row output tiles, so y is
// written without a cross-CTA reduction. Gate/up items are handed out so that
// every CTA moves about the same number of bytes in phase B, counting its down
// and shared-down rows.
//
// Cross-call state (counters) lives at the start of the workspace and must be
// zero before the first call; the last CTA of a call resets it. Every wait is
// bounded (kSpinBudget); on timeout the kernel sets MOE_DEV_TIMEOUT and
// carries on.
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode.h"
#include "host_util.h"
#include "mma_tile.cuh"
#include "topk.cuh"

namespace moe {
namespace {

#ifdef MOE_DECODE_TRACE
// Debug builds only: per-CTA globaltimer stamps at phase boundaries.
constexpr int kTracePoints = 16;
__device__ unsigned long long g_trace[1024][kTracePoints];
__device__ __forceinline__ void trace(int point) {
  if (threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_trace[blockIdx.x][point] = t;
  }
}
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_put(int point, unsigned long long v) {
  if (threadIdx.x == 0) g_trace[blockIdx.x][point] = v;
}
#else
__device__ __forceinline__ void trace(int) {}
__device__ __forceinline__ unsigned long long gtime() { return 0; }
__device__ __forceinline__ void trace_put(int, unsigned long long) {}
#endif

constexpr int kWarps = 15;                  // compute warps
constexpr int kThreads = (kWarps + 1) * 32; // + one producer warp that issues the bulk copies
constexpr int kComputeThreads = kWarps * 32;
constexpr int kPairsMax = (kDecodeMaxT + 1) / 2;
constexpr int kRowsPerLoad = 8;   // max rows of a "few long rows" GEMV load (split-K over warps)
constexpr int kMaxKbPerWarp = 8;  // routed gate/up: d <= kWarps * 8 * 32 = 3840

// Barrier among the compute warps only (the producer warp never joins it).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory"); }
__device__ __forceinline__ bool csync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kComputeThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float dot8_bf16(uint4 w, uint4 x) {
  float s = bf16_lo(w.x) * bf16_lo(x.x);
  s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
  s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
  s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
  s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
  s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
  s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
  s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
  return s;
}
__device__ __forceinline__ float dot8_f32(uint4 w, const float* h) {
  const float4 a = *reinterpret_cast<const float4*>(h);
  const float4 b = *reinterpret_cast<const float4*>(h + 4);
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// bf16 rows (row-major, K elements each, in shared memory) times T bf16
// activation vectors (shared memory), split over all warps along K.
// out[r * kDecodeMaxT + t] (shared) receives the dot products. n <= kRowsPerLoad.
template <int T>
__device__ void gemv_bf16_rows(const uint8_t* rows, int n, int K, const __nv_bfloat16* xs,
                               float* red, float* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = K / 8;
  float acc[kRowsPerLoad][T];
#pragma unroll
  for (int r = 0; r < kRowsPerLoad; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t) acc[r][t] = 0.0f;
  for (int j = tid; j < chunks; j += kComputeThreads) {
    uint4 xv[T];
#pragma unroll
    for (int t = 0; t < T; ++t) xv[t] = reinterpret_cast<const uint4*>(xs + (size_t)t * K)[j];
#pragma unroll
    for (int r = 0; r < kRowsPerLoad; ++r) {
      if (r < n) {
        const uint4 wv = reinterpret_cast<const uint4*>(rows + (size_t)r * K * 2)[j];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[r][t] += dot8_bf16(wv, xv[t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerLoad; ++r) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      if (r < n) {
        const float v = warp_sum(acc[r][t]);
        if (lane == 0) red[(warp * kRowsPerLoad + r) * kDecodeMaxT + t] = v;
      }
    }
  }
  csync();
  if (tid < n * kDecodeMaxT) {
    const int r = tid / kDecodeMaxT, t = tid % kDecodeMaxT;
    float v = 0.0f;
    if (t < T)
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += red[(w * kRowsPerLoad + r) * kDecodeMaxT + t];
    out[tid] = v;
  }
  csync();
}

// Shared-memory carve-up (byte offsets), identical on host and device. The
// phase-A buffers (xs, xb, xe, hsh) and the phase-B h terms (hbs, hes) share
// one region: the former are dead once the down units start.
struct Smem {
  uint32_t ring, bars, ov, xs, xb, xe, hsh, hbs, hes, hblk, yacc, red, gout, sel_e, sel_w, act, act_n,
      act_slot, act_tok, first, misc, total;
};
__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline uint32_t he_stride(int I) { return align_up(uint32_t(I / kMxBlock), 8); }
__host__ __device__ inline Smem smem_plan(int T, int d, int I, int k, int stages, uint32_t slot_bytes) {
  Smem s{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = align_up(at, align);
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  s.ring = take(uint32_t(stages) * slot_bytes, 128);
  s.bars = take(8u * uint32_t(2 * stages + 3), 8);   // full[S], empty[S], h staging, routing, x
  // overlay: phase A layout
  const uint32_t xs_b = align_up(uint32_t(T) * d * 2, 16);
  const uint32_t xb_b = align_up(uint32_t(T) * (d / 32) * kActRowKbBytes, 16);
  const uint32_t xe_b = align_up(uint32_t(T) * (d / 32) * 2, 16);
  const uint32_t hsh_b = align_up(uint32_t(T) * I * 4, 16);
  const uint32_t a_bytes = xs_b + xb_b + xe_b + hsh_b;
  // overlay: phase B layout (h terms of every slot)
  const uint32_t slots = uint32_t(T) * k;
  const uint32_t hbs_b = align_up(slots * (I / 32) * kActRowKbBytes, 16);
  const uint32_t hes_b = align_up(slots * he_stride(I) * 2, 16);
  const uint32_t b_bytes = hbs_b + hes_b;
  s.ov = take(a_bytes > b_bytes ? a_bytes : b_bytes, 128);
  s.xs = s.ov;
  s.xb = s.xs + xs_b;
  s.xe = s.xb + xb_b;
  s.hsh = s.xe + xe_b;
  s.hbs = s.ov;
  s.hes = s.hbs + hbs_b;
  s.hblk = take(kDecodeMaxT * 32 * 4, 16);
  s.yacc = take(uint32_t(T) * kDecodeMaxTiles * 16 * 4, 16);
  const uint32_t red_mma = kWarps * kPairsMax * 32 * 2 * 4;
  const uint32_t red_gemv = kWarps * kRowsPerLoad * kDecodeMaxT * 4;
  const uint32_t red_dn = kWarps * kDecodeMaxT * 32 * 2 * 4;
  uint32_t red_b = red_mma > red_gemv ? red_mma : red_gemv;
  red_b = red_b > red_dn ? red_b : red_dn;
  s.red = take(red_b, 16);
  s.gout = take(kRowsPerLoad * kDecodeMaxT * 4, 16);
  s.sel_e = take(kDecodeMaxT * 32 * 4, 4);
  s.sel_w = take(kDecodeMaxT * 32 * 4, 4);
  s.act = take(kDecodeMaxT * 32 * 4, 4);
  s.act_n = take(kDecodeMaxT * 32 * 4, 4);
  s.act_slot = take(kDecodeMaxT * 32 * kDecodeMaxT * 4, 4);
  s.act_tok = take(kDecodeMaxT * 32 * kDecodeMaxT * 4, 4);
  s.first = take(kDecodeMaxT * 32 * 4, 4);
  s.misc = take(16 * 4, 8);
  s.total = at;
  return s;
}

// Per-CTA load sequence: [0,nR) router, [nR,bF) shared gate/up, [bF,bSD)
// shared down, [bSD,bGU) routed gate/up tiles (4 per item), [bGU,bDN) routed
// down loads (dnch units each).
struct Seq {
  int r0, r1, f0, f1, t0, ntl;
  int nR, nF, nSD;
  int rch, fch, sdch, dnch;
  int D, i0, i1, nDN;
  int bF, bSD, bGU, bDN;
};

template <int T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  trace(0);
  constexpr int kPairs = (T + 1) / 2;
  const int d = a.d, I = a.I, E = a.E, k = a.k;
  const int KBd = d / kMxBlock, KBi = I / kMxBlock, HES = int(he_stride(I));
  const int NTd = d / kTileRows;
  const int G = gridDim.x, c = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const Smem L = smem_plan(T, d, I, k, a.stages, a.slot_bytes);
  uint8_t* ring = sm + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + a.stages;
  uint64_t* hbar = empty + a.stages;
  uint64_t* rbar = hbar + 1;
  uint64_t* xbar = rbar + 1;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(sm + L.xs);
  uint8_t* xb = sm + L.xb;
  int16_t* xe = reinterpret_cast<int16_t*>(sm + L.xe);
  float* hsh = reinterpret_cast<float*>(sm + L.hsh);
  uint8_t* hbs = sm + L.hbs;
  int16_t* hes = reinterpret_cast<int16_t*>(sm + L.hes);
  float* hblk = reinterpret_cast<float*>(sm + L.hblk);
  float* yacc = reinterpret_cast<float*>(sm + L.yacc);
  float* red = reinterpret_cast<float*>(sm + L.red);
  float* gout = reinterpret_cast<float*>(sm + L.gout);
  int* sel_e = reinterpret_cast<int*>(sm + L.sel_e);
  float* sel_w = reinterpret_cast<float*>(sm + L.sel_w);
  int* act = reinterpret_cast<int*>(sm + L.act);
  int* act_n = reinterpret_cast<int*>(sm + L.act_n);
  int* act_slot = reinterpret_cast<int*>(sm + L.act_slot);
  int* act_tok = reinterpret_cast<int*>(sm + L.act_tok);   // token of each act_slot entry
  int* first = reinterpret_cast<int*>(sm + L.first);
  int* misc = reinterpret_cast<int*>(sm + L.misc);

  DecodeState* st = a.state;
  const uint32_t U_gu = uint32_t(KBd) * kUnitBytes, U_dn = uint32_t(KBi) * kUnitBytes;
  const uint32_t row_bytes = uint32_t(d) * 2, sdrow_bytes = uint32_t(I) * 2;
  const int ystride = kDecodeMaxTiles * kTileRows;

  Seq s;
  s.r0 = int((long long)c * E / G);
  s.r1 = int((long long)(c + 1) * E / G);
  s.f0 = a.has_shared ? int((long long)c * I / G) : 0;
  s.f1 = a.has_shared ? int((long long)(c + 1) * I / G) : 0;
  s.t0 = int((long long)c * NTd / G);
  s.ntl = int((long long)(c + 1) * NTd / G) - s.t0;
  s.rch = min(kRowsPerLoad, max(1, int(a.slot_bytes / row_bytes)));
  s.fch = min(kRowsPerLoad / 2, max(1, int(a.slot_bytes / (2 * row_bytes))));
  s.sdch = max(1, int(a.slot_bytes / sdrow_bytes));
  s.dnch = max(1, int(a.slot_bytes / U_dn));
  s.nR = (s.r1 - s.r0 + s.rch - 1) / s.rch;
  s.nF = (s.f1 - s.f0 + s.fch - 1) / s.fch;
  s.nSD = a.has_shared ? (s.ntl * kTileRows + s.sdch - 1) / s.sdch : 0;
  s.bF = s.nR + s.nF;
  s.bSD = s.bF + s.nSD;
  s.D = 0;
  s.i0 = s.i1 = 0;
  s.nDN = 0;
  s.bGU = s.bDN = s.bSD;

  // bulk-copy requests of load i into its ring slot (thread 0 only)
  auto issue = [&](int i) {
    const int slot = i % a.stages;
    uint8_t* dst = ring + (size_t)slot * a.slot_bytes;
    uint64_t* bar = &full[slot];
    if (i < s.nR) {
      const int r = s.r0 + i * s.rch, n = min(s.rch, s.r1 - r);
      mbar_arrive_expect_tx(bar, n * row_bytes);
      bulk_g2s(dst, a.router_w + (size_t)r * d, n * row_bytes, bar);
    } else if (i < s.bF) {
      const int f = s.f0 + (i - s.nR) * s.fch, n = min(s.fch, s.f1 - f);
      mbar_arrive_expect_tx(bar, 2 * n * row_bytes);
      bulk_g2s(dst, a.sh_gate + (size_t)f * d, n * row_bytes, bar);
      bulk_g2s(dst + (size_t)n * row_bytes, a.sh_up + (size_t)f * d, n * row_bytes, bar);
    } else if (i < s.bSD) {
      const int r = s.t0 * kTileRows + (i - s.bF) * s.sdch;
      const int n = min(s.sdch, (s.t0 + s.ntl) * kTileRows - r);
      mbar_arrive_expect_tx(bar, n * sdrow_bytes);
      bulk_g2s(dst, a.sh_down + (size_t)r * I, n * sdrow_bytes, bar);
    } else if (i < s.bGU) {
      const int j = i - s.bSD;
      const int item = s.i0 + j / 4, tile = (item % KBi) * 4 + (j % 4);
      const int e = act[item / KBi];
      mbar_arrive_expect_tx(bar, U_gu);
      bulk_g2s(dst, a.gate_up + (size_t)e * a.gu_mat + (size_t)tile * U_gu, U_gu, bar);
    } else {
      const int u0 = (i - s.bGU) * s.dnch, n = min(s.dnch, s.ntl * s.D - u0);
      mbar_arrive_expect_tx(bar, n * U_dn);
      for (int j = 0; j < n; ++j) {
        const int u = u0 + j, tl = u / s.D, ai = u % s.D;
        const int e = act[ai], tile = s.t0 + tl;
        bulk_g2s(dst + (size_t)j * U_dn, a.down + (size_t)e * a.dn_mat + (size_t)tile * U_dn, U_dn, bar);
      }
    }
  };

  if (tid == 0) {
    for (int i = 0; i < 2 * a.stages + 3; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
  }
  __syncthreads();   // the only full-CTA barrier: barriers initialised

  if (warp == kWarps) {
    // ---- producer warp: issues every bulk copy, in load order ----------------
    if (lane == 0) {
      // the activations first, so they are not queued behind the weights
      mbar_arrive_expect_tx(xbar, uint32_t(T) * d * 2);
      bulk_g2s(xs, a.x, uint32_t(T) * d * 2, xbar);
      int n_loads = s.bSD;
      for (int j = 0; j < n_loads || j == s.bSD; ++j) {
        if (j == s.bSD) {
          // phase B is known once the compute warps have routed
          if (!mbar_wait(rbar, 0u, a.status, 256)) break;
          s.D = misc[0];
          s.i0 = misc[1];
          s.i1 = misc[2] > misc[1] ? misc[2] : misc[1];
          s.nDN = (s.ntl * s.D + s.dnch - 1) / s.dnch;
          s.bGU = s.bSD + 4 * (s.i1 - s.i0);
          s.bDN = s.bGU + s.nDN;
          n_loads = s.bDN;
          if (j >= n_loads) break;
        }
        if (j >= a.stages && !mbar_wait(&empty[j % a.stages], uint32_t(j / a.stages - 1) & 1u, a.status, 256)) break;
        issue(j);
      }
#ifdef MOE_DECODE_TRACE
      g_trace[blockIdx.x][15] = gtime();
#endif
    }
    return;
  }

  for (int i = tid; i < T * ystride; i += kComputeThreads) yacc[i] = 0.0f;
  mbar_wait(xbar, 0u, a.status);   // bf16 activations for the CUDA-core GEMVs
  csync();
  trace(1);
  if (tid == 0) {
    if (s.nR == 0) {
      __threadfence();
      atomicAdd(&st->bar, 1ull);
    }
    if (s.nF == 0) {
      __threadfence();
      atomicAdd(&st->shcnt, 1u);
    }
  }

  // per-lane down accumulators of the current output tile: [token][row g / row g+8]
  float dacc[T][2];
#pragma unroll
  for (int t = 0; t < T; ++t) dacc[t][0] = dacc[t][1] = 0.0f;
  int dn_tile = -1;
  // cross-warp sum of the down accumulators into y for output tile tl; the
  // four lanes of a quad hold the same two rows (different columns/slots)
  auto flush_tile = [&](int tl) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      red[((warp * kDecodeMaxT + t) * 32 + lane) * 2 + 0] = dacc[t][0];
      red[((warp * kDecodeMaxT + t) * 32 + lane) * 2 + 1] = dacc[t][1];
      dacc[t][0] = dacc[t][1] = 0.0f;
    }
    csync();
    if (tid < T * kTileRows) {
      const int t = tid / kTileRows, r = tid % kTileRows;
      const int gg = r & 7, half = r >> 3;
      float v = 0.0f;
      for (int w = 0; w < kWarps; ++w)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) v += red[((w * kDecodeMaxT + t) * 32 + gg * 4 + qq) * 2 + half];
      yacc[t * ystride + tl * kTileRows + r] += v;
    }
    csync();
  };

  int total = s.bSD;
  unsigned long long t_wait = 0, t_gu = 0;   // debug builds: time waiting for loads / in gate-up tiles
  for (int i = 0;; ++i) {
    if (i == s.bF) {
      // ---- routing: every CTA has written its router rows -------------------
      trace(3);
      if (tid == 0) wait_geq_u64(&st->bar, (unsigned long long)G, a.status);
      csync();
      trace(4);
      if (warp < T) {
        int e_sel;
        float w_sel;
        const float* brow = a.bias ? a.bias + (size_t)warp * a.bias_stride : nullptr;
        warp_topk<16, true>(a.logits + (size_t)warp * E, brow, E, k, lane, &e_sel, &w_sel);
        if (lane < k) {
          sel_e[warp * k + lane] = e_sel;
          sel_w[warp * k + lane] = w_sel;
          if (c == 0) {
            if (a.idx_out) a.idx_out[warp * k + lane] = e_sel;
            if (a.w_out) a.w_out[warp * k + lane] = w_sel;
          }
        }
      } else {
        // meanwhile the other warps turn the activations into e4m3 terms
        for (int u = warp - T; u < T * KBd; u += kWarps - T) {
          const float v = __bfloat162float(xs[(size_t)u * kMxBlock + lane]);
          const int ex = split_block(v, lane, xb + (size_t)u * kActRowKbBytes);
          if (lane == 0) xe[u] = int16_t(ex);
        }
      }
      csync();
      trace(11);
      // active experts ascending; each with its slots (slot = t*k + j) in token order
      const int n = T * k;
      if (tid < n) {
        const int e = sel_e[tid];
        int f = 1;
        for (int j = 0; j < tid; ++j) f &= sel_e[j] != e ? 1 : 0;
        first[tid] = f;
      }
      csync();
      if (tid < n) {
        const int e = sel_e[tid];
        int rank = 0, pos = 0, cnt = 0;
        for (int j = 0; j < n; ++j) {
          const int ej = sel_e[j];
          rank += (first[j] && ej < e) ? 1 : 0;
          pos += (j < tid && ej == e) ? 1 : 0;
          cnt += ej == e ? 1 : 0;
        }
        act_slot[rank * kDecodeMaxT + pos] = tid;
        act_tok[rank * kDecodeMaxT + pos] = tid / k;
        if (first[tid]) {
          act[rank] = e;
          act_n[rank] = cnt;
        }
      }
      if (tid == 0) {
        int D = 0;
        for (int j = 0; j < n; ++j) D += first[j];
        // gate/up items (32-feature blocks): contiguous ranges, balanced by bytes
        // together with each CTA's down units and shared-down rows. W(c) is the
        // cumulative budget left for items before CTA c (non-decreasing).
        const int n_items = D * KBi;
        const float U = 4.0f * float(U_gu);
        const float DT = float(D) * float(U_dn) + (a.has_shared ? float(kTileRows) * float(sdrow_bytes) : 0.0f);
        const float target = (float(n_items) * U + float(NTd) * DT) / float(G);
        const int qt = NTd / G;
        const float w0 = fmaxf(0.0f, target - DT * float(qt)), w1 = fmaxf(0.0f, target - DT * float(qt + 1));
        auto W = [&](int cc) {
          const int big = (cc * NTd) / G - cc * qt;
          return float(cc - big) * w0 + float(big) * w1;
        };
        const float WG = W(G);
        auto cut = [&](int cc) {
          if (cc >= G) return n_items;
          if (WG <= 0.0f) return 0;
          const int v = int(floorf(float(n_items) * (W(cc) / WG) + 0.5f));
          return v < 0 ? 0 : (v > n_items ? n_items : v);
        };
        misc[0] = D;
        misc[1] = cut(c);
        misc[2] = cut(c + 1);
      }
      csync();
      s.D = misc[0];
      s.i0 = misc[1];
      s.i1 = misc[2] > misc[1] ? misc[2] : misc[1];
      s.nDN = (s.ntl * s.D + s.dnch - 1) / s.dnch;
      s.bGU = s.bSD + 4 * (s.i1 - s.i0);
      s.bDN = s.bGU + s.nDN;
      total = s.bDN;
      if (tid == 0) mbar_arrive(rbar);   // hands phase B to the producer warp
      trace(5);
      if (s.nSD > 0) {
        // shared down needs every CTA's slice of h_sh
        if (tid == 0) wait_geq_u32(&st->shcnt, uint32_t(G), a.status);
        csync();
        for (int j = tid; j < T * I; j += kComputeThreads) hsh[j] = __ldcg(a.h_sh + j);
      }
      csync();
      trace(6);
    }
    if (i == s.bSD) trace(7);
    if (i == s.bGU) {
      // ---- all h blocks of every CTA: publish mine, wait, stage them ----------
      trace(8);
      if (tid == 0) {
        red_release_add(&st->gudone, 1u);
        wait_geq_u32(&st->gudone, uint32_t(G), a.status);
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint32_t hb_bytes = uint32_t(T * k) * KBi * kActRowKbBytes;
        const uint32_t he_bytes = uint32_t(T * k) * HES * 2;
        mbar_arrive_expect_tx(hbar, hb_bytes + he_bytes);
        bulk_g2s(hbs, a.hB, hb_bytes, hbar);
        bulk_g2s(hes, a.hE, he_bytes, hbar);
      }
      csync();
      mbar_wait(hbar, 0u, a.status);
      csync();
      trace(9);
    }
    if (i >= total) break;

    const int slot = i % a.stages;
    const uint8_t* buf = ring + (size_t)slot * a.slot_bytes;
    const unsigned long long tw0 = gtime();
    const bool ok = csync_and(mbar_wait(&full[slot], uint32_t(i / a.stages) & 1u, a.status));
    const unsigned long long tw1 = gtime();
    t_wait += tw1 - tw0;
    if (ok && i < s.nR) {
      // ---- router rows -> logits ----------------------------------------------
      const int r = s.r0 + i * s.rch, n = min(s.rch, s.r1 - r);
      gemv_bf16_rows<T>(buf, n, d, xs, red, gout);
      if (tid < n * kDecodeMaxT && (tid % kDecodeMaxT) < T)
        a.logits[(size_t)(tid % kDecodeMaxT) * E + r + tid / kDecodeMaxT] = gout[tid];
    } else if (ok && i < s.bF) {
      // ---- shared gate/up rows -> h_sh -----------------------------------------
      const int f = s.f0 + (i - s.nR) * s.fch, n = min(s.fch, s.f1 - f);
      gemv_bf16_rows<T>(buf, 2 * n, d, xs, red, gout);   // rows 0..n-1 gate, n..2n-1 up
      if (tid < n * kDecodeMaxT && (tid % kDecodeMaxT) < T) {
        const int ff = tid / kDecodeMaxT, t = tid % kDecodeMaxT;
        a.h_sh[(size_t)t * I + f + ff] = silu_f(gout[ff * kDecodeMaxT + t]) * gout[(n + ff) * kDecodeMaxT + t];
      }
    } else if (ok && i < s.bSD) {
      // ---- shared down rows of my tiles -> y accumulators (warp per row) -------
      const int r = s.t0 * kTileRows + (i - s.bF) * s.sdch;
      const int n = min(s.sdch, (s.t0 + s.ntl) * kTileRows - r);
      for (int rr = warp; rr < n; rr += kWarps) {
        const uint4* wrow = reinterpret_cast<const uint4*>(buf + (size_t)rr * sdrow_bytes);
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.0f;
        for (int j = lane; j < I / 8; j += 32) {
          const uint4 wv = wrow[j];
#pragma unroll
          for (int t = 0; t < T; ++t) acc[t] += dot8_f32(wv, hsh + (size_t)t * I + j * 8);
        }
        const int row_local = r + rr - s.t0 * kTileRows;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float v = warp_sum(acc[t]);
          if (lane == 0) yacc[t * ystride + row_local] = v;
        }
      }
    } else if (ok && i < s.bGU) {
      // ---- routed gate/up tile (one of the 4 of a 32-feature item) -------------
      const int j = i - s.bSD, sub = j % 4;
      const int item = s.i0 + j / 4;
      const int ai = item / KBi, fb = item % KBi;
      const int nt = act_n[ai];
      const int* slots = act_slot + ai * kDecodeMaxT;
      const int* toks = act_tok + ai * kDecodeMaxT;
      // lane-invariant-over-K operand offsets: B rows (token, term column), exponent rows
      int boff[kPairs], eoff[kPairs];
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        const int sb = 2 * p + (g >> 2), sc = 2 * p + (q >> 1);
        boff[p] = (sb < nt && (g & 3) < kActTerms) ? toks[sb] * KBd * kActRowKbBytes + (g & 3) * 32 + q * 8 : -1;
        eoff[p] = sc < nt ? toks[sc] * KBd : -1;
      }
      float acc[kPairs][2];
#pragma unroll
      for (int p = 0; p < kPairs; ++p) acc[p][0] = acc[p][1] = 0.0f;
#pragma unroll
      for (int jj = 0; jj < kMaxKbPerWarp; ++jj) {
        const int kb = warp + jj * kWarps;
        if (kb < KBd) {
          const UnitFrag f = load_unit(buf + (size_t)kb * kUnitBytes, lane);
#pragma unroll
          for (int p = 0; p < kPairs; ++p) {
            if (2 * p < nt) {
              const uint2 bv = boff[p] >= 0 ? *reinterpret_cast<const uint2*>(xb + boff[p] + kb * kActRowKbBytes)
                                            : make_uint2(0u, 0u);
              const int ex = eoff[p] >= 0 ? int(xe[eoff[p] + kb]) : int(kActZeroExp);
              unit_mma(f, bv, ex, acc[p][0], acc[p][1]);
            }
          }
        }
      }
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        red[((warp * kPairsMax + p) * 32 + lane) * 2 + 0] = acc[p][0];
        red[((warp * kPairsMax + p) * 32 + lane) * 2 + 1] = acc[p][1];
      }
      csync();
      if (warp == 0) {
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          if (2 * p < nt) {
            float v0 = 0.0f, v1 = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
              v0 += red[((w * kPairsMax + p) * 32 + lane) * 2 + 0];
              v1 += red[((w * kPairsMax + p) * 32 + lane) * 2 + 1];
            }
            v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
            v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
            const int sc = 2 * p + (q >> 1);
            if ((q & 1) == 0 && sc < nt) hblk[sc * 32 + sub * 8 + g] = silu_f(v0) * v1;
          }
        }
      }
      csync();
      if (sub == 3 && warp < nt) {
        // the item's 32 features are complete: write them as e4m3 terms
        const int sl = slots[warp];
        const int ex = split_block(hblk[warp * 32 + lane], lane, a.hB + ((size_t)sl * KBi + fb) * kActRowKbBytes);
        if (lane == 0) a.hE[(size_t)sl * HES + fb] = int16_t(ex);
      }
    } else if (ok) {
      // ---- routed down units of my tiles -> per-lane accumulators --------------
      const int u0 = (i - s.bGU) * s.dnch, n = min(s.dnch, s.ntl * s.D - u0);
      for (int j = 0; j < n; ++j) {
        const int u = u0 + j, tl = u / s.D, ai = u % s.D;
        if (tl != dn_tile) {
          if (dn_tile >= 0) flush_tile(dn_tile);
  trace_put(13, t_wait);
  trace_put(14, t_gu);
          dn_tile = tl;
        }
        const int nt = act_n[ai];
        const int* slots = act_slot + ai * kDecodeMaxT;
        const int* toks = act_tok + ai * kDecodeMaxT;
        const uint8_t* ubuf = buf + (size_t)j * U_dn;
        int boff[kPairs], eoff[kPairs], tok[kPairs];
        float wgt[kPairs];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const int sb = 2 * p + (g >> 2), sc = 2 * p + (q >> 1);
          boff[p] = (sb < nt && (g & 3) < kActTerms) ? slots[sb] * KBi * kActRowKbBytes + (g & 3) * 32 + q * 8 : -1;
          eoff[p] = sc < nt ? slots[sc] * HES : -1;
          tok[p] = sc < nt ? toks[sc] : -1;
          wgt[p] = sc < nt ? sel_w[slots[sc]] : 0.0f;
        }
        for (int kb = warp; kb < KBi; kb += kWarps) {
          const UnitFrag f = load_unit(ubuf + (size_t)kb * kUnitBytes, lane);
#pragma unroll
          for (int p = 0; p < kPairs; ++p) {
            if (2 * p < nt) {
              const uint2 bv = boff[p] >= 0 ? *reinterpret_cast<const uint2*>(hbs + boff[p] + kb * kActRowKbBytes)
                                            : make_uint2(0u, 0u);
              float d4[4];
              mma_e4m3(d4, f.a0, f.a1, f.a2, f.a3, bv.x, bv.y);
              if (eoff[p] >= 0) {
                const int ex = int(hes[eoff[p] + kb]);
                const float vlo = (d4[0] + d4[1]) * (wgt[p] * block_factor(f.s_lo, ex));
                const float vhi = (d4[2] + d4[3]) * (wgt[p] * block_factor(f.s_hi, ex));
#pragma unroll
                for (int tt = 0; tt < T; ++tt) {
                  if (tt == tok[p]) {
                    dacc[tt][0] += vlo;
                    dacc[tt][1] += vhi;
                  }
                }
              }
            }
          }
        }
      }
    }
    if (i >= s.bSD && i < s.bGU) t_gu += gtime() - tw1;
    // after the last router load: this CTA's logits are written
    if (i == s.nR - 1) trace(2);
    if (i == s.nR - 1 && tid == 0) {
      __threadfence();
      atomicAdd(&st->bar, 1ull);
    }
    if (s.nF > 0 && i == s.bF - 1 && tid == 0) {
      __threadfence();
      atomicAdd(&st->shcnt, 1u);
    }
    csync();
    if (tid == 0) mbar_arrive(&empty[slot]);   // slot free for load i + stages
  }
  trace(12);

  if (dn_tile >= 0) flush_tile(dn_tile);
  trace_put(13, t_wait);
  trace_put(14, t_gu);

  // y rows of my tiles
  for (int j = tid; j < T * s.ntl * kTileRows; j += kComputeThreads) {
    const int t = j / (s.ntl * kTileRows), r = j % (s.ntl * kTileRows);
    a.y[(size_t)t * d + s.t0 * kTileRows + r] = __float2bfloat16_rn(yacc[t * ystride + r]);
  }
  csync();
  trace(10);
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&st->done, 1u);
    if (old % uint32_t(G) == uint32_t(G) - 1u) {
      // last CTA of this call: every CTA is past every wait of this call
      st->bar = 0ull;
      st->shcnt = 0u;
      st->gudone = 0u;
      __threadfence();
    }
  }
}

}  // namespace

#ifdef MOE_DECODE_TRACE
int decode_trace_copy(unsigned long long* host, int n_cta) {
  MOE_CUDA_TRY(cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * kTracePoints * n_cta));
  return MOE_OK;
}
#endif

size_t decode_state_bytes(int E, int I) {
  (void)E;
  (void)I;
  return (size_t)kDecodeStateWords * 4;
}

uint32_t decode_he_stride(int I) { return he_stride(I); }

int decode_plan(const DecodeArgs& a, const DeviceInfo& di, int* stages, uint32_t* slot_bytes,
                uint32_t* smem_bytes) {
  if (a.T < 1 || a.T > kDecodeMaxT) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.d % 32 || a.I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.k < 1 || a.k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.E > 512 || a.d > kWarps * kMaxKbPerWarp * kMxBlock) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int NTd = a.d / kTileRows;
  if (di.sm_count < 1 || (NTd + di.sm_count - 1) / di.sm_count > kDecodeMaxTiles) return MOE_ERR_UNSUPPORTED_SHAPE;
  uint32_t sb = uint32_t(a.d / kMxBlock) * kUnitBytes;   // one routed gate/up tile
  const uint32_t cands[4] = {uint32_t(2 * a.d), uint32_t(4 * a.d), uint32_t(2 * a.I),
                             uint32_t(a.I / kMxBlock) * kUnitBytes};
  for (uint32_t v : cands) sb = sb > v ? sb : v;         // router row, shared feature, shared-down row, down unit
  sb = align_up(sb, 128);
  const Smem fixed = smem_plan(a.T, a.d, a.I, a.k, 0, sb);
  const size_t budget = di.smem_optin > fixed.total + 1024 ? di.smem_optin - fixed.total - 1024 : 0;
  int S = int(budget / (sb + 8));
  if (S > kDecodeMaxStages) S = kDecodeMaxStages;
  if (S < 3) return MOE_ERR_UNSUPPORTED_SHAPE;
  *stages = S;
  *slot_bytes = sb;
  *smem_bytes = smem_plan(a.T, a.d, a.I, a.k, S, sb).total;
  return MOE_OK;
}

template <int T>
int launch_decode_t(DecodeArgs a, uint32_t smem, const DeviceInfo& di, cudaStream_t s) {
  MOE_CUDA_TRY(cudaFuncSetAttribute(decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  int per_sm = 0;
  MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T>, kThreads, smem));
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(di.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, decode_kernel<T>, a));
  return MOE_OK;
}

int launch_decode(DecodeArgs a, const DeviceInfo& di, cudaStream_t s) {
  uint32_t smem = 0;
  int st = decode_plan(a, di, &a.stages, &a.slot_bytes, &smem);
  if (st != MOE_OK) return st;
  switch (a.T) {
    case 1: return launch_decode_t<1>(a, smem, di, s);
    case 2: return launch_decode_t<2>(a, smem, di, s);
    case 3: return launch_decode_t<3>(a, smem, di, s);
    default: return launch_decode_t<4>(a, smem, di, s);
  }
}

}  // namespace moe
