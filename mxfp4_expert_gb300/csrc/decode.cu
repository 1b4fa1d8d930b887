// Single-launch decode path (T <= 4 tokens): the whole layer in one kernel
// launch, one CTA per SM, 32 warps per CTA. The layer is the mixture-of-
// experts block of page "3 ways to speed up MoE inference on NVIDIA DGX
// Spark": 512 routed experts, top-8, one shared expert (§2), expert
// intermediate size 768 (§3); T = 1 is the single-token decode, T = 4 the
// verify step of the 4-token speculative decoding in §5.
//
// Phases of one CTA c of G:
//   0. griddepcontrol.launch_dependents, then L2 prefetch of this CTA's
//      router rows, shared gate/up rows and shared-down rows (routing-
//      independent; one prefetch per warp), then griddepcontrol.wait: under
//      programmatic dependent launch the next layer's prefetches overlap the
//      end of the previous one, and nothing written by the previous kernel is
//      read before the wait.
//   1. x -> shared memory; router rows [c E/G, (c+1) E/G) and shared gate/up
//      features [c I/G, (c+1) I/G), one bf16 row per warp (16-byte loads of
//      the whole row in flight, fp32 FMAs); logits and h_sh to global memory,
//      then one release increment.
//   2. x -> 3 e4m3 terms per 32-block (B operand of the routed MMAs, in the
//      K order of the A fragments) while the other CTAs finish; wait for
//      every CTA's logits; top-k in every CTA (the best k of each 32-expert
//      chunk on all warps, then a k-way merge per token). The selected
//      experts' gate/up matrices go into L2 at once, cut into G slices (one
//      per CTA). The active experts with their slots (one warp, match_any);
//      this CTA's contiguous range of gate/up tiles, balanced by bytes against
//      its down and shared-down work; the first round of down items.
//   3. Routed gate/up: items (16-row tile, 8 units of 272 B = 16 rows x 32 K
//      of E2M1 codes + E8M0 scales), item j on warp j % 32. Each warp keeps 1-2
//      items in flight, copied with cp.async into its own shared-memory
//      buffers, and multiplies them on the e4m3 warp MMA (m16n8k32) against
//      the x terms. The warp that finishes a tile's last item adds the tile's
//      partials in K order, applies SwiGLU and writes the tile's 8 features of
//      h as 2 e4m3 terms per feature with one factor per 8 features (routing
//      weight folded in); then (3-4 tokens) one L2 prefetch per active
//      expert's down units of this CTA's output tiles, the first down items'
//      copies, and one release increment per CTA.
//   4. Shared down rows of this CTA's 16-row output tiles (every CTA's h_sh is
//      in since the routing barrier), fp32 FMAs, while the first down items are
//      already being copied (cp.async, from L2) into the warps' buffers.
//   5. Routed down: after every CTA's h is in, the h terms of all slots go to
//      shared memory; items (output tile, active expert, up to 8 units, sized
//      so every warp gets one) into per-item partials, added in a fixed order
//      (one warp per output, a fixed tree) into y (bf16). Each CTA owns whole
//      output tiles, so y needs no cross-CTA reduction.
//
// The counters live at the head of the workspace and must be zero before the
// first call; the last CTA of a call resets them. Every wait is bounded
// (kSpinBudget); on timeout the kernel sets MOE_DEV_TIMEOUT and carries on, so
// it always terminates. Results are deterministic: every sum is taken in a
// fixed order.
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode.h"
#include "host_util.h"
#include "mma_tile.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kWarps = 32;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 8;                // MXFP4 units a warp loads together
constexpr int kRowVec = 10;          // 16-byte vectors of a bf16 row a lane loads together
constexpr int kMaxGuItems = 96;      // gate/up (tile, K-range) items per round
// items a warp keeps in flight (cp.async into its own shared-memory buffers):
// 2 for one or two tokens, 1 when the activations need more shared memory
__host__ __device__ constexpr int stage_items(int T) { return T <= 2 ? 2 : 1; }
constexpr uint32_t kItemBytes = kU * kUnitBytes;   // one item: kU units of a 16-row tile
constexpr int kMaxDnItems = 64;      // down (tile, expert, K-range) items per round
constexpr int kMergeChunks = 16;     // top-k: E <= 16 chunks of 32 experts
constexpr int kHTermBytes = 64;      // h of one (slot, K-block): 2 e4m3 terms x 32 features
constexpr int kHGroups = 4;          // 8-feature groups per K-block, one factor each
constexpr int kYStride = kDecodeMaxTiles * kTileRows;   // y accumulator row stride (per token)

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
// L2 prefetch of [p, p + bytes) (16-byte aligned, multiple of 16) in 32 KB pieces.
__device__ __noinline__ void prefetch_range(const void* p, uint32_t bytes) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  for (uint32_t o = 0; o < bytes; o += 32768u) prefetch_l2(b + o, min(32768u, bytes - o));
}

// 16-byte asynchronous global -> shared copy through L2 (no L1 allocation).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Weight scale bytes (row g in the low byte, row g+8 in the high byte) ->
// 2^(s-127) as fp32 (s = 0 gives 0).
__device__ __forceinline__ float scale_lo(uint32_t sc16) { return __uint_as_float((sc16 << 23) & 0x7F800000u); }
__device__ __forceinline__ float scale_hi(uint32_t sc16) { return __uint_as_float((sc16 << 15) & 0x7F800000u); }

// Factor that turns an MMA result over one (weight block, activation block)
// into its value, apart from the weight scale: weights were decoded as 2^-6 x
// the E2M1 value and the activation block stored as terms x 2^-e, so the
// factor is w x 2^(e+6) (0 for an all-zero block).
__device__ __forceinline__ float act_factor(int e, float w) { return e == kActZeroExp ? 0.0f : scale2(w, e + 6); }

// Shared-memory carve-up (byte offsets), identical on host and device.
// Region ov holds x, its e4m3 terms and factors (phases 1-3) and later the h
// terms of every slot (phase 5); region cg holds the gate/up partials.
struct Smem {
  uint32_t ov, xs, xb, xfa, hbs, hfa, gpart, rpart, hsh, dpart, yacc, sel_e, sel_w, act, act_n, act_slot, act_tok,
      tcnt, gtab, dtab, misc, wbuf, total;
};
__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int max_row_items(int E, int I, int G) { return ceil_div(E, G) + 2 * ceil_div(I, G); }
__host__ __device__ inline Smem smem_plan(int T, int d, int I, int E, int k, int G) {
  Smem s{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = align_up(at, align);
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  const uint32_t KBd = uint32_t(d / kMxBlock), KBi = uint32_t(I / kMxBlock), slots = uint32_t(T * k);
  const uint32_t pairs = uint32_t((T + 1) / 2);
  const uint32_t xs_b = align_up(uint32_t(T) * d * 2, 16);
  const uint32_t xb_b = align_up(uint32_t(T) * KBd * kActRowKbBytes, 16);
  const uint32_t xfa_b = align_up(uint32_t(T) * KBd * 4, 16);
  const uint32_t hbs_b = align_up(slots * KBi * kHTermBytes, 16);
  const uint32_t hfa_b = align_up(slots * KBi * kHGroups * 4, 16);
  const uint32_t a_b = xs_b + xb_b + xfa_b, b_b = hbs_b + hfa_b;
  s.ov = take(a_b > b_b ? a_b : b_b, 128);
  s.xs = s.ov;
  s.xb = s.xs + xs_b;
  s.xfa = s.xb + xb_b;
  s.hbs = s.ov;
  s.hfa = s.hbs + hbs_b;
  s.gpart = take(uint32_t(kMaxGuItems) * pairs * 32u * 4u, 16);
  s.rpart = take(uint32_t(max_row_items(E, I, G)) * T * 4u, 16);
  s.hsh = take(align_up(uint32_t(T) * I * 4, 16), 16);
  s.dpart = take(uint32_t(kMaxDnItems) * T * kTileRows * 4u, 16);
  s.yacc = take(uint32_t(T) * kYStride * 4u, 16);
  s.sel_e = take(kDecodeMaxT * 32 * 4, 4);
  s.sel_w = take(kDecodeMaxT * 32 * 4, 4);
  s.act = take(kDecodeMaxT * 32 * 4, 4);
  s.act_n = take(kDecodeMaxT * 32 * 4, 4);
  s.act_slot = take(kDecodeMaxT * 32 * kDecodeMaxT * 4, 4);
  s.act_tok = take(kDecodeMaxT * 32 * kDecodeMaxT * 4, 4);
  s.tcnt = take(kMaxGuItems * 4, 4);
  s.gtab = take(kMaxGuItems * 8, 8);
  s.dtab = take(kMaxDnItems * 8, 8);
  s.misc = take(16 * 4, 8);
  s.wbuf = take(uint32_t(kWarps * stage_items(T)) * kItemBytes, 128);
  s.total = at;
  return s;
}
template <int T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a, Smem L) {
  extern __shared__ __align__(128) uint8_t sm[];
  constexpr int kPairs = (T + 1) / 2;
  constexpr int kStageItems = stage_items(T);
  const int d = a.d, I = a.I, E = a.E, k = a.k;
  const int KBd = d / kMxBlock, KBi = I / kMxBlock;
  const int NTd = d / kTileRows, NTg = 2 * I / kTileRows;
  const int G = gridDim.x, c = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int r0 = c * E / G, r1 = (c + 1) * E / G;
  const int f0 = a.has_shared ? c * I / G : 0, f1 = a.has_shared ? (c + 1) * I / G : 0;
  const int t0 = c * NTd / G, ntl = (c + 1) * NTd / G - t0;
  const uint32_t row_bytes = uint32_t(d) * 2, sdrow_bytes = uint32_t(I) * 2;
  const uint32_t U_gu = uint32_t(KBd) * kUnitBytes, U_dn = uint32_t(KBi) * kUnitBytes;

  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(sm + L.xs);
  uint8_t* xb = sm + L.xb;
  float* xfa = reinterpret_cast<float*>(sm + L.xfa);
  uint8_t* hbs = sm + L.hbs;
  float* hfa = reinterpret_cast<float*>(sm + L.hfa);
  float* gpart = reinterpret_cast<float*>(sm + L.gpart);
  float* rpart = reinterpret_cast<float*>(sm + L.rpart);
  float* hsh = reinterpret_cast<float*>(sm + L.hsh);
  float* dpart = reinterpret_cast<float*>(sm + L.dpart);
  float* yacc = reinterpret_cast<float*>(sm + L.yacc);
  int* sel_e = reinterpret_cast<int*>(sm + L.sel_e);
  float* sel_w = reinterpret_cast<float*>(sm + L.sel_w);
  int* act = reinterpret_cast<int*>(sm + L.act);
  int* act_n = reinterpret_cast<int*>(sm + L.act_n);
  int* act_slot = reinterpret_cast<int*>(sm + L.act_slot);
  int* act_tok = reinterpret_cast<int*>(sm + L.act_tok);
  int* tcnt = reinterpret_cast<int*>(sm + L.tcnt);
  int2* gtab = reinterpret_cast<int2*>(sm + L.gtab);
  uint8_t* wb = sm + L.wbuf + (size_t)warp * kStageItems * kItemBytes;   // this warp's item buffers
  int2* dtab = reinterpret_cast<int2*>(sm + L.dtab);
  int* misc = reinterpret_cast<int*>(sm + L.misc);

  DecodeState* st = a.state;

  // ---- 0. next launch, routing-independent prefetch, previous kernel ---------
  // one prefetch per warp (each bulk prefetch takes a while to issue)
  if (lane == 0) {
    if (warp == 0) {
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      if (r1 > r0) prefetch_range(a.router_w + (size_t)r0 * d, uint32_t(r1 - r0) * row_bytes);
    } else if (warp == 1 && f1 > f0) {
      prefetch_range(a.sh_gate + (size_t)f0 * d, uint32_t(f1 - f0) * row_bytes);
    } else if (warp == 2 && f1 > f0) {
      prefetch_range(a.sh_up + (size_t)f0 * d, uint32_t(f1 - f0) * row_bytes);
    } else if (warp == 3 && a.has_shared && ntl > 0) {
      prefetch_range(a.sh_down + (size_t)t0 * kTileRows * I, uint32_t(ntl * kTileRows) * sdrow_bytes);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");



  // ---- 1. x; router rows and shared gate/up rows ------------------------------
  #pragma unroll 1
  for (int j = tid; j < T * d / 8; j += kThreads)
    reinterpret_cast<uint4*>(xs)[j] = __ldg(reinterpret_cast<const uint4*>(a.x) + j);
  #pragma unroll 1
  for (int j = tid; j < T * kYStride; j += kThreads) yacc[j] = 0.0f;
  __syncthreads();
  const int nr = r1 - r0, nf = f1 - f0, n_rows = nr + 2 * nf;
  auto row_ptr = [&](int it) -> const uint4* {
    if (it < nr) return reinterpret_cast<const uint4*>(a.router_w + (size_t)(r0 + it) * d);
    const int j = it - nr;
    return reinterpret_cast<const uint4*>(((j & 1) ? a.sh_up : a.sh_gate) + (size_t)(f0 + (j >> 1)) * d);
  };
  {
    const int n8 = d / 8;
    const uint4* x4 = reinterpret_cast<const uint4*>(xs);
    uint4 w[kRowVec];
    for (int it = warp; it < n_rows; it += kWarps) {
      const uint4* r4 = row_ptr(it);
      float acc[T];
#pragma unroll
      for (int t = 0; t < T; ++t) acc[t] = 0.0f;
      for (int j0 = 0; j0 < n8; j0 += 32 * kRowVec) {
#pragma unroll
        for (int m = 0; m < kRowVec; ++m) {
          const int j = j0 + lane + 32 * m;
          w[m] = j < n8 ? ldg_nc_stream_u4(r4 + j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < kRowVec; ++m) {
          const int j = j0 + lane + 32 * m;
          if (j < n8) {
#pragma unroll
            for (int t = 0; t < T; ++t) acc[t] += dot8_bf16(w[m], x4[t * n8 + j]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) rpart[it * T + t] = v;
      }
    }
  }
  __syncthreads();
  // logits and h_sh of this CTA -> global memory, then one release increment
  // (by the last warp, so warp 0 starts polling at once)
  #pragma unroll 1
  for (int j = tid; j < nr * T; j += kThreads) {
    const int t = j / nr, r = j - t * nr;
    a.logits[(size_t)t * E + r0 + r] = rpart[r * T + t];
  }
  #pragma unroll 1
  for (int j = tid; j < nf * T; j += kThreads) {
    const int t = j / nf, f = j - t * nf;
    const float gv = rpart[(nr + 2 * f) * T + t], uv = rpart[(nr + 2 * f + 1) * T + t];
    a.h_sh[(size_t)t * I + f0 + f] = silu_f(gv) * uv;
  }
  __syncthreads();
  if (warp == kWarps - 1 && lane == 0) red_release_add(&st->routed, 1u);

  // ---- 2. x -> e4m3 terms (B operand of the routed gate/up MMAs) while the
  // other CTAs finish their rows; then every CTA's logits (and h_sh) are in
#pragma unroll 1
  for (int u = warp; u < T * KBd; u += kWarps) {
    const float v = __bfloat162float(xs[(size_t)u * kMxBlock + lane]);
    const int ex = split_block(v, lane, xb + (size_t)u * kActRowKbBytes);
    if (lane == 0) xfa[u] = act_factor(ex, 1.0f);
  }
  if (tid == 0) wait_geq_u32(&st->routed, uint32_t(G), a.status);
  __syncthreads();
  {
    // top-k, stage 1 (all warps): the best min(k, 32) of every (token,
    // 32-expert chunk), by key descending, equal keys -> lower expert index
    const int nch = (E + 31) / 32, kk = k < 32 ? k : 32;
    uint32_t* ckey = reinterpret_cast<uint32_t*>(sm + L.gpart);
    uint32_t* cidx = ckey + T * nch * kk;
#pragma unroll 1
    for (int task = warp; task < T * nch; task += kWarps) {
      const int t = task / nch, e = (task - t * nch) * 32 + lane;
      uint32_t key = 0u;
      if (e < E) {
        float v = __ldcg(a.logits + (size_t)t * E + e);
        if (a.bias) v = __fadd_rn(v, a.bias[(size_t)t * a.bias_stride + e]);
        key = rank_key(v);
      }
#pragma unroll 1
      for (int r = 0; r < kk; ++r) {
        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, key);
        const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, (mx != 0u && key == mx) ? uint32_t(e) : 0xFFFFFFFFu);
        if (lane == 0) {
          ckey[task * kk + r] = mx;
          cidx[task * kk + r] = win;
        }
        if (uint32_t(e) == win) key = 0u;
      }
    }
    __syncthreads();
    // stage 2: one warp per token merges the sorted chunk lists; lane c holds
    // the head of chunk c
    if (warp < T) {
      const int t = warp;
      const uint32_t* lk = ckey + (size_t)(t * nch + lane) * kk;
      const uint32_t* li = cidx + (size_t)(t * nch + lane) * kk;
      int ptr = 0;
      uint32_t hk = lane < nch ? lk[0] : 0u, hi = lane < nch ? li[0] : 0xFFFFFFFFu;
      uint32_t my_e = 0u, my_key = 0u;
#pragma unroll 1
      for (int r = 0; r < k; ++r) {
        const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, hk);
        const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, hk == wmax ? hi : 0xFFFFFFFFu);
        if (lane == r) {
          my_e = emin;
          my_key = wmax;
        }
        if (hk == wmax && hi == emin) {
          ++ptr;
          hk = ptr < kk ? lk[ptr] : 0u;
          hi = ptr < kk ? li[ptr] : 0xFFFFFFFFu;
        }
      }
      const float v = rank_value(my_key);
      const float v0 = __shfl_sync(0xFFFFFFFFu, v, 0);
      const float ex = lane < k ? expf(v - v0) : 0.0f;
      const float sum = warp_sum(ex);
      if (lane < k) {
        const float w = ex / sum;
        sel_e[t * k + lane] = int(my_e);
        sel_w[t * k + lane] = w;
        if (c == 0) {
          if (a.idx_out) a.idx_out[t * k + lane] = int(my_e);
          if (a.w_out) a.w_out[t * k + lane] = w;
        }
      }
    }
  }
  __syncthreads();
  // ---- gate/up matrices of the selected experts into L2 at once: the
  // concatenation of the distinct experts' matrices (first-occurrence order)
  // cut into G equal slices, slice c prefetched by this CTA, lane r taking
  // its part of the r-th matrix (up to 32 selections; larger T * k leaves the
  // prefetch to the per-tile one below)
  const bool early_pf = T * k <= 32;
  if (warp == 1 && early_pf) {
    const int n = T * k;
    const int ev = lane < n ? sel_e[lane] : -1 - lane;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, ev);
    const bool first = lane < n && (peers & ((1u << lane) - 1u)) == 0u;
    const unsigned firsts = __ballot_sync(0xFFFFFFFFu, first);
    if (first) {
      const uint64_t m = a.gu_mat, S = (uint64_t)__popc(firsts) * m;
      const uint64_t lo = (S * (uint64_t)c / (uint64_t)G) & ~uint64_t(15);
      const uint64_t hi = c + 1 == G ? S : (S * (uint64_t)(c + 1) / (uint64_t)G) & ~uint64_t(15);
      const uint64_t r0m = (uint64_t)__popc(firsts & ((1u << lane) - 1u)) * m;
      const uint64_t b0 = lo > r0m ? lo : r0m, b1 = hi < r0m + m ? hi : r0m + m;
      if (b1 > b0) prefetch_range(a.gate_up + (size_t)ev * m + (b0 - r0m), uint32_t(b1 - b0));
    }
  }
  // ---- active experts (ascending) with their slots, and this CTA's gate/up
  // range, by warp 0 alone -----------------------------------------------------------
  if (warp == 0) {
    // slot j = lane + 32 m holds expert ev[m]. Up to 32 slots (every decode
    // shape with k <= 8): match_any gives each slot its expert's slot set
    // (first occurrence, count, place), and one pass over the first
    // occurrences gives the rank; larger T * k compares through shuffles.
    const int n = T * k;
    int ev[4], fst[4], rank[4], pos[4], cnt[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j = lane + 32 * m;
      ev[m] = j < n ? sel_e[j] : 0x7FFFFFFF;
      fst[m] = j < n ? 1 : 0;
      rank[m] = pos[m] = cnt[m] = 0;
    }
    int D = 0;
    if (n <= 32) {
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, ev[0]);
      const unsigned lt = (1u << lane) - 1u;
      fst[0] = (lane < n && (peers & lt) == 0u) ? 1 : 0;
      cnt[0] = __popc(peers);
      pos[0] = __popc(peers & lt);
      const unsigned firsts = __ballot_sync(0xFFFFFFFFu, fst[0] != 0);
      D = __popc(firsts);
#pragma unroll 1
      for (unsigned f = firsts; f; f &= f - 1u) {
        const int i = __ffs(f) - 1;
        rank[0] += __shfl_sync(0xFFFFFFFFu, ev[0], i) < ev[0] ? 1 : 0;
      }
    } else {
      auto slot_e = [&](int i) {
        const int a0 = __shfl_sync(0xFFFFFFFFu, ev[0], i & 31), a1 = __shfl_sync(0xFFFFFFFFu, ev[1], i & 31);
        const int a2 = __shfl_sync(0xFFFFFFFFu, ev[2], i & 31), a3 = __shfl_sync(0xFFFFFFFFu, ev[3], i & 31);
        return i < 32 ? a0 : (i < 64 ? a1 : (i < 96 ? a2 : a3));
      };
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int ei = slot_e(i);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = lane + 32 * m;
          if (ei == ev[m]) {
            ++cnt[m];
            if (i < j) {
              ++pos[m];
              fst[m] = 0;
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) D += __popc(__ballot_sync(0xFFFFFFFFu, fst[m] != 0));
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int ei = slot_e(i);
        const int f0_ = __shfl_sync(0xFFFFFFFFu, fst[0], i & 31), f1_ = __shfl_sync(0xFFFFFFFFu, fst[1], i & 31);
        const int f2_ = __shfl_sync(0xFFFFFFFFu, fst[2], i & 31), f3_ = __shfl_sync(0xFFFFFFFFu, fst[3], i & 31);
        const int fi = i < 32 ? f0_ : (i < 64 ? f1_ : (i < 96 ? f2_ : f3_));
#pragma unroll
        for (int m = 0; m < 4; ++m) rank[m] += (fi && ei < ev[m]) ? 1 : 0;
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j = lane + 32 * m;
      if (j < n) {
        act_slot[rank[m] * kDecodeMaxT + pos[m]] = j;
        act_tok[rank[m] * kDecodeMaxT + pos[m]] = j / k;
        if (fst[m]) {
          act[rank[m]] = ev[m];
          act_n[rank[m]] = cnt[m];
        }
      }
    }
    if (lane < 2) {
      // gate/up tiles: contiguous ranges, balanced by bytes together with each
      // CTA's down units and shared-down rows. W(c) is the cumulative budget
      // left for tiles before CTA c (non-decreasing). Lane 0 finds where this
      // CTA's range starts, lane 1 where it ends.
      const int n_tiles = D * NTg;
      const float U = float(U_gu);
      const float DT = float(D) * float(U_dn) + (a.has_shared ? float(kTileRows) * float(sdrow_bytes) : 0.0f);
      const float target = (float(n_tiles) * U + float(NTd) * DT) / float(G);
      const int qt = NTd / G;
      const float w0 = fmaxf(0.0f, target - DT * float(qt)), w1 = fmaxf(0.0f, target - DT * float(qt + 1));
      auto W = [&](int cc) {
        const int big = (cc * NTd) / G - cc * qt;
        return float(cc - big) * w0 + float(big) * w1;
      };
      const int cc = c + lane;
      int v = n_tiles;
      if (cc < G) {
        const float WG = W(G);
        v = WG <= 0.0f ? 0 : int(floorf(float(n_tiles) * (W(cc) / WG) + 0.5f));
        v = v < 0 ? 0 : (v > n_tiles ? n_tiles : v);
      }
      misc[1 + lane] = v;
      if (lane == 0) misc[0] = D;
    }
  }
  __syncthreads();
  const int D = misc[0], i0 = misc[1], i1 = misc[2] > misc[1] ? misc[2] : misc[1];

  // this CTA's gate/up tiles into L2 (one prefetch per tile, unless the
  // slices above covered them), spread over the warps
  if (lane == 0) {
#pragma unroll 1
    for (int gt = i0 + warp; !early_pf && gt < i1; gt += kWarps) {
      const int ai = gt / NTg;
      prefetch_l2(a.gate_up + (size_t)act[ai] * a.gu_mat + (size_t)(gt - ai * NTg) * U_gu, U_gu);
    }
  }
  // down items (output tile, active expert, K-range of kU units), in rounds
  // of kMaxDnItems; the first round's table is built now, its copies are
  // issued as soon as this CTA's gate/up is done
  // units per item: up to kU, fewer when that gives every warp one item
  const int uD = D * ntl > 0 ? min(kU, ceil_div(KBi, max(1, kWarps / (D * ntl)))) : kU;
  const int KPD = ceil_div(KBi, uD);
  const int per_tile = D * KPD;
  const int n_dn = ntl * per_tile;
  // item j: byte offset of its first unit, (expert rank << 12 | kb0 << 4 | n)
  auto dn_table = [&](int rb) {
#pragma unroll 1
    for (int j = tid; j < min(kMaxDnItems, n_dn - rb); j += kThreads) {
      const int it = rb + j, tl = it / per_tile, rem = it - tl * per_tile, ai = rem / KPD;
      const int kb = (rem - ai * KPD) * uD;
      dtab[j] = make_int2(int(act[ai] * a.dn_mat + (uint64_t)(t0 + tl) * U_dn + (uint64_t)kb * kUnitBytes),
                          (ai << 12) | (kb << 4) | min(uD, KBi - kb));
    }
  };
  auto dn_issue = [&](int rb, int m) {   // this warp's m-th item of the round starting at rb
    const int it = rb + warp + m * kWarps;
    if (it < min(n_dn, rb + kMaxDnItems)) {
      const int2 e = dtab[it - rb];
      const uint8_t* src = a.down + uint32_t(e.x);
      uint8_t* dst = wb + (size_t)(m % kStageItems) * kItemBytes;
      const int n16 = (e.y & 15) * (kUnitBytes / 16);
#pragma unroll 1
      for (int c = lane; c < n16; c += 32) cp_async16(dst + c * 16, src + c * 16);
    }
    cp_async_commit();
  };
  dn_table(0);
  if (i1 == i0) __syncthreads();   // otherwise the gate/up round barrier orders it

  // ---- 3. routed gate/up: items (tile, K-range of kU units), item j of a round
  // on warp j % kWarps; every warp keeps kStageItems items in flight, copied
  // with cp.async into its own shared-memory buffers. The warp that finishes a
  // tile's last item adds the tile's partials in order, applies SwiGLU and
  // writes the tile's 8 features of h as 2 e4m3 terms per feature with one
  // factor per 8 features.
  {
    uint8_t* hT = a.h;
    float* hF = reinterpret_cast<float*>(a.h + (size_t)T * k * KBi * kHTermBytes);
    const int n_tiles = i1 - i0;
    const int KP = ceil_div(KBd, kU);
    const int tiles_per_round = kMaxGuItems / KP > 0 ? kMaxGuItems / KP : 1;
#pragma unroll 1
    for (int rb = 0; rb < n_tiles; rb += tiles_per_round) {
      const int nt_round = min(tiles_per_round, n_tiles - rb);
      const int n_items = nt_round * KP;
      if (rb > 0) __syncthreads();
      // item j: byte offset of its first unit, and (expert rank << 12 | kb0 << 4 | n)
#pragma unroll 1
      for (int j = tid; j < n_items; j += kThreads) {
        const int tl = j / KP, gt = i0 + rb + tl, ai = gt / NTg, kb = (j - tl * KP) * kU;
        gtab[j] = make_int2(int(act[ai] * a.gu_mat + (uint64_t)(gt - ai * NTg) * U_gu + (uint64_t)kb * kUnitBytes),
                            (ai << 12) | (kb << 4) | min(kU, KBd - kb));
      }
      for (int j = tid; j < nt_round; j += kThreads) tcnt[j] = 0;
      __syncthreads();
      auto issue = [&](int m) {   // this warp's m-th item of the round -> buffer m % kStageItems
        const int it = warp + m * kWarps;
        if (it < n_items) {
          const int2 e = gtab[it];
          const uint8_t* src = a.gate_up + uint32_t(e.x);
          uint8_t* dst = wb + (size_t)(m % kStageItems) * kItemBytes;
          const int n16 = (e.y & 15) * (kUnitBytes / 16);
#pragma unroll 1
          for (int c = lane; c < n16; c += 32) cp_async16(dst + c * 16, src + c * 16);
        }
        cp_async_commit();   // one group per item (empty past the end)
      };
#pragma unroll
      for (int m = 0; m < kStageItems; ++m) issue(m);
#pragma unroll 1
      for (int m = 0, it = warp; it < n_items; ++m, it += kWarps) {
        cp_async_wait<kStageItems - 1>();
        __syncwarp();
        const uint8_t* base = wb + (size_t)(m % kStageItems) * kItemBytes;
        const int meta = gtab[it].y;
        const int kb0 = (meta >> 4) & 255, n = meta & 15, ai = meta >> 12;
        const int tl = it / KP;
        const int nt = act_n[ai];
        const int* toks = act_tok + ai * kDecodeMaxT;
        int boff[kPairs], foff[kPairs];
        float acc[kPairs][2];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const int sb = 2 * p + (g >> 2), scol = 2 * p + (q >> 1);
          boff[p] = (sb < nt && (g & 3) < kActTerms) ? toks[sb] * KBd * kActRowKbBytes + (g & 3) * 32 + q * 8 : -1;
          foff[p] = scol < nt ? toks[scol] * KBd : -1;
          acc[p][0] = acc[p][1] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (u < n) {
            const uint8_t* unit = base + (size_t)u * kUnitBytes;
            const AFrag af = load_afrag(unit, g, q);
            const uint32_t sc = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
            const int kb = kb0 + u;
            const float fwl = scale_lo(sc), fwh = scale_hi(sc);
#pragma unroll
            for (int p = 0; p < kPairs; ++p) {
              const uint2 bv = boff[p] >= 0 ? *reinterpret_cast<const uint2*>(xb + boff[p] + kb * kActRowKbBytes)
                                            : make_uint2(0u, 0u);
              const float fa = foff[p] >= 0 ? xfa[foff[p] + kb] : 0.0f;
              float dd[4];
              mma_e4m3(dd, af.a0, af.a1, af.a2, af.a3, bv.x, bv.y);
              acc[p][0] = fmaf((dd[0] + dd[1]) * fa, fwl, acc[p][0]);
              acc[p][1] = fmaf((dd[2] + dd[3]) * fa, fwh, acc[p][1]);
            }
          }
        }
        __syncwarp();   // every lane is done with the buffer before it is refilled
        issue(m + kStageItems);
        // the term pairs of a token sit in lanes q and q^1
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const float v0 = acc[p][0] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][0], 1);
          const float v1 = acc[p][1] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][1], 1);
          if ((q & 1) == 0) {
            float* o = gpart + (size_t)(it * kPairs + p) * 32;
            o[g * 2 + (q >> 1)] = v0;        // gate row g, token column q>>1
            o[16 + g * 2 + (q >> 1)] = v1;   // up row g
          }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence_block();
          last = atomicAdd(&tcnt[tl], 1) == KP - 1;
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (last) {
          // this warp finished the tile's last item: partials in K order, SwiGLU, h
          __threadfence_block();
          const int gt = i0 + rb + tl, tt = gt - ai * NTg, kbh = tt >> 2, grp = tt & 3;
          const int* slots = act_slot + ai * kDecodeMaxT;
#pragma unroll
          for (int p = 0; p < kPairs; ++p) {
            if (2 * p < nt) {
              float v = 0.0f;
#pragma unroll 1
              for (int kp = 0; kp < KP; ++kp) v += gpart[(size_t)((tl * KP + kp) * kPairs + p) * 32 + lane];
              const float up = __shfl_down_sync(0xFFFFFFFFu, v, 16);
              const float hv = lane < 16 ? silu_f(v) * up : 0.0f;   // feature lane>>1, token column lane&1
              float am = fabsf(hv);
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 8));
              int ex = kActZeroExp;
              uint32_t e0 = 0u, e1 = 0u;
              if (am > 0.0f) {
                ex = floor_log2(am) - 7;
                const float sv = scale2(hv, -ex);
                e0 = f32x2_to_e4m3x2(sv, 0.0f) & 0xFFu;
                e1 = f32x2_to_e4m3x2(sv - e4m3_to_f32_hw(e0), 0.0f) & 0xFFu;
              }
              const int scol = 2 * p + (lane & 1);
              if (lane < 16 && scol < nt) {
                const int slx = slots[scol];
                // feature 8 grp + (lane >> 1) of K-block kbh, at its B-fragment position
                const size_t base_h = ((size_t)slx * KBi + kbh) * kHTermBytes + bfrag_pos(grp * 8 + (lane >> 1));
                hT[base_h] = uint8_t(e0);
                hT[base_h + 32] = uint8_t(e1);
                if ((lane >> 1) == 0) hF[((size_t)slx * KBi + kbh) * kHGroups + grp] = act_factor(ex, sel_w[slx]);
              }
            }
          }
        }
      }
      cp_async_wait<0>();
      __syncthreads();
    }
  }
  // 3-4 tokens: the down units of this CTA's output tiles for every active
  // expert into L2 (one prefetch per expert), now that its gate/up weights
  // are in (issued earlier they compete with them for DRAM); 1-2 tokens need
  // none: the first down items below are copied during the h exchange
  if constexpr (T >= 3) {
    if (lane == 0 && ntl > 0)
#pragma unroll 1
      for (int ai = kWarps - 1 - warp; ai < D; ai += kWarps)
        prefetch_range(a.down + (size_t)act[ai] * a.dn_mat + (size_t)t0 * U_dn, uint32_t(ntl) * U_dn);
  }
  // the first down items into each warp's (now free) buffers, then this CTA's
  // h is written: publish (the last warp; the others go on)
#pragma unroll
  for (int m = 0; m < kStageItems; ++m) dn_issue(0, m);
  if (warp == kWarps - 1 && lane == 0) red_release_add(&st->gudone, 1u);

  // ---- 4. shared-down rows of this CTA's output tiles while the other CTAs
  // finish their gate/up
  if (a.has_shared && ntl > 0) {
#pragma unroll 1
    for (int j = tid; j < T * I; j += kThreads) hsh[j] = __ldcg(a.h_sh + j);
    __syncthreads();
    const int n8 = I / 8;
#pragma unroll 1
    for (int rr = warp; rr < ntl * kTileRows; rr += kWarps) {
      const uint4* w4 = reinterpret_cast<const uint4*>(a.sh_down + (size_t)(t0 * kTileRows + rr) * I);
      float acc[T];
#pragma unroll
      for (int t = 0; t < T; ++t) acc[t] = 0.0f;
#pragma unroll 1
      for (int j0 = 0; j0 < n8; j0 += 32 * 4) {
        uint4 w[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = j0 + lane + 32 * m;
          w[m] = j < n8 ? ldg_nc_stream_u4(w4 + j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = j0 + lane + 32 * m;
          if (j < n8) {
#pragma unroll
            for (int t = 0; t < T; ++t) acc[t] += dot8_f32(w[m], hsh + (size_t)t * I + j * 8);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) yacc[t * kYStride + rr] = v;
      }
    }
  }

  // ---- 5. down: item j of a round on warp j % kWarps, copied from L2
  // (prefetched during gate/up) into the warp's buffers before the wait for
  // every CTA's h -----------------------------------------------------------------------

  if (n_dn > 0) {
    if (tid == 0) wait_geq_u32(&st->gudone, uint32_t(G), a.status);
    __syncthreads();
    // every slot's h terms and group factors (contiguous in the workspace and
    // in shared memory); x and its terms are dead now
    const int n16h = T * k * KBi * (kHTermBytes + kHGroups * 4) / 16;
#pragma unroll 1
    for (int j = tid; j < n16h; j += kThreads)
      reinterpret_cast<uint4*>(hbs)[j] = __ldcg(reinterpret_cast<const uint4*>(a.h) + j);
    __syncthreads();
    // B columns of a down MMA: 4 groups of 8 features x 2 terms (column g =
    // group g / 2, term g % 2). Lane (g, q) supplies MMA K positions whose
    // elements (8q + 0..7, see load_afrag) all lie in group q, so its B words
    // are nonzero only for column group q; it holds the C columns of group q,
    // and the quad sum adds the groups.
    const bool grp_ok = (g >> 1) == q;
#pragma unroll 1
    for (int rb = 0; rb < n_dn; rb += kMaxDnItems) {
      const int round_end = min(n_dn, rb + kMaxDnItems);
      if (rb > 0) {
        __syncthreads();
        dn_table(rb);
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kStageItems; ++m) dn_issue(rb, m);
      }
#pragma unroll 1
      for (int m = 0, it = rb + warp; it < round_end; ++m, it += kWarps) {
        cp_async_wait<kStageItems - 1>();
        __syncwarp();
        const uint8_t* base = wb + (size_t)(m % kStageItems) * kItemBytes;
        const int meta = dtab[it - rb].y;
        const int kb0 = (meta >> 4) & 255, n = meta & 15, ai = meta >> 12;
        const int nt = act_n[ai];
        const int* slots = act_slot + ai * kDecodeMaxT;
        const int* toks = act_tok + ai * kDecodeMaxT;
        int hbo[T], hfo[T], tok[T];
        float dacc[T][2];
#pragma unroll
        for (int si = 0; si < T; ++si) {
          const int sl = si < nt ? slots[si] : 0;
          hbo[si] = sl * KBi * kHTermBytes + (g & 1) * 32 + 8 * q;
          hfo[si] = sl * KBi * kHGroups + q;
          tok[si] = si < nt ? toks[si] : -1;
          dacc[si][0] = dacc[si][1] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (u < n) {
            const uint8_t* unit = base + (size_t)u * kUnitBytes;
            const AFrag af = load_afrag(unit, g, q);
            const uint32_t sc = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
            const int kb = kb0 + u;
            const float fwl = scale_lo(sc), fwh = scale_hi(sc);
#pragma unroll
            for (int si = 0; si < T; ++si) {
              if (T > 1 && si >= nt) continue;
              const uint2 bw = grp_ok ? *reinterpret_cast<const uint2*>(hbs + hbo[si] + kb * kHTermBytes)
                                      : make_uint2(0u, 0u);
              const float fa = hfa[hfo[si] + kb * kHGroups];
              float dd[4];
              mma_e4m3(dd, af.a0, af.a1, af.a2, af.a3, bw.x, bw.y);
              const float vlo = (dd[0] + dd[1]) * fa * fwl;
              const float vhi = (dd[2] + dd[3]) * fa * fwh;
#pragma unroll
              for (int tt = 0; tt < T; ++tt) {
                dacc[tt][0] += tt == tok[si] ? vlo : 0.0f;
                dacc[tt][1] += tt == tok[si] ? vhi : 0.0f;
              }
            }
          }
        }
        __syncwarp();
        dn_issue(rb, m + kStageItems);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          float v0 = dacc[t][0], v1 = dacc[t][1];
          v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
          v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
          v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
          v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
          if (q == 0) {
            float* o = dpart + (size_t)((it - rb) * T + t) * kTileRows;
            o[g] = v0;
            o[8 + g] = v1;
          }
        }
      }
      cp_async_wait<0>();
      __syncthreads();
      // add this round's partials into the y accumulators: one warp per
      // output, lane i taking items i, i + 32 (fixed order, tree sum)
#pragma unroll 1
      for (int j = warp; j < T * ntl * kTileRows; j += kWarps) {
        const int t = j / (ntl * kTileRows), r = j - t * (ntl * kTileRows);
        const int tl = r / kTileRows, rr = r - tl * kTileRows;
        const int lo = max(rb, tl * per_tile), hi = min(round_end, (tl + 1) * per_tile);
        float v = 0.0f;
#pragma unroll 1
        for (int it = lo + lane; it < hi; it += 32) v += dpart[(size_t)((it - rb) * T + t) * kTileRows + rr];
        v = warp_sum(v);
        if (lane == 0) yacc[t * kYStride + r] += v;
      }
    }
    __syncthreads();
  } else {
    cp_async_wait<0>();
    __syncthreads();
  }
#pragma unroll 1
  for (int j = tid; j < T * ntl * kTileRows; j += kThreads) {
    const int t = j / (ntl * kTileRows), r = j - t * (ntl * kTileRows);
    a.y[(size_t)t * d + t0 * kTileRows + r] = __float2bfloat16_rn(yacc[t * kYStride + r]);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&st->done, 1u);
    if (old % uint32_t(G) == uint32_t(G) - 1u) {
      // last CTA of this call: every CTA is past every wait of this call
      st->routed = 0u;
      st->gudone = 0u;
      __threadfence();
    }
  }
}

}  // namespace

size_t decode_state_bytes(int T, int E) {
  (void)T;
  (void)E;
  return (size_t)kDecodeStateWords * 4;
}

uint32_t decode_he_stride(int I) { return align_up(uint32_t(I / kMxBlock), 8); }

size_t decode_h_bytes(int T, int k, int I) {
  return (size_t)T * k * (I / kMxBlock) * (kHTermBytes + kHGroups * 4);
}

int decode_plan(const DecodeArgs& a, const DeviceInfo& di, uint32_t* smem_bytes) {
  if (a.T < 1 || a.T > kDecodeMaxT) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.d % 32 || a.I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.k < 1 || a.k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.E > 32 * kMergeChunks) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int G = di.sm_count;
  if (G < 1 || ceil_div(a.d / kTileRows, G) > kDecodeMaxTiles) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (a.T * a.k > kThreads) return MOE_ERR_UNSUPPORTED_SHAPE;
  const Smem s = smem_plan(a.T, a.d, a.I, a.E, a.k, G);
  if (s.total + 1024 > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  *smem_bytes = s.total;
  return MOE_OK;
}

template <int T>
int launch_decode_t(const DecodeArgs& a, uint32_t smem, const DeviceInfo& di, cudaStream_t s) {
  const Smem L = smem_plan(T, a.d, a.I, a.E, a.k, di.sm_count);
  MOE_CUDA_TRY(cudaFuncSetAttribute(decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  int per_sm = 0;
  MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T>, kThreads, smem));
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  // One CTA per SM; every CTA waits for the others, which is safe because the
  // whole grid fits on the device at once (per_sm >= 1, grid = SM count).
  // Programmatic stream serialisation lets the next kernel on the stream start
  // its weight prefetches while this one finishes; it reads nothing this one
  // writes before its griddepcontrol.wait.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(di.sm_count);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, decode_kernel<T>, a, L));
  return MOE_OK;
}

int launch_decode(const DecodeArgs& a, const DeviceInfo& di, cudaStream_t s) {
  uint32_t smem = 0;
  const int st = decode_plan(a, di, &smem);
  if (st != MOE_OK) return st;
  switch (a.T) {
    case 1: return launch_decode_t<1>(a, smem, di, s);
    case 2: return launch_decode_t<2>(a, smem, di, s);
    case 3: return launch_decode_t<3>(a, smem, di, s);
    default: return launch_decode_t<4>(a, smem, di, s);
  }
}

}  // namespace moe
