// Single-launch decode path (T <= 4 tokens): one cooperative persistent kernel,
// one CTA per SM, so a layer call is a single launch with no host round trips.
//
// Every CTA walks a private sequence of "loads". A producer warp fills the
// slots of a shared-memory ring with 1-D bulk copies, in load order; the 15
// compute warps consume every load independently (no CTA-wide barrier per
// load): each waits for the slot, does its share, and releases the slot
// (the slot is refilled once all 15 have released it).
//
//   R   its slice of router rows          -> logits (global)      warp per row
//   F   its slice of shared gate/up rows  -> h_sh (global)        warp per feature
//   GU  its routed gate/up tiles          -> h (global, fp32)     needs routing
//   SD  shared-down rows of its tiles     -> y accumulators       needs all h_sh
//   DN  routed-down units of its tiles    -> y accumulators       needs all h
//
// A routed gate/up tile (16 rows: 8 gate + 8 up rows of one active expert) is
// split along K over the warps. Every warp writes its partial sums to one of a
// few reduction buffers, and the last warp to arrive (a shared-memory counter)
// adds the fifteen partials in warp order, so results do not depend on timing,
// and writes 8 features of h.
//
// Routing: once its router rows are in the logits a CTA increments a global
// counter. While the other CTAs catch up, its warps turn the activations into
// e4m3 terms; then every CTA reads all logits and runs the top-k itself (all
// warps: the best k of every 32-expert chunk, then one merge warp per token),
// so no second exchange is needed, and hands its routed loads to the producer.
// Gate/up tiles are handed out so every CTA moves about the same number of
// bytes in the routed phase (tiles, down units and shared-down rows counted
// together). The shared-down rows are prefetched into L2 while the routing is
// under way.
//
// After its gate/up tiles a CTA publishes with one release increment; before
// its down units it waits for all CTAs, splits every slot's h into e4m3 terms
// (with the routing weight folded into the block factor), and runs its down
// units, which accumulate in registers per output tile. The cross-warp sum is
// taken once per tile at the end; each CTA owns whole 16-row output tiles, so
// y is written without a cross-CTA reduction.
//
// Cross-call state (counters) lives at the start of the workspace and must be
// zero before the first call; the last CTA of a call resets it. Every wait is
// bounded (kSpinBudget); on timeout the kernel sets MOE_DEV_TIMEOUT and
// carries on, so it always terminates.
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode.h"
#include "host_util.h"
#include "mma_tile.cuh"
#include "topk.cuh"

namespace moe {
namespace {

#ifdef MOE_DECODE_TRACE
// Debug builds only: per-CTA globaltimer stamps at phase boundaries and cycle
// sums of thread 0.
constexpr int kTracePoints = 32;
__device__ unsigned long long g_trace[1024][kTracePoints];
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace(int point) {
  if (threadIdx.x == 0) g_trace[blockIdx.x][point] = gtime();
}
__device__ __forceinline__ void trace_put(int point, unsigned long long v) {
  if (threadIdx.x == 0) g_trace[blockIdx.x][point] = v;
}
__device__ __forceinline__ long long dclk() { return clock64(); }
#else
__device__ __forceinline__ void trace(int) {}
__device__ __forceinline__ void trace_put(int, unsigned long long) {}
__device__ __forceinline__ long long dclk() { return 0; }
#endif

constexpr int kWarps = 15;                  // compute warps
constexpr int kThreads = (kWarps + 1) * 32; // + one producer warp that issues the bulk copies
constexpr int kComputeThreads = kWarps * 32;
// Warps that share one routed gate/up tile (K split among them), and tiles in
// flight per CTA. At T = 1 a CTA holds 5 or 6 tiles: 3 groups of 5 warps take
// two short rounds for either count, where 5 groups of 3 would need a second
// full-length round for a sixth tile. At T = 2..4 (about 20 tiles per CTA)
// 5 groups of 3 keep more tiles in flight.
template <int T>
struct GroupCfg {
  static constexpr int kWarpsPer = T == 1 ? 5 : 3;
  static constexpr int kCount = kWarps / kWarpsPer;
};
constexpr int kGroupSlots = kWarps;   // groups x warps per group, for every T
constexpr int kRowsPerLoad = 4;   // bf16 rows per load: router rows, or 2 shared features x (gate, up)
constexpr int kMaxKbPerWarp = 8;  // routed gate/up: d <= kWarps * 8 * 32 = 3840
constexpr int kMergeChunks = 16;  // top-k: E <= 16 chunks of 32 experts
// gate/up MMA items per warp issued back to back (no branches in between):
// 8 at T = 1 (16 K-blocks per warp and tile), 6 otherwise (27 per warp);
// a build may fix it with MOE_DECODE_UNROLL
template <int T>
__host__ __device__ constexpr int unroll_for() {
#ifdef MOE_DECODE_UNROLL
  return MOE_DECODE_UNROLL;
#else
  return T == 1 ? 8 : 6;
#endif
}
constexpr int kHTermBytes = 64;   // h of one (slot, K-block): 2 e4m3 terms x 32 features
constexpr int kHGroups = 4;       // 8-feature groups per K-block, one exponent each

#ifndef MOE_DECODE_STAGE_CAP
#define MOE_DECODE_STAGE_CAP kDecodeMaxStages
#endif
// Ring depth limit (slots per CTA).
constexpr int kDecodeStageCap = MOE_DECODE_STAGE_CAP;

// Barrier among the compute warps only (the producer warp never joins it).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory"); }
// Count of compute threads with v != 0; also a barrier among them.
__device__ __forceinline__ int csync_count(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %1, 0;\n bar.red.popc.u32 %0, 1, %2, p;\n}\n"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kComputeThreads)
      : "memory");
  return int(r);
}

// Barrier among the GW warps of group gid (ids 2.. are free).
template <int GW>
__device__ __forceinline__ void group_sync(int gid) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + gid), "n"(GW * 32) : "memory");
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
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Weight scale byte -> 2^(s-127) as fp32 (s = 0 gives 0, s = 255 gives +inf).
__device__ __forceinline__ float scale_lo(uint32_t sc16) { return __uint_as_float((sc16 << 23) & 0x7F800000u); }
__device__ __forceinline__ float scale_hi(uint32_t sc16) { return __uint_as_float((sc16 << 15) & 0x7F800000u); }

// Factor that turns an MMA result over one (weight block, activation block)
// into its true value, apart from the weight scale: weights were decoded as
// 2^-6 x E2M1 value and the activation block stored as terms x 2^-e, so the
// factor is w x 2^(e+6) (0 for an all-zero block).
__device__ __forceinline__ float act_factor(int e, float w) {
  return e == kActZeroExp ? 0.0f : scale2(w, e + 6);
}

// Row (bf16, n8 chunks of 8 elements in shared memory) times T activation
// rows: one warp, lanes strided over the chunks; every lane gets the sums.
template <int T>
__device__ __forceinline__ void warp_row_dot(const uint4* row, const uint4* xs4, int n8, int lane, float (&out)[T]) {
  float acc[T];
#pragma unroll
  for (int t = 0; t < T; ++t) acc[t] = 0.0f;
#pragma unroll 4
  for (int j = lane; j < n8; j += 32) {
    const uint4 w = row[j];
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t] += dot8_bf16(w, xs4[t * n8 + j]);
  }
#pragma unroll
  for (int t = 0; t < T; ++t) out[t] = warp_sum(acc[t]);
}

// Shared-memory carve-up (byte offsets), identical on host and device. The
// activation terms (xs, xb, xfa; dead after the gate/up tiles), the shared h
// (hsh; dead after the shared-down rows) and the h terms (hbs, hfa) share
// one region.
struct Smem {
  uint32_t ring, bars, red, ov, xs, xb, xfa, hsh, hbs, hfa, dnred, ysd, sel_e, sel_w, act, act_n,
      act_slot, act_tok, first, misc, total;
};
__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline uint32_t he_stride(int I) { return align_up(uint32_t(I / kMxBlock), 8); }
__host__ __device__ inline int red_floats(int T) { return 32 * ((T + 1) / 2); }
__host__ __device__ inline int max_tiles_per_cta(int d, int G) { return (d / kTileRows + G - 1) / G; }
__host__ __device__ inline Smem smem_plan(int T, int d, int I, int E, int k, int stages, uint32_t slot_bytes,
                                          int max_tiles) {
  Smem s{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = align_up(at, align);
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  const uint32_t KBd = uint32_t(d / kMxBlock), KBi = uint32_t(I / kMxBlock), slots = uint32_t(T * k);
  s.ring = take(uint32_t(stages) * slot_bytes, 128);
  s.bars = take(8u * uint32_t(2 * stages + 1), 8);   // full[S], empty[S], routing
  const uint32_t nch = uint32_t((E + 31) / 32), kk = uint32_t(k < 32 ? k : 32);
  // gate/up partials: per group, two tiles in turn, one row per warp
  const uint32_t red_b = uint32_t(2 * kGroupSlots * red_floats(T)) * 4u;
  const uint32_t cand_b = uint32_t(T) * nch * kk * 8u;
  s.red = take(red_b > cand_b ? red_b : cand_b, 16);
  const uint32_t xs_b = align_up(uint32_t(T) * d * 2, 16);
  const uint32_t xb_b = align_up(uint32_t(T) * KBd * kActRowKbBytes, 16);
  const uint32_t xfa_b = align_up(uint32_t(T) * KBd * 4, 16);
  const uint32_t a_b = xs_b + xb_b + xfa_b;
  const uint32_t hsh_b = align_up(uint32_t(T) * I * 4, 16);
  const uint32_t hbs_b = align_up(slots * KBi * kHTermBytes, 16);
  const uint32_t hfa_b = align_up(slots * KBi * kHGroups * 4, 16);
  const uint32_t b_b = hbs_b + hfa_b;
  uint32_t ov = a_b > hsh_b ? a_b : hsh_b;
  ov = ov > b_b ? ov : b_b;
  s.ov = take(ov, 128);
  s.xs = s.ov;
  s.xb = s.xs + xs_b;
  s.xfa = s.xb + xb_b;
  s.hsh = s.ov;
  s.hbs = s.ov;
  s.hfa = s.hbs + hbs_b;
  s.dnred = take(uint32_t(max_tiles * kWarps * T * kTileRows) * 4u, 16);
  s.ysd = take(uint32_t(T * max_tiles * kTileRows) * 4u, 16);
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

// Per-CTA load sequence: [0,nR) router, [nR,bF) shared gate/up, [bF,bGU)
// routed gate/up tiles, [bGU,bSD) shared down, [bSD,bDN) routed down loads
// (nL loads of at most dnch units per output tile).
struct Seq {
  int r0, r1, f0, f1, t0, ntl;
  int nR, nF, nSD;
  int rch, fch, sdch, dnch;
  int D, i0, i1, nL, nDN;
  int bF, bGU, bSD, bDN;
  __device__ void set_routed(int D_, int i0_, int i1_) {
    D = D_;
    i0 = i0_;
    i1 = i1_ > i0_ ? i1_ : i0_;
    bGU = bF + (i1 - i0);
    bSD = bGU + nSD;
    nL = (D + dnch - 1) / dnch;
    nDN = ntl * nL;
    bDN = bSD + nDN;
  }
};

// L: the shared-memory carve-up, computed once on the host (smem_plan).
template <int T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a, Smem L) {
  extern __shared__ __align__(128) uint8_t sm[];
  trace(0);
  trace_put(17, (unsigned long long)clock64());
  long long tacc[12] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};   // debug builds: cycle sums of thread 0
  auto trace_add = [&](int point, long long v) { tacc[point - 20] += v; };
  constexpr int kGroupWarps = GroupCfg<T>::kWarpsPer, kGroups = GroupCfg<T>::kCount;
  constexpr int kUnroll = unroll_for<T>();
  constexpr int kPairs = (T + 1) / 2;
  constexpr int kRF = 32 * kPairs;
  const int d = a.d, I = a.I, E = a.E, k = a.k;
  const int KBd = d / kMxBlock, KBi = I / kMxBlock;
  const int NTd = d / kTileRows, NTg = 2 * I / kTileRows;
  const int G = gridDim.x, c = blockIdx.x, S = a.stages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int max_tiles = max_tiles_per_cta(d, G);
  uint8_t* ring = sm + L.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* rbar = empty + S;
  float* red = reinterpret_cast<float*>(sm + L.red);
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(sm + L.xs);
  const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
  uint8_t* xb = sm + L.xb;
  float* xfa = reinterpret_cast<float*>(sm + L.xfa);
  float* hsh = reinterpret_cast<float*>(sm + L.hsh);
  uint8_t* hbs = sm + L.hbs;
  float* hfa = reinterpret_cast<float*>(sm + L.hfa);
  float* dnred = reinterpret_cast<float*>(sm + L.dnred);
  float* ysd = reinterpret_cast<float*>(sm + L.ysd);
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
  const int ystride = max_tiles * kTileRows;

  Seq s;
  s.r0 = c * E / G;
  s.r1 = (c + 1) * E / G;
  s.f0 = a.has_shared ? c * I / G : 0;
  s.f1 = a.has_shared ? (c + 1) * I / G : 0;
  s.t0 = c * NTd / G;
  s.ntl = (c + 1) * NTd / G - s.t0;
  s.rch = min(kRowsPerLoad, max(1, int(a.slot_bytes / row_bytes)));
  s.fch = min(kRowsPerLoad / 2, max(1, int(a.slot_bytes / (2 * row_bytes))));
  s.sdch = max(1, int(a.slot_bytes / sdrow_bytes));
  s.dnch = max(1, int(a.slot_bytes / U_dn));
  s.nR = (s.r1 - s.r0 + s.rch - 1) / s.rch;
  s.nF = (s.f1 - s.f0 + s.fch - 1) / s.fch;
  s.nSD = a.has_shared ? (s.ntl * kTileRows + s.sdch - 1) / s.sdch : 0;
  s.bF = s.nR + s.nF;
  s.D = 0;
  s.i0 = s.i1 = 0;
  s.nL = s.nDN = 0;
  s.bGU = s.bSD = s.bDN = s.bF;

  // bulk-copy requests of load i into its ring slot (producer lane only)
  auto issue = [&](int i) {
    const int slot = i % S;
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
    } else if (i < s.bGU) {
      const int gt = s.i0 + (i - s.bF), ai = gt / NTg, tt = gt - ai * NTg;
      mbar_arrive_expect_tx(bar, U_gu);
      bulk_g2s(dst, a.gate_up + (size_t)act[ai] * a.gu_mat + (size_t)tt * U_gu, U_gu, bar);
    } else if (i < s.bSD) {
      const int r = s.t0 * kTileRows + (i - s.bGU) * s.sdch;
      const int n = min(s.sdch, (s.t0 + s.ntl) * kTileRows - r);
      mbar_arrive_expect_tx(bar, n * sdrow_bytes);
      bulk_g2s(dst, a.sh_down + (size_t)r * I, n * sdrow_bytes, bar);
    } else {
      const int l = i - s.bSD, tl = l / s.nL, a0 = (l - tl * s.nL) * s.dnch, n = min(s.dnch, s.D - a0);
      mbar_arrive_expect_tx(bar, n * U_dn);
      for (int j = 0; j < n; ++j)
        bulk_g2s(dst + (size_t)j * U_dn, a.down + (size_t)act[a0 + j] * a.dn_mat + (size_t)(s.t0 + tl) * U_dn,
                 U_dn, bar);
    }
  };

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarps);
    }
    mbar_init(rbar, 1);
    mbar_fence_init();
  }
  __syncthreads();   // the only full-CTA barrier: barriers and counters initialised

  if (warp == kWarps) {
    // ---- producer warp: issues every bulk copy, in load order ----------------
    if (lane == 0) {
      int n_loads = s.bF;
      for (int j = 0;; ++j) {
        if (j == s.bF) {
          // shared-down rows into L2 while the routing is under way
          if (s.nSD > 0) {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(a.sh_down + (size_t)s.t0 * kTileRows * I);
            const uint32_t bytes = uint32_t(s.ntl * kTileRows) * sdrow_bytes;
            for (uint32_t o = 0; o < bytes; o += 32768u) prefetch_l2(src + o, min(32768u, bytes - o));
          }
          // the routed loads are known once the compute warps have routed
          if (!mbar_wait(rbar, 0u, a.status, 256)) break;
          s.set_routed(misc[0], misc[1], misc[2]);
          n_loads = s.bDN;
        }
        if (j >= n_loads) break;
        if (j >= S && !mbar_wait(&empty[j % S], uint32_t(j / S - 1) & 1u, a.status, 256)) break;
        issue(j);
      }
#ifdef MOE_DECODE_TRACE
      g_trace[blockIdx.x][16] = gtime();
#endif
    }
    return;
  }

  // activations: plain loads by the compute warps (read-only during the call)
  for (int j = tid; j < T * d / 8; j += kComputeThreads)
    reinterpret_cast<uint4*>(xs)[j] = __ldg(reinterpret_cast<const uint4*>(a.x) + j);
  for (int i = tid; i < T * ystride; i += kComputeThreads) ysd[i] = 0.0f;
  if (tid == 0) {
    if (s.nR == 0) red_release_add_u64(&st->bar, 1ull);
    if (s.nF == 0) red_release_add(&st->shcnt, 1u);
  }
  csync();
  trace(1);

  // per-lane down accumulators of the current output tile: [token][row g / row g+8]
  float dacc[T][2];
#pragma unroll
  for (int t = 0; t < T; ++t) dacc[t][0] = dacc[t][1] = 0.0f;
  int dn_tile = -1;
  // this warp's down partials of output tile tl -> dnred (the four lanes of a
  // quad hold the same two rows for different columns)
  auto flush_tile = [&](int tl) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float v0 = dacc[t][0], v1 = dacc[t][1];
      v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
      v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
      v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
      v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
      if (q == 0) {
        float* o = dnred + ((size_t)(tl * kWarps + warp) * T + t) * kTileRows;
        o[g] = v0;
        o[8 + g] = v1;
      }
      dacc[t][0] = dacc[t][1] = 0.0f;
    }
  };

  for (int i = 0;; ++i) {
    if (i == s.nR) {
      // ---- routing ----------------------------------------------------------
      csync();   // every router row of this CTA is in the logits
      if (tid == 0 && s.nR > 0) red_release_add_u64(&st->bar, 1ull);
      // activations -> e4m3 terms (B operand of the gate/up MMAs)
#pragma unroll 1
      for (int u = warp; u < T * KBd; u += kWarps) {
        const float v = __bfloat162float(xs[(size_t)u * kMxBlock + lane]);
        const int ex = split_block(v, lane, xb + (size_t)u * kActRowKbBytes);
        if (lane == 0) xfa[u] = act_factor(ex, 1.0f);
      }
      trace(3);
      if (tid == 0) wait_geq_u64(&st->bar, (unsigned long long)G, a.status);
      csync();
      trace(4);
      // stage 1: the best min(k, 32) of every (token, 32-expert chunk), by
      // key descending, equal keys -> lower expert index
      const int nch = (E + 31) / 32, kk = k < 32 ? k : 32;
      uint32_t* ckey = reinterpret_cast<uint32_t*>(red);
      uint32_t* cidx = ckey + T * nch * kk;
      // all my tasks' logits are requested before the first round
      constexpr int kTasksPerWarp = (kDecodeMaxT * kMergeChunks + kWarps - 1) / kWarps;
      uint32_t keys[kTasksPerWarp];
#pragma unroll
      for (int m = 0; m < kTasksPerWarp; ++m) {
        const int task = warp + m * kWarps, t = task / nch;
        const int e = (task - t * nch) * 32 + lane;
        keys[m] = 0u;
        if (task < T * nch && e < E) {
          float v = __ldcg(a.logits + (size_t)t * E + e);
          if (a.bias) v = __fadd_rn(v, a.bias[(size_t)t * a.bias_stride + e]);
          keys[m] = rank_key(v);
        }
      }
#pragma unroll
      for (int m = 0; m < kTasksPerWarp; ++m) {
        const int task = warp + m * kWarps;
        if (task >= T * nch) break;
        const uint32_t e = uint32_t((task % nch) * 32 + lane);
        uint32_t key = keys[m];
#pragma unroll 1
        for (int r = 0; r < kk; ++r) {
          const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, key);
          const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, (m != 0u && key == m) ? e : 0xFFFFFFFFu);
          if (lane == 0) {
            ckey[task * kk + r] = m;
            cidx[task * kk + r] = win;
          }
          if (e == win) key = 0u;
        }
      }
      csync();
      trace(5);
      // stage 2: one warp per token merges the sorted chunk lists; lane c
      // holds the head of chunk c
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
      csync();
      trace(6);
      // active experts ascending; each with its slots (slot = t*k + j) in token order
      const int n = T * k;
      int f = 0;
      if (tid < n) {
        const int e = sel_e[tid];
        f = 1;
        for (int j = 0; j < tid; ++j) f &= sel_e[j] != e ? 1 : 0;
        first[tid] = f;
      }
      const int D = csync_count(f != 0);
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
      if (tid < 2) {
        // gate/up tiles: contiguous ranges, balanced by bytes together with
        // each CTA's down units and shared-down rows. W(c) is the cumulative
        // budget left for tiles before CTA c (non-decreasing). Thread 0 finds
        // where my range starts, thread 1 where it ends.
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
        const int cc = c + tid;
        int v = n_tiles;
        if (cc < G) {
          const float WG = W(G);
          v = WG <= 0.0f ? 0 : int(floorf(float(n_tiles) * (W(cc) / WG) + 0.5f));
          v = v < 0 ? 0 : (v > n_tiles ? n_tiles : v);
        }
        misc[1 + tid] = v;
        if (tid == 0) misc[0] = D;
      }
      csync();
      s.set_routed(D, misc[1], misc[2]);
      if (tid == 0) mbar_arrive(rbar);   // hands the routed loads to the producer warp
      trace(7);
    }
    if (i == s.bF && s.nF > 0) {
      csync();   // every shared gate/up feature of this CTA is in h_sh
      if (tid == 0) red_release_add(&st->shcnt, 1u);
    }
    if (i == s.bGU) {
      // ---- publish my h; collect every CTA's h_sh ------------------------------
      csync();
      trace(9);
      if (tid == 0) red_release_add(&st->gudone, 1u);
      if (a.has_shared) {
        if (tid == 0) wait_geq_u32(&st->shcnt, uint32_t(G), a.status);
        csync();
        for (int j = tid; j < T * I; j += kComputeThreads) hsh[j] = __ldcg(a.h_sh + j);
        csync();
      }
      trace(10);
    }
    if (i == s.bSD) {
      // ---- every CTA's h -> e4m3 terms (routing weight folded into the factor)
      if (tid == 0) wait_geq_u32(&st->gudone, uint32_t(G), a.status);
      csync();
      trace(11);
      // every slot's h terms and group factors (contiguous in the workspace
      // and in shared memory)
      const int n16 = T * k * KBi * (kHTermBytes + kHGroups * 4) / 16;
      for (int j = tid; j < n16; j += kComputeThreads)
        reinterpret_cast<uint4*>(hbs)[j] = __ldcg(reinterpret_cast<const uint4*>(a.h) + j);
      csync();
      trace(12);
    }
    if (i >= s.bDN) break;

    const int slot = i % S;
    const uint8_t* buf = ring + (size_t)slot * a.slot_bytes;
    const long long c0 = dclk();
    mbar_wait(&full[slot], uint32_t(i / S) & 1u, a.status);
    const long long c1 = dclk();
    trace_add(20, c1 - c0);
    if (i < s.nR) {
      // ---- router rows -> logits (warp per row) ---------------------------------
      const int r = s.r0 + i * s.rch, n = min(s.rch, s.r1 - r);
      if (warp < n) {
        float v[T];
        warp_row_dot<T>(reinterpret_cast<const uint4*>(buf + (size_t)warp * row_bytes), xs4, d / 8, lane, v);
        if (lane == 0)
#pragma unroll
          for (int t = 0; t < T; ++t) a.logits[(size_t)t * E + r + warp] = v[t];
      }
    } else if (i < s.bF) {
      // ---- shared gate/up features -> h_sh (warp per feature) --------------------
      const int fb = (i - s.nR) * s.fch;
      const int f = s.f0 + fb, n = min(s.fch, s.f1 - f);
      const int ff = (warp - fb % kWarps + kWarps) % kWarps;
      if (ff < n) {
        float gv[T], uv[T];
        warp_row_dot<T>(reinterpret_cast<const uint4*>(buf + (size_t)ff * row_bytes), xs4, d / 8, lane, gv);
        warp_row_dot<T>(reinterpret_cast<const uint4*>(buf + (size_t)(n + ff) * row_bytes), xs4, d / 8, lane, uv);
        if (lane == 0)
#pragma unroll
          for (int t = 0; t < T; ++t) a.h_sh[(size_t)t * I + f + ff] = silu_f(gv[t]) * uv[t];
      }
      trace_add(24, dclk() - c1);
    } else if (i < s.bGU) {
      // ---- routed gate/up tile: 8 gate + 8 up rows of one active expert -------
      // Tile jb belongs to warp group jb % kGroups; its warps split K, and
      // the group's first warp adds the 3 partials (in warp order) and writes
      // the tile's 8 features of h per slot as the B operand of the down MMA:
      // 2 e4m3 terms with one exponent for the 8 features.
      if (i == s.bF) trace(8);
      const int jb = i - s.bF, gid = warp / kGroupWarps, gw = warp - gid * kGroupWarps;
      if (gid == jb % kGroups) {
        const int gt = s.i0 + jb, ai = gt / NTg, tt = gt - ai * NTg;
        const int nt = act_n[ai];
        const int* toks = act_tok + ai * kDecodeMaxT;
        const int* slots = act_slot + ai * kDecodeMaxT;
        int boff[kPairs], foff[kPairs];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const int sb = 2 * p + (g >> 2), sc = 2 * p + (q >> 1);
          boff[p] = (sb < nt && (g & 3) < kActTerms) ? toks[sb] * KBd * kActRowKbBytes + (g & 3) * 32 + q * 8 : -1;
          foff[p] = sc < nt ? toks[sc] * KBd : -1;
        }
        float acc[kPairs][2];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) acc[p][0] = acc[p][1] = 0.0f;
        // my K-blocks gw, gw + kGroupWarps, ...: groups of kUnroll without branches (a
        // K-block past the end is clamped and weighted 0)
        for (int kb0 = gw; kb0 < KBd; kb0 += kUnroll * kGroupWarps) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int kb = kb0 + u * kGroupWarps;
            const bool ok = kb < KBd;
            const int kbc = ok ? kb : KBd - 1;
            const uint8_t* unit = buf + (size_t)kbc * kUnitBytes;
            const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
            const uint32_t sc16 = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
            const float fwl = ok ? scale_lo(sc16) : 0.0f, fwh = ok ? scale_hi(sc16) : 0.0f;
#pragma unroll
            for (int p = 0; p < kPairs; ++p) {
              const uint2 bv = boff[p] >= 0 ? *reinterpret_cast<const uint2*>(xb + boff[p] + kbc * kActRowKbBytes)
                                            : make_uint2(0u, 0u);
              const float fa = foff[p] >= 0 ? xfa[foff[p] + kbc] : 0.0f;
              float dd[4];
              mma_e4m3(dd, decode_rowlo(wv.x), decode_rowhi(wv.x), decode_rowlo(wv.y), decode_rowhi(wv.y), bv.x,
                       bv.y);
              acc[p][0] = fmaf((dd[0] + dd[1]) * fa, fwl, acc[p][0]);
              acc[p][1] = fmaf((dd[2] + dd[3]) * fa, fwh, acc[p][1]);
            }
          }
        }
        trace_add(21, dclk() - c1);
        float* gbuf = red + (size_t)(gid * 2 + ((jb / kGroups) & 1)) * kGroupWarps * kRF;
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const float v0 = acc[p][0] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][0], 1);
          const float v1 = acc[p][1] + __shfl_xor_sync(0xFFFFFFFFu, acc[p][1], 1);
          if ((q & 1) == 0) {
            gbuf[gw * kRF + p * 32 + g * 2 + (q >> 1)] = v0;        // gate row g, slot column q>>1
            gbuf[gw * kRF + p * 32 + 16 + g * 2 + (q >> 1)] = v1;   // up row g
          }
        }
        group_sync<kGroupWarps>(gid);
        if (gw == 0) {
          uint8_t* hT = reinterpret_cast<uint8_t*>(a.h);
          float* hF = reinterpret_cast<float*>(hT + (size_t)T * k * KBi * kHTermBytes);
          const int kbh = tt >> 2, grp = tt & 3;
#pragma unroll
          for (int p = 0; p < kPairs; ++p) {
            if (2 * p < nt) {
              float v = gbuf[p * 32 + lane];
#pragma unroll
              for (int w = 1; w < kGroupWarps; ++w) v += gbuf[w * kRF + p * 32 + lane];
              const float up = __shfl_down_sync(0xFFFFFFFFu, v, 16);
              const float hv = lane < 16 ? silu_f(v) * up : 0.0f;   // feature lane>>1, slot column lane&1
              float am = fabsf(hv);
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
              am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 8));
              int ex = kActZeroExp;
              uint32_t t0 = 0u, t1 = 0u;
              if (am > 0.0f) {
                ex = floor_log2(am) - 7;
                const float sv = scale2(hv, -ex);
                t0 = f32x2_to_e4m3x2(sv, 0.0f) & 0xFFu;
                t1 = f32x2_to_e4m3x2(sv - e4m3_to_f32_hw(t0), 0.0f) & 0xFFu;
              }
              const int sc = 2 * p + (lane & 1);
              if (lane < 16 && sc < nt) {
                const int sl = slots[sc];
                const size_t base = ((size_t)sl * KBi + kbh) * kHTermBytes + grp * 8 + (lane >> 1);
                hT[base] = uint8_t(t0);
                hT[base + 32] = uint8_t(t1);
                if ((lane >> 1) == 0) hF[((size_t)sl * KBi + kbh) * kHGroups + grp] = act_factor(ex, sel_w[sl]);
              }
            }
          }
        }
        trace_add(23, dclk() - c1);
      }
    } else if (i < s.bSD) {
      // ---- shared down rows of my tiles -> y accumulators (warp per row) -------
      const int r = s.t0 * kTileRows + (i - s.bGU) * s.sdch;
      const int n = min(s.sdch, (s.t0 + s.ntl) * kTileRows - r);
      for (int rr = warp; rr < n; rr += kWarps) {
        const uint4* wrow = reinterpret_cast<const uint4*>(buf + (size_t)rr * sdrow_bytes);
        float acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = 0.0f;
#pragma unroll 3
        for (int j = lane; j < I / 8; j += 32) {
          const uint4 wv = wrow[j];
#pragma unroll
          for (int t = 0; t < T; ++t) acc[t] += dot8_f32(wv, hsh + (size_t)t * I + j * 8);
        }
        const int row_local = r + rr - s.t0 * kTileRows;
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const float v = warp_sum(acc[t]);
          if (lane == 0) ysd[t * ystride + row_local] = v;
        }
      }
    } else {
      // ---- routed down units (one output tile per load) -> per-lane accumulators
      trace_add(28, 1);
      const int l = i - s.bSD, tl = l / s.nL, a0 = (l - tl * s.nL) * s.dnch, n = min(s.dnch, s.D - a0);
      if (tl != dn_tile) {
        const long long f0 = dclk();
        if (dn_tile >= 0) flush_tile(dn_tile);
        dn_tile = tl;
        trace_add(29, dclk() - f0);
      }
      // half units (one expert, half of K) per warp: half h of unit j of tile
      // tl goes to warp (2 (tl * D + a0 + j) + h) % 15, so the unit's tables are
      // read once per half and all warps take part
      const int KBh = (KBi + 1) / 2;
      for (int jh = 0; jh < 2 * n; ++jh) {
        if ((2 * (tl * s.D + a0) + jh) % kWarps != warp) continue;
        const int j = jh >> 1, kbb = (jh & 1) * KBh, kbe = min(KBi, kbb + KBh);
        const int ai = a0 + j;
        const int nt = act_n[ai];
        const int* slots = act_slot + ai * kDecodeMaxT;
        const int* toks = act_tok + ai * kDecodeMaxT;
        const uint8_t* ub = buf + (size_t)j * U_dn;
        // B columns: 4 groups of 8 features x 2 terms; lane (g, q) holds the
        // C columns of group q, so the quad sum in flush_tile adds the groups
        const int grp = g >> 1;
        int hbo[T], hfo[T], tok[T];
#pragma unroll
        for (int si = 0; si < T; ++si) {
          const int sl = si < nt ? slots[si] : 0;
          hbo[si] = sl * KBi * kHTermBytes + (g & 1) * 32 + 4 * q + (grp == (q >> 1) ? 0 : 16);
          hfo[si] = sl * KBi * kHGroups + q;
          tok[si] = si < nt ? toks[si] : -1;
        }
        const bool lo_ok = grp == (q >> 1), hi_ok = grp == 2 + (q >> 1);
        const long long k0 = dclk();
        for (int kb0 = kbb; kb0 < kbe; kb0 += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int kb = kb0 + u;
            const bool ok = kb < kbe;
            const int kc = ok ? kb : kbe - 1;
            const uint8_t* unit = ub + (size_t)kc * kUnitBytes;
            const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
            const uint32_t sc16 = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
            const float fwl = ok ? scale_lo(sc16) : 0.0f, fwh = ok ? scale_hi(sc16) : 0.0f;
            // T = 1: no branch (one slot per expert); else skip the expert's
            // missing slots
#pragma unroll
            for (int si = 0; si < T; ++si) {
              if (T > 1 && si >= nt) continue;
              const uint32_t bw = *reinterpret_cast<const uint32_t*>(hbs + hbo[si] + kc * kHTermBytes);
              const float fa = hfa[hfo[si] + kc * kHGroups];
              float dd[4];
              mma_e4m3(dd, decode_rowlo(wv.x), decode_rowhi(wv.x), decode_rowlo(wv.y), decode_rowhi(wv.y),
                       lo_ok ? bw : 0u, hi_ok ? bw : 0u);
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
        trace_add(26, dclk() - k0);
        trace_add(27, 1);
      }
    }
    if (i >= s.bSD) trace_add(25, dclk() - c1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);   // my share of load i is done
  }
  trace(13);

  if (dn_tile >= 0) flush_tile(dn_tile);
  csync();

  // y rows of my tiles: shared-down part + the warps' down partials, in warp order
  for (int j = tid; j < T * s.ntl * kTileRows; j += kComputeThreads) {
    const int t = j / (s.ntl * kTileRows), r = j - t * (s.ntl * kTileRows);
    const int tl = r / kTileRows, rr = r - tl * kTileRows;
    float v = ysd[t * ystride + r];
    if (s.D > 0)
      for (int w = 0; w < kWarps; ++w) v += dnred[((size_t)(tl * kWarps + w) * T + t) * kTileRows + rr];
    a.y[(size_t)t * d + s.t0 * kTileRows + r] = __float2bfloat16_rn(v);
  }
  csync();
  trace(14);
  trace_put(18, (unsigned long long)clock64());
#pragma unroll
  for (int z = 0; z < 12; ++z) trace_put(20 + z, (unsigned long long)tacc[z]);
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
  if (a.E > 32 * kMergeChunks || a.d > kWarps * kMaxKbPerWarp * kMxBlock) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (di.sm_count < 1 || max_tiles_per_cta(a.d, di.sm_count) > kDecodeMaxTiles) return MOE_ERR_UNSUPPORTED_SHAPE;
  uint32_t sb = uint32_t(a.d / kMxBlock) * kUnitBytes;   // one routed gate/up tile
  const uint32_t cands[4] = {uint32_t(2 * a.d), uint32_t(4 * a.d), uint32_t(2 * a.I),
                             uint32_t(a.I / kMxBlock) * kUnitBytes};
  for (uint32_t v : cands) sb = sb > v ? sb : v;         // router row, shared feature, shared-down row, down unit
  sb = align_up(sb, 128);
  const int mt = max_tiles_per_cta(a.d, di.sm_count);
  const Smem fixed = smem_plan(a.T, a.d, a.I, a.E, a.k, 0, sb, mt);
  const size_t budget = di.smem_optin > fixed.total + 1024 ? di.smem_optin - fixed.total - 1024 : 0;
  int S = int(budget / (sb + 16));
  if (S > kDecodeStageCap) S = kDecodeStageCap;
  if (S > kDecodeMaxStages) S = kDecodeMaxStages;
  if (S < 3) return MOE_ERR_UNSUPPORTED_SHAPE;
  *stages = S;
  *slot_bytes = sb;
  *smem_bytes = smem_plan(a.T, a.d, a.I, a.E, a.k, S, sb, mt).total;
  return MOE_OK;
}

template <int T>
int launch_decode_t(DecodeArgs a, uint32_t smem, const DeviceInfo& di, cudaStream_t s) {
  const Smem L = smem_plan(T, a.d, a.I, a.E, a.k, a.stages, a.slot_bytes, max_tiles_per_cta(a.d, di.sm_count));
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
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, decode_kernel<T>, a, L));
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
