// Routed-expert GEMVs over MXFP4 weights (gate/up with SwiGLU, and down):
// the W4 experts of page "3 ways to speed up MoE inference on NVIDIA DGX
// Spark", §2-§3, each run once over the tokens sorted to it (page
// "MoE-SpeQ ...", §4.2).
//
// Each work item is one 16-row tile of one active expert's matrix over the
// whole K, for one chunk of at most 8 of that expert's activation rows. The
// tile (K/32 units of 272 bytes) is fetched with one 1-D bulk copy into a ring
// of shared-memory stages; all items of a CTA are requested up front as far
// as the ring allows, so the HBM queue stays full. The chunk's activation
// terms are copied into shared memory once per (expert, chunk). Eight warps
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

constexpr int kRoutedWarps = 16;
constexpr int kPairs = 4;                 // activation-row pairs per MMA pass
constexpr int kChunk = 2 * kPairs;        // activation rows staged in shared memory at a time
constexpr int kRoutedThreads = kRoutedWarps * 32;
constexpr int kMaxActive = 1024;          // E <= 1024

// Work items are (active expert a, chunk c of its rows, tile), ordered
// expert-major, then chunk, then tile, and split into contiguous ranges per
// CTA. A CTA copies a chunk's activation terms (at most 8 rows) into shared
// memory once and reuses them for every tile of that (expert, chunk); an
// expert with more than 8 rows reads its weight tiles once per chunk (the
// later reads mostly hit L2).
struct RoutedSmem {
  uint32_t ring, bst, est, red, cofs, bars, total;
};
__host__ __device__ inline RoutedSmem routed_smem(int stages, uint32_t item_bytes, int KB) {
  RoutedSmem m{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = (at + align - 1) / align * align;
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  m.ring = take(uint32_t(stages) * item_bytes, 128);
  m.bst = take(uint32_t(kChunk * KB * kActRowKbBytes), 16);
  m.est = take(uint32_t(kChunk * KB * 4), 16);
  m.red = take(uint32_t(kRoutedWarps * kPairs * 32 * 2 * 4), 16);
  m.cofs = take(uint32_t((kMaxActive + 1) * 4), 16);
  m.bars = take(uint32_t(stages * 8), 8);
  m.total = at;
  return m;
}

// Weight scale byte -> 2^(s-127) as fp32 (s = 0 gives 0, s = 255 gives +inf).
__device__ __forceinline__ float wscale_lo(uint32_t sc16) { return __uint_as_float((sc16 << 23) & 0x7F800000u); }
__device__ __forceinline__ float wscale_hi(uint32_t sc16) { return __uint_as_float((sc16 << 15) & 0x7F800000u); }

// One warp's K-blocks (kb_first, kb_first + kb_step, ...) of one tile against NP pairs of
// staged activation rows. acc[p][0] / [1]: rows g / g+8 for the columns of
// this lane. No branch inside a group of K-blocks (a block past the end is
// clamped and weighted 0), so the MMAs of a group overlap.
template <int NP>
__device__ __forceinline__ void routed_tile(const uint8_t* st, const uint8_t* bst, const float* est, int KB,
                                            int nr, bool ok, int kb_first, int kb_step, int lane,
                                            float (&acc)[kPairs][2]) {
  const int g = lane >> 2, q = lane & 3;
  int boff[NP], erow[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int sb = 2 * p + (g >> 2), sc = 2 * p + (q >> 1);
    boff[p] = (ok && sb < nr && (g & 3) < kActTerms) ? sb * KB * kActRowKbBytes + (g & 3) * 32 + q * 8 : -1;
    erow[p] = sc * KB;   // rows past nr hold factor 0
  }
#pragma unroll
  for (int p = 0; p < kPairs; ++p) acc[p][0] = acc[p][1] = 0.0f;
  constexpr int kGroup = 5;
  for (int kb0 = kb_first; kb0 < KB; kb0 += kGroup * kb_step) {
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int kb = kb0 + u * kb_step;
      const bool in = kb < KB;
      const int kc = in ? kb : KB - 1;
      const uint8_t* unit = st + (size_t)kc * kUnitBytes;
      const AFrag af = load_afrag(unit, g, q);
      const uint32_t sc16 = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
      const float fwl = in ? wscale_lo(sc16) : 0.0f, fwh = in ? wscale_hi(sc16) : 0.0f;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const uint2 bv = boff[p] >= 0 ? *reinterpret_cast<const uint2*>(bst + boff[p] + kc * kActRowKbBytes)
                                      : make_uint2(0u, 0u);
        const float fa = est[erow[p] + kc];
        float d[4];
        mma_e4m3(d, af.a0, af.a1, af.a2, af.a3, bv.x, bv.y);
        acc[p][0] = fmaf((d[0] + d[1]) * fa, fwl, acc[p][0]);
        acc[p][1] = fmaf((d[2] + d[3]) * fa, fwh, acc[p][1]);
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kRoutedThreads, 1)
routed_kernel(RoutedArgs a, int stages, uint32_t item_bytes, int tpi, RoutedSmem L) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem + L.ring;
  uint8_t* bst = smem + L.bst;                                   // [kChunk][KB][96]
  float* est = reinterpret_cast<float*>(smem + L.est);           // [kChunk][KB] 2^(e+6) per block
  float* red = reinterpret_cast<float*>(smem + L.red);
  int* cofs = reinterpret_cast<int*>(smem + L.cofs);             // chunk offsets per active expert
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int D = *a.n_active;
  const int KB = a.KB;

  // cofs[i] = sum over active experts j < i of ceil(rows_j / kChunk)
  {
    constexpr int kPer = kMaxActive / kRoutedThreads;   // 4 experts per thread
    int v[kPer], run = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int ai = tid * kPer + r;
      int c = 0;
      if (ai < D) {
        const int e = a.active[ai];
        c = (a.offsets[e + 1] - a.offsets[e] + kChunk - 1) / kChunk;
      }
      v[r] = run;
      run += c;
    }
    // exclusive scan of the per-thread totals
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    int* wsum = reinterpret_cast<int*>(red);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = incl - run;
    for (int w = 0; w < warp; ++w) base += wsum[w];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int ai = tid * kPer + r;
      if (ai < D) cofs[ai] = base + v[r];
    }
    if (tid == kRoutedThreads - 1) cofs[D] = base + run;   // total number of chunks
    __syncthreads();
  }
  const int n_chunks = cofs[D];
  // an item is a group of tpi consecutive tiles (one bulk copy); each tile
  // gets wpt warps, which split its K-blocks
  const int n_groups = (a.n_tiles + tpi - 1) / tpi, wpt = kRoutedWarps / tpi;
  const uint32_t tile_bytes = uint32_t(KB) * kUnitBytes;
  const long long n_items = (long long)n_chunks * n_groups;
  const int lo = int((long long)blockIdx.x * n_items / gridDim.x);
  const int hi = int((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  if (lo >= hi) return;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  // active expert of global chunk gc (cofs is non-decreasing)
  auto expert_of = [&](int gc) {
    int l = 0, h = D - 1;
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (cofs[m] <= gc) l = m; else h = m - 1;
    }
    return l;
  };
  auto issue = [&](int item, int s) {
    const int gc = item / n_groups, tile0 = (item - gc * n_groups) * tpi;
    const uint32_t bytes = uint32_t(min(tpi, a.n_tiles - tile0)) * tile_bytes;
    const int e = a.active[expert_of(gc)];
    const uint8_t* src = a.w + (uint64_t)e * a.mat_bytes + (uint64_t)tile0 * tile_bytes;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_g2s(ring + (size_t)s * item_bytes, src, bytes, &full[s]);
  };
  if (tid == 0)
    for (int s = 0; s < stages && lo + s < hi; ++s) issue(lo + s, s);

  int staged = -1;   // global chunk whose activation rows are in bst / est
  int pos0 = 0, nr = 0;
  for (int it = lo; it < hi; ++it) {
    const int rel = it - lo, s = rel % stages;
    const int gc = it / n_groups, tile0 = (it - gc * n_groups) * tpi;
    const int nti = min(tpi, a.n_tiles - tile0);   // tiles in this item
    const int tw = warp / wpt;                      // my tile within the item
    if (gc != staged) {
      // ---- this chunk's activation rows -> shared memory -------------------
      const int ai = expert_of(gc), e = a.active[ai];
      const int c = gc - cofs[ai];
      const int n = a.offsets[e + 1] - a.offsets[e];
      pos0 = a.offsets[e] + c * kChunk;
      nr = min(kChunk, n - c * kChunk);
      const int per_row = KB * kActRowKbBytes / 16;
      for (int j = tid; j < nr * per_row; j += kRoutedThreads) {
        const int r = j / per_row, o = j - r * per_row;
        const int row = a.act_by_token ? a.perm[pos0 + r] / a.k : pos0 + r;
        reinterpret_cast<uint4*>(bst)[r * per_row + o] =
            __ldg(reinterpret_cast<const uint4*>(a.act_b + (size_t)row * KB * kActRowKbBytes) + o);
      }
      for (int j = tid; j < kChunk * KB; j += kRoutedThreads) {
        const int r = j / KB, kb = j - r * KB;
        float f = 0.0f;   // rows past the chunk, and all-zero blocks, weigh 0
        if (r < nr) {
          const int row = a.act_by_token ? a.perm[pos0 + r] / a.k : pos0 + r;
          const int ev = __ldg(a.act_e + (size_t)row * KB + kb);
          if (ev != kActZeroExp) f = scale2(1.0f, ev + 6);
        }
        est[j] = f;
      }
      staged = gc;
      __syncthreads();
    }
    // block-uniform, so every __syncthreads below is reached by all threads
    const bool ok = __syncthreads_and(mbar_wait(&full[s], uint32_t(rel / stages) & 1u, a.status));
    const uint8_t* st = ring + (size_t)s * item_bytes + (size_t)tw * tile_bytes;
    float acc[kPairs][2];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) acc[p][0] = acc[p][1] = 0.0f;
    const int np = (nr + 1) / 2, kbf = warp - tw * wpt;
    if (tw < nti) {
      if (np == 1) routed_tile<1>(st, bst, est, KB, nr, ok, kbf, wpt, lane, acc);
      else if (np == 2) routed_tile<2>(st, bst, est, KB, nr, ok, kbf, wpt, lane, acc);
      else routed_tile<kPairs>(st, bst, est, KB, nr, ok, kbf, wpt, lane, acc);
    }
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      red[((warp * kPairs + p) * 32 + lane) * 2 + 0] = acc[p][0];
      red[((warp * kPairs + p) * 32 + lane) * 2 + 1] = acc[p][1];
    }
    __syncthreads();
    if (kbf == 0 && tw < nti) {
      // the first warp of each tile adds the tile's wpt partials in warp order
      const int tile = tile0 + tw;
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        if (2 * p >= nr) break;
        float v0 = 0.0f, v1 = 0.0f;
        for (int w = warp; w < warp + wpt; ++w) {
          v0 += red[((w * kPairs + p) * 32 + lane) * 2 + 0];
          v1 += red[((w * kPairs + p) * 32 + lane) * 2 + 1];
        }
        v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);   // terms 0,1 + terms 2,3
        v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
        const int sc = 2 * p + (q >> 1);
        if ((q & 1) == 0 && sc < nr) {
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
    __syncthreads();   // ring slot, partials and staged rows are free again
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
  // warps per tile: the largest power of two up to 16 that leaves each warp
  // about 5 K-blocks; the rest of the 16 warps take further tiles of the item
  int wpt = kRoutedWarps;
  while (wpt > 1 && a.KB < 5 * wpt) wpt >>= 1;
  const int tpi = kRoutedWarps / wpt;
  const uint32_t item_bytes = uint32_t(tpi) * uint32_t(a.KB) * kUnitBytes;
  const RoutedSmem fixed = routed_smem(0, item_bytes, a.KB);
  const size_t budget = (di.smem_optin > fixed.total + 4096 ? di.smem_optin - fixed.total - 4096 : 0);
  int stages = int(budget / (item_bytes + 8));
  if (stages > 16) stages = 16;
  if (stages < 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  const RoutedSmem L = routed_smem(stages, item_bytes, a.KB);
  int grid = di.sm_count;
  if (a.max_items < grid) grid = a.max_items > 0 ? a.max_items : 1;
  if (mode == kModeGateUp) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(routed_kernel<kModeGateUp>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)));
    routed_kernel<kModeGateUp><<<grid, kRoutedThreads, L.total, s>>>(a, stages, item_bytes, tpi, L);
  } else {
    MOE_CUDA_TRY(cudaFuncSetAttribute(routed_kernel<kModeDown>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)));
    routed_kernel<kModeDown><<<grid, kRoutedThreads, L.total, s>>>(a, stages, item_bytes, tpi, L);
  }
  return launch_status();
}

}  // namespace moe
