// Routed-expert GEMMs on the 5th-generation tensor cores (tcgen05), for large
// token counts (prefill): gate/up with SwiGLU, and down.
//
// Work items are (active expert, block of 128 weight rows = 8 packed 16-row
// tiles, block of that expert's rows / tokens), split into contiguous ranges
// per CTA (one CTA per SM, persistent). Along K an item goes in slices of two
// 32-wide K-blocks:
//   * a producer thread streams the slice's packed MXFP4 bytes (8 tiles x 2
//     units of 272 bytes) into a ring of shared-memory slots with 1-D bulk
//     copies, several slices ahead;
//   * the 8 warps decode them (one tile each) into bf16 with the E8M0 block
//     scale applied (exact), in the K-major no-swizzle layout the MMA reads
//     (8-row x 16-byte core matrices);
//   * the slice of the activation rows (bf16 x; for the down projection h as
//     two bf16 terms, hi and lo, in separate columns) is copied into the same
//     layout with cp.async two slices ahead;
//   * one thread issues the slice's tcgen05.mma (kind::f16, M = 128, N = the
//     item's column count, K = 16 each) into an fp32 accumulator in tensor
//     memory and commits them to an mbarrier.
// Slices use four shared-memory buffers in turn, so the loads and the decode
// of the next slices overlap the MMAs of the previous ones. At the end of an
// item the accumulator is read back with tcgen05.ld: SwiGLU of the gate and up
// rows of a tile (they sit 8 TMEM lanes apart), written as bf16 hi and lo
// terms for the down pass; or, for the down pass, the sum of the hi and lo
// columns.
#include <cuda_runtime.h>
#ifdef MOE_UMMA_TRACE
#include <cstdio>
#endif

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kUWarps = 8;
constexpr int kUThreads = kUWarps * 32;
constexpr int kURows = 128;                 // weight rows per item (MMA M)
constexpr int kUTiles = kURows / kTileRows; // packed tiles per item (one per warp)
constexpr int kUSliceKb = 2;                // 32-wide K-blocks per slice
constexpr int kUSliceK = kUSliceKb * kMxBlock;
constexpr int kUBuf = 4;                    // operand buffers (slice s uses s % 4)
constexpr int kURing = 10;                  // packed weight slices in flight
constexpr int kUCols = 128;                 // TMEM columns = largest MMA N
constexpr int kUMaxActive = 1024;
constexpr uint32_t kURawBytes = kUTiles * kUSliceKb * kUnitBytes;   // one slice of packed weights
constexpr uint32_t kUABytes = kURows * kUSliceK * 2;                 // one slice of bf16 weights
constexpr uint32_t kUBBytes = kUCols * kUSliceK * 2;                 // one slice of bf16 activations

struct UmmaSmem {
  uint32_t ring, a, b, iofs, bars, tslot, total;
};
__host__ __device__ inline UmmaSmem umma_smem() {
  UmmaSmem m{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = (at + align - 1) / align * align;
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  m.ring = take(kURing * kURawBytes, 128);
  m.a = take(kUBuf * kUABytes, 1024);
  m.b = take(kUBuf * kUBBytes, 1024);
  m.iofs = take((kUMaxActive + 1) * 4, 16);
  m.bars = take((kURing + kUBuf) * 8, 8);
  m.tslot = take(16, 16);
  m.total = at;
  return m;
}

// byte offset of element (row r, k) in a K-major no-swizzle operand of `rows`
// rows: core matrix (k / 8, r / 8) at ((k / 8) * rows / 8 + r / 8) * 128
__device__ __forceinline__ uint32_t kmajor_off(int r, int k, int rows) {
  return (uint32_t)(((k >> 3) * (rows >> 3) + (r >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// four e4m3 bytes (each 2^-6 x an E2M1 value) times f -> four bf16 (exact
// when f is a power of two and the result is in range)
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t v, float f) {
  uint32_t h01, h23;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n"
      " cvt.rn.f16x2.e4m3x2 %1, hi;\n}\n"
      : "=r"(h01), "=r"(h23)
      : "r"(v));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  const __nv_bfloat162 p = __floats2bfloat162_rn(a.x * f, a.y * f);
  const __nv_bfloat162 q = __floats2bfloat162_rn(b.x * f, b.y * f);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&p), *reinterpret_cast<const uint32_t*>(&q));
}

// 16-byte asynchronous global -> shared copy; zero-filled when !valid
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int MODE>
__global__ void __launch_bounds__(kUThreads, 1) umma_routed_kernel(RoutedArgs a, UmmaSmem L) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem + L.ring;
  uint8_t* abuf = smem + L.a;
  uint8_t* bbuf = smem + L.b;
  int* iofs = reinterpret_cast<int*>(smem + L.iofs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* mdone = full + kURing;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int D = *a.n_active, KB = a.KB, K = KB * kMxBlock;
  const int nrb = (a.n_tiles + kUTiles - 1) / kUTiles;
  // tokens per item: gate/up columns are tokens; down columns are hi and lo terms of h
  constexpr int kNTok = MODE == kModeGateUp ? kUCols : kUCols / 2;
  const int ns = (KB + kUSliceKb - 1) / kUSliceKb;   // slices per item

  // iofs[i] = items of the active experts before i (nrb per block of kNTok rows)
  {
    constexpr int kPer = kUMaxActive / kUThreads;
    int v[kPer], run = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int ai = tid * kPer + r;
      int c = 0;
      if (ai < D) {
        const int e = a.active[ai];
        c = nrb * ((a.offsets[e + 1] - a.offsets[e] + kNTok - 1) / kNTok);
      }
      v[r] = run;
      run += c;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    int* wsum = reinterpret_cast<int*>(bbuf);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = incl - run;
    for (int w = 0; w < warp; ++w) base += wsum[w];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int ai = tid * kPer + r;
      if (ai < D) iofs[ai] = base + v[r];
    }
    if (tid == kUThreads - 1) iofs[D] = base + run;
    __syncthreads();
  }
  const int n_items = iofs[D];
  const int lo = int((long long)blockIdx.x * n_items / gridDim.x);
  const int hi = int((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  if (lo >= hi) return;
  const int n_stream = (hi - lo) * ns;   // my slices, item after item

  if (tid == 0) {
    for (int i = 0; i < kURing + kUBuf; ++i) mbar_init(&full[i], 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tslot, kUCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // active expert of item it (iofs is strictly increasing)
  auto expert_of = [&](int it) {
    int l = 0, h = D - 1;
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (iofs[m] <= it) l = m; else h = m - 1;
    }
    return l;
  };
  // packed bytes of stream slice p -> ring slot p % kURing (producer thread,
  // which keeps the item it last looked up)
  int pr_it = -1, pr_rb = 0, pr_nt = 0;
  const uint8_t* pr_wm = nullptr;
  auto issue = [&](int p) {
    const int it = lo + p / ns, sl = p - (p / ns) * ns;
    if (it != pr_it) {
      const int ai = expert_of(it), rem = it - iofs[ai];
      pr_it = it;
      pr_rb = rem % nrb;
      pr_nt = min(kUTiles, a.n_tiles - pr_rb * kUTiles);
      pr_wm = a.w + (uint64_t)a.active[ai] * a.mat_bytes + (uint64_t)pr_rb * kUTiles * KB * kUnitBytes;
    }
    const int kb0 = sl * kUSliceKb, nkb = min(kUSliceKb, KB - kb0);
    uint8_t* dst = ring + (size_t)(p % kURing) * kURawBytes;
    uint64_t* bar = &full[p % kURing];
    mbar_arrive_expect_tx(bar, uint32_t(pr_nt * nkb) * kUnitBytes);
    for (int t = 0; t < pr_nt; ++t)
      bulk_g2s(dst + (size_t)t * kUSliceKb * kUnitBytes, pr_wm + ((uint64_t)t * KB + kb0) * kUnitBytes,
               uint32_t(nkb) * kUnitBytes, bar);
  };
  constexpr int kProducer = 32;   // lane 0 of warp 1: thread 0 issues the MMAs
  if (tid == kProducer)
    for (int p = 0; p < kURing && p < n_stream; ++p) issue(p);

  // item of stream slice p: expert row block, first row (slot), rows, MMA N
  struct Item {
    int rb, pos0, ntok, nmma, n16;
  };
  auto item_of = [&](int p) {
    Item f;
    const int it = lo + p / ns, ai = expert_of(it), rem = it - iofs[ai];
    const int e = a.active[ai], tb = rem / nrb, n_e = a.offsets[e + 1] - a.offsets[e];
    f.rb = rem % nrb;
    f.pos0 = a.offsets[e] + tb * kNTok;
    f.ntok = min(kNTok, n_e - tb * kNTok);
    if (MODE == kModeGateUp) {
      f.n16 = 0;
      f.nmma = (f.ntok + 15) & ~15;
    } else {
      f.n16 = (f.ntok + 7) & ~7;   // hi columns [0, n16), lo columns [n16, 2 n16)
      f.nmma = 2 * f.n16;
    }
    return f;
  };
  // activation rows of stream slice p -> operand buffer p % kUBuf (one
  // cp.async group per call, empty past the stream). Chunk j = 8 r + c is row
  // r, 16-byte chunk c; a thread's rows are the same in every slice of an
  // item, so their source rows are looked up once per item.
  constexpr int kRowsPerThread = kUCols * 8 / kUThreads;
  int b_it = -1;
  Item b_f{};
  int b_row[kRowsPerThread];
  auto issue_b = [&](int p) {
    if (p < n_stream) {
      const int it = lo + p / ns;
      if (it != b_it) {
        b_it = it;
        b_f = item_of(p);
#pragma unroll
        for (int m = 0; m < kRowsPerThread; ++m) {
          const int r = (tid + m * kUThreads) >> 3;
          b_row[m] = r < b_f.ntok ? (MODE == kModeGateUp ? a.perm[b_f.pos0 + r] / a.k : b_f.pos0 + r) : 0;
        }
      }
      const int kb0 = (p % ns) * kUSliceKb, nc = min(kUSliceKb, KB - kb0) * kMxBlock / 8;
      uint8_t* bb = bbuf + (size_t)(p % kUBuf) * kUBBytes;
      const __nv_bfloat16* src0 = static_cast<const __nv_bfloat16*>(a.act_raw);
      const __nv_bfloat16* src1 = static_cast<const __nv_bfloat16*>(a.act_raw2);
      const int nrow = MODE == kModeGateUp ? b_f.nmma : b_f.n16;
#pragma unroll
      for (int m = 0; m < kRowsPerThread; ++m) {
        const int j = tid + m * kUThreads, r = j >> 3, c = j & 7;
        if (r < nrow && c < nc) {
          const bool valid = r < b_f.ntok;
          const size_t o = (size_t)b_row[m] * K + kb0 * kMxBlock + c * 8;
          cp_async16(bb + kmajor_off(r, c * 8, b_f.nmma), src0 + o, valid);
          if (MODE == kModeDown) cp_async16(bb + kmajor_off(b_f.n16 + r, c * 8, b_f.nmma), src1 + o, valid);
        }
      }
    }
    cp_async_commit();
  };
  issue_b(0);
  issue_b(1);

  Item cur{};
#ifdef MOE_UMMA_TRACE
  long long tt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  long long tm[3] = {0, 0, 0};
  long long tc0 = clock64();
#define UT(i) do { const long long _t = clock64(); tt[i] += _t - tc0; tc0 = _t; } while (0)
#else
#define UT(i) do { } while (0)
#endif
  for (int p = 0; p < n_stream; ++p) {
    const int sl = p % ns, buf = p % kUBuf;
    if (sl == 0) cur = item_of(p);
    UT(7);
    // buffer (p + 2) % 4 was last read by the MMAs of slice p - 2
    if (p >= 2) mbar_wait(&mdone[(p + 2) % kUBuf], uint32_t((p - 2) / kUBuf) & 1u, a.status);
    UT(0);
    issue_b(p + 2);
    UT(1);
    const int kb0 = sl * kUSliceKb, nkb = min(kUSliceKb, KB - kb0);
    uint8_t* ab = abuf + (size_t)buf * kUABytes;
    uint8_t* bb = bbuf + (size_t)buf * kUBBytes;

    // ---- weights: packed MXFP4 -> bf16 (warp w decodes tile w) ---------------
    mbar_wait(&full[p % kURing], uint32_t(p / kURing) & 1u, a.status);
    UT(2);
    {
      const int t = warp, tile = cur.rb * kUTiles + t;
      const uint8_t* raw = ring + (size_t)(p % kURing) * kURawBytes + (size_t)t * kUSliceKb * kUnitBytes;
#pragma unroll
      for (int u = 0; u < kUSliceKb; ++u) {
        const int r0 = t * kTileRows + g, r1 = r0 + 8;
        uint2 c0 = make_uint2(0u, 0u), c1 = c0, c2 = c0, c3 = c0;
        if (u < nkb && tile < a.n_tiles) {
          const uint8_t* unit = raw + (size_t)u * kUnitBytes;
          const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
          const uint32_t sc16 = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
          // weights were decoded as 2^-6 x value: scale by 2^(s-127) * 64
          const float flo = __uint_as_float((sc16 << 23) & 0x7F800000u) * 64.0f;
          const float fhi = __uint_as_float((sc16 << 15) & 0x7F800000u) * 64.0f;
          c0 = e4m3x4_to_bf16x4(decode_rowlo(wv.x), flo);   // row g,   k 4q .. 4q+3
          c1 = e4m3x4_to_bf16x4(decode_rowhi(wv.x), fhi);   // row g+8
          c2 = e4m3x4_to_bf16x4(decode_rowlo(wv.y), flo);   // row g,   k 16+4q ..
          c3 = e4m3x4_to_bf16x4(decode_rowhi(wv.y), fhi);   // row g+8
        }
        const int k0 = u * kMxBlock + 4 * q;
        *reinterpret_cast<uint2*>(ab + kmajor_off(r0, k0, kURows)) = c0;
        *reinterpret_cast<uint2*>(ab + kmajor_off(r1, k0, kURows)) = c1;
        *reinterpret_cast<uint2*>(ab + kmajor_off(r0, k0 + 16, kURows)) = c2;
        *reinterpret_cast<uint2*>(ab + kmajor_off(r1, k0 + 16, kURows)) = c3;
      }
    }
    UT(3);
    cp_async_wait<2>();   // this slice's activation rows (issued two slices ago) have landed
    fence_async_smem();
    __syncthreads();   // operands written; ring slot p % kURing is free again
    UT(4);
    if (tid == kProducer && p + kURing < n_stream) issue(p + kURing);
    if (tid == 0) {
      // ---- the slice's MMAs ---------------------------------------------------
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(kURows, cur.nmma);
      const uint32_t a_lbo = (kURows / 8) * 128, b_lbo = uint32_t(cur.nmma / 8) * 128;
#ifdef MOE_UMMA_TRACE
      const long long m0 = clock64();
#endif
      for (int kk = 0; kk < nkb * 2; ++kk) {
        const uint64_t ad = umma_desc(smem_addr(ab) + 2 * kk * a_lbo, a_lbo, 128);
        const uint64_t bd = umma_desc(smem_addr(bb) + 2 * kk * b_lbo, b_lbo, 128);
        umma_bf16(tmem, ad, bd, idesc, sl > 0 || kk > 0);
#ifdef MOE_UMMA_TRACE
        if (kk == 0) tm[0] += clock64() - m0;
#endif
      }
#ifdef MOE_UMMA_TRACE
      const long long m1 = clock64();
      tm[1] += m1 - m0;
#endif
      umma_commit(&mdone[buf]);
#ifdef MOE_UMMA_TRACE
      tm[2] += clock64() - m1;
#endif
    }
    UT(5);
    if (sl == ns - 1) {
      // ---- item done: accumulator -> outputs ------------------------------------
      mbar_wait(&mdone[buf], uint32_t(p / kUBuf) & 1u, a.status);
      tc_fence_after();
      const int quarter = warp & 3, half = warp >> 2;
      const int row = quarter * 32 + lane;   // TMEM lane = weight row of the item
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      if (MODE == kModeGateUp) {
        // rows 16t .. 16t+7: gate of features 8 (rb*8 + t) + 0..7; rows +8: up.
        // h goes out as bf16 terms: hi = bf16(h), lo = bf16(h - hi)
        __nv_bfloat16* hhi = reinterpret_cast<__nv_bfloat16*>(a.out);
        __nv_bfloat16* hlo = hhi + (size_t)a.n_rows * a.out_ld;
        const int t = row >> 4, r16 = row & 15, tile = cur.rb * kUTiles + t;
        const int f = tile * 8 + (r16 & 7);
        for (int c0 = half * 8; c0 < cur.nmma; c0 += 16) {
          uint32_t v[8];
          tmem_ld8(trow + c0, v);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float gv = __uint_as_float(v[j]);
            const float uv = __shfl_down_sync(0xFFFFFFFFu, gv, 8);
            if (r16 < 8 && tile < a.n_tiles && c0 + j < cur.ntok) {
              const float h = silu_f(gv) * uv;
              const __nv_bfloat16 hb = __float2bfloat16_rn(h);
              const size_t o = (size_t)(cur.pos0 + c0 + j) * a.out_ld + f;
              hhi[o] = hb;
              hlo[o] = __float2bfloat16_rn(h - __bfloat162float(hb));
            }
          }
        }
      } else {
        const int r = cur.rb * kURows + row;   // output feature
        for (int c0 = half * 8; c0 < cur.n16; c0 += 16) {
          uint32_t vh[8], vl[8];
          tmem_ld8(trow + c0, vh);
          tmem_ld8(trow + cur.n16 + c0, vl);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (r < a.n_tiles * kTileRows && c0 + j < cur.ntok)
              a.out[(size_t)(cur.pos0 + c0 + j) * a.out_ld + r] = __uint_as_float(vh[j]) + __uint_as_float(vl[j]);
        }
      }
      tc_fence_before();
      __syncthreads();   // accumulator read; the next item may overwrite it
      tc_fence_after();
      UT(6);
    }
  }
  cp_async_wait<0>();
#ifdef MOE_UMMA_TRACE
  if (blockIdx.x == 0 && tid == 0)
    printf("umma mode %d: %d slices; cycles per slice: mdone %lld, issue_b %lld, full %lld, decode %lld, "
           "bwait+sync %lld, mma issue %lld, epilogue %lld, other %lld\n",
           MODE, n_stream, tt[0] / n_stream, tt[1] / n_stream, tt[2] / n_stream, tt[3] / n_stream,
           tt[4] / n_stream, tt[5] / n_stream, tt[6] / n_stream, tt[7] / n_stream);
  if (blockIdx.x == 0 && tid == 0)
    printf("  thread 0 per slice: first MMA %lld, all MMAs %lld, commit %lld\n", tm[0] / n_stream, tm[1] / n_stream,
           tm[2] / n_stream);
#endif
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kUCols);
}

}  // namespace

int launch_umma_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s) {
  const UmmaSmem L = umma_smem();
  if (L.total > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int grid = di.sm_count;
  if (mode == kModeGateUp) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(L.total)));
    umma_routed_kernel<kModeGateUp><<<grid, kUThreads, L.total, s>>>(a, L);
  } else {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(L.total)));
    umma_routed_kernel<kModeDown><<<grid, kUThreads, L.total, s>>>(a, L);
  }
  return launch_status();
}

}  // namespace moe
