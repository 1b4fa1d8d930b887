// Routed-expert GEMMs on the 5th-generation tensor cores (tcgen05), for large
// token counts (prefill): gate/up with SwiGLU, and down.
//
// Work items are (active expert, block of 128 weight rows = 8 packed 16-row
// tiles, block of that expert's rows / tokens), split into contiguous ranges
// per CTA (one CTA per SM, persistent). Along K an item goes in slices of two
// 32-wide K-blocks. The CTA is a pipeline of warp roles that meet only at
// mbarriers (no block-wide barrier per slice):
//   * producer (one thread): 1-D bulk copies of the packed MXFP4 bytes of a
//     chunk of 4 slices (8 tiles x 8 units of 272 bytes; one copy per tile,
//     since small copies are issued too slowly) into a ring of raw slots.
//     The ring is too small to cover the HBM latency on its own, so whole
//     items are also prefetched into L2 about 8 chunks ahead;
//   * 16 decode warps (two per tile): raw slot -> bf16 with the E8M0 block
//     scale applied (exact, integer and bf16-multiply instructions only), in
//     the K-major 128-byte-swizzled operand layout the MMA reads;
//   * 4 loader warps: the slice of the activation rows (bf16 x gathered by
//     token; for the down projection h as two bf16 terms, hi and lo, in
//     separate columns) copied with cp.async into the same layout; a loader
//     announces slice p once its copies have landed (it waits for them two
//     slices later) and it has made them visible to the async proxy;
//   * MMA (one thread): tcgen05.mma kind::f16, M = 128, N = the item's column
//     count, K = 16, into one of two fp32 accumulators in tensor memory; each
//     slice's MMAs are committed to the barrier that frees its operand stage,
//     the item's last slice also to the accumulator's "full" barrier;
//   * 4 epilogue warps (one per 32-lane quarter of tensor memory): tcgen05.ld,
//     then SwiGLU of the gate and up rows of a tile (8 lanes apart) written as
//     bf16 hi and lo terms, or for the down pass the sum of the hi and lo
//     columns; then the accumulator is released to the next item but one.
// Every wait is bounded; a timeout sets MOE_DEV_TIMEOUT and an abort flag that
// ends the other roles' waits at once, and the kernel drains its own copies
// and MMAs before it frees tensor memory and returns.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kURows = 128;                  // weight rows per item (MMA M)
constexpr int kUTiles = kURows / kTileRows;  // packed tiles per item (one per decode warp)
constexpr int kUSliceKb = 2;                 // 32-wide K-blocks per slice
constexpr int kUSliceK = kUSliceKb * kMxBlock;
constexpr int kUStages = 5;                  // operand stages (bf16 weights + activations)
constexpr int kUChunk = 4;                   // slices per raw weight copy
constexpr int kURing = 3;                    // raw weight chunks in flight
constexpr int kUPrefetchChunks = 8;          // weights prefetched into L2 about this many chunks ahead
constexpr int kULag = 2;                     // activation slices a loader keeps in flight
static_assert(kUStages > kULag, "a loader announces slice p - kULag only after it has claimed slice p's stage");
constexpr int kUAcc = 2;                     // accumulators in tensor memory
constexpr int kUCols = 128;                  // columns per accumulator = largest MMA N
constexpr int kUMaxActive = 1024;
constexpr int kUTable = 256;                 // items per CTA with a precomputed table entry
constexpr uint32_t kUTileChunk = kUChunk * kUSliceKb * kUnitBytes;   // one tile's part of a chunk
constexpr uint32_t kURawBytes = kUTiles * kUTileChunk;                  // one chunk of packed weights
constexpr uint32_t kUABytes = kURows * kUSliceK * 2;                 // one slice of bf16 weights
constexpr uint32_t kUBBytes = kUCols * kUSliceK * 2;                 // one slice of bf16 activations

// warp roles
constexpr int kWProducer = 0, kWMma = 1, kWEpi = 2, kNEpi = 4, kWLoad = kWEpi + kNEpi, kNLoad = 4,
              kWDec = kWLoad + kNLoad, kDecPerTile = 2, kNDec = kUTiles * kDecPerTile;
constexpr int kUBlock = (kWDec + kNDec) * 32;
constexpr int kScanThreads = 256;

struct UmmaSmem {
  uint32_t ring, a, b, iofs, itab, bars, misc, total;
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
  m.a = take(kUStages * kUABytes, 1024);
  m.b = take(kUStages * kUBBytes, 1024);
  m.iofs = take((kUMaxActive + 1) * 4, 16);
  m.itab = take(kUTable * 16, 16);
  m.bars = take((2 * kURing + 3 * kUStages + 2 * kUAcc) * 8, 8);
  m.misc = take(16, 16);   // tensor-memory address, abort flag
  m.total = at + 1024;     // slack: the swizzled buffers are aligned to 1024 in the shared window
  return m;
}

// byte offset of element (row r, k < 64) in a K-major operand with 128-byte
// swizzle: row r in atom r / 8 (1024 bytes each), line r % 8 (128 bytes), its
// 16-byte chunk k / 8 stored at chunk (k / 8) ^ (r % 8)
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// E2M1 -> bf16 without conversion instructions. Input: four codes in the
// byte form of decode_rowlo (sign in bit 7, the 3 magnitude bits e1 e0 m in
// bits 4..2 of each byte). The magnitude bits are moved to bf16 bits 8..6
// and the sign to bit 15: that bf16 number is the E2M1 value times 2^-126
// (the E2M1 subnormal 0.5 lands on the bf16 subnormal 2^-127). One exact bf16
// multiply by 2^(s-1) then gives value * 2^(s-127); block scales s > 128
// (2^(s-1) not a bf16) take a second multiply.
__device__ __forceinline__ uint32_t e2m1_pair_raw(uint32_t b, uint32_t sel) {
  const uint32_t p = __byte_perm(b, 0u, sel);   // two code bytes into the high bytes of the halves
  return (p & 0x80008000u) | ((p >> 4) & 0x01C001C0u);
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r =
      __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
// the two factors of block scale s (E8M0), as bf16 pairs: 2^(min(s,128)-1)
// and 2^(s-min(s,128))
__device__ __forceinline__ uint32_t scale_f1(uint32_t s) { return ((min(s, 128u) + 126u) << 7) * 0x10001u; }
__device__ __forceinline__ uint32_t scale_f2(uint32_t s) { return ((s - min(s, 128u) + 127u) << 7) * 0x10001u; }
__device__ __forceinline__ uint2 e2m1x4_to_bf16x4(uint32_t b, uint32_t f1, uint32_t f2, bool big) {
  uint32_t lo = bf16x2_mul(e2m1_pair_raw(b, 0x1404u), f1);   // codes 0, 1
  uint32_t hi = bf16x2_mul(e2m1_pair_raw(b, 0x3424u), f1);   // codes 2, 3
  if (big) {
    lo = bf16x2_mul(lo, f2);
    hi = bf16x2_mul(hi, f2);
  }
  return make_uint2(lo, hi);
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

// mbarrier.try_wait with an explicit suspend-time limit: the thread sleeps in
// hardware until the phase completes or about `ns` nanoseconds pass, instead
// of spinning (a spinning warp takes issue slots from the decode warps)
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded mbarrier wait that also gives up when another role of the CTA has
// timed out (*abort set; seen within one suspend period).
__device__ __forceinline__ bool uwait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_for(bar, parity, 100000u)) {
    if (*abort) return false;
    if (clock64() - t0 > kSpinBudget) {
      *abort = 1;
      if (status) atomicOr(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

template <int MODE>
__global__ void __launch_bounds__(kUBlock, 1) umma_routed_kernel(RoutedArgs a, UmmaSmem L) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle is a function of the shared address: align the plan's base to 1024
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem + L.ring;
  uint8_t* abuf = smem + L.a;
  uint8_t* bbuf = smem + L.b;
  int* iofs = reinterpret_cast<int*>(smem + L.iofs);
  uint64_t* full_raw = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty_raw = full_raw + kURing;
  uint64_t* a_full = empty_raw + kURing;
  uint64_t* b_full = a_full + kUStages;
  uint64_t* op_empty = b_full + kUStages;
  uint64_t* acc_full = op_empty + kUStages;
  uint64_t* acc_empty = acc_full + kUAcc;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = *a.n_active, KB = a.KB, K = KB * kMxBlock;
  const int nrb = (a.n_tiles + kUTiles - 1) / kUTiles;
  // tokens per item: gate/up columns are tokens; down columns are hi and lo terms of h
  constexpr int kNTok = MODE == kModeGateUp ? kUCols : kUCols / 2;
  const int ns = (KB + kUSliceKb - 1) / kUSliceKb;   // slices per item

  // iofs[i] = items of the active experts before i (nrb per block of kNTok rows)
  {
    constexpr int kPer = kUMaxActive / kScanThreads;
    int v[kPer], run = 0, incl = 0;
    int* wsum = reinterpret_cast<int*>(bbuf);
    if (tid < kScanThreads) {
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
      incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
    }
    __syncthreads();
    if (tid < kScanThreads) {
      int base = incl - run;
      for (int w = 0; w < warp; ++w) base += wsum[w];
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int ai = tid * kPer + r;
        if (ai < D) iofs[ai] = base + v[r];
      }
      if (tid == kScanThreads - 1) iofs[D] = base + run;
    }
    __syncthreads();
  }
  const int n_items = iofs[D];
  const int lo = int((long long)blockIdx.x * n_items / gridDim.x);
  const int hi = int((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  if (lo >= hi) return;
  const int n_mine = hi - lo;
  const int n_stream = n_mine * ns;   // my slices, item after item
  const int nch = (ns + kUChunk - 1) / kUChunk;   // raw chunks per item
  const int n_chunks = n_mine * nch;

  // active expert of item it (iofs is strictly increasing)
  auto expert_of = [&](int it) {
    int l = 0, h = D - 1;
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (iofs[m] <= it) l = m; else h = m - 1;
    }
    return l;
  };
  // my item j: expert, row block, first row (sorted slot), rows, MMA N
  struct Item {
    int e, rb, pos0, ntok, nmma, n16;
  };
  auto item_slow = [&](int j) {
    Item f;
    const int it = lo + j, ai = expert_of(it), rem = it - iofs[ai];
    const int tb = rem / nrb;
    f.e = a.active[ai];
    const int n_e = a.offsets[f.e + 1] - a.offsets[f.e];
    f.rb = rem - tb * nrb;
    f.pos0 = a.offsets[f.e] + tb * kNTok;
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
  // the first kUTable items of the CTA, looked up once (in parallel) in the prologue
  int4* itab = reinterpret_cast<int4*>(smem + L.itab);
  auto item_of = [&](int j) {
    if (j >= kUTable) return item_slow(j);
    const int4 v = itab[j];
    Item f;
    f.e = v.x;
    f.rb = v.y;
    f.pos0 = v.z;
    f.ntok = v.w;
    if (MODE == kModeGateUp) {
      f.n16 = 0;
      f.nmma = (f.ntok + 15) & ~15;
    } else {
      f.n16 = (f.ntok + 7) & ~7;
      f.nmma = 2 * f.n16;
    }
    return f;
  };
  for (int j = tid; j < n_mine && j < kUTable; j += blockDim.x) {
    const Item f = item_slow(j);
    itab[j] = make_int4(f.e, f.rb, f.pos0, f.ntok);
  }

  if (tid == 0) {
    for (int i = 0; i < kURing; ++i) {
      mbar_init(&full_raw[i], 1);
      mbar_init(&empty_raw[i], kNDec);
    }
    for (int i = 0; i < kUStages; ++i) {
      mbar_init(&a_full[i], kNDec);
      mbar_init(&b_full[i], kNLoad);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < kUAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kNEpi);
    }
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == kWProducer) tmem_alloc(tslot, kUAcc * kUCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == kWProducer) {
    // ---- packed weights -> raw ring ----------------------------------------------
    if (lane == 0) {
      int issued = 0, pf_next = 0;
      const int pf_items = (kUPrefetchChunks + nch - 1) / nch;
      const uint8_t* wm = nullptr;
      int nt = 0;
      auto item_base = [&](const Item& f) {
        return a.w + (uint64_t)f.e * a.mat_bytes + (uint64_t)f.rb * kUTiles * KB * kUnitBytes;
      };
      for (int c = 0; c < n_chunks; ++c) {
        const int j = c / nch, cc = c - j * nch, s = c % kURing;
        if (c >= kURing && !uwait(&empty_raw[s], uint32_t(c / kURing - 1) & 1u, abort, a.status)) break;
        if (cc == 0) {
          const Item f = item_of(j);
          nt = min(kUTiles, a.n_tiles - f.rb * kUTiles);
          wm = item_base(f);
          // items j .. j + pf_items into L2 (each tile's units over all K are contiguous)
          for (; pf_next <= j + pf_items && pf_next < n_mine; ++pf_next) {
            const Item g = item_of(pf_next);
            const int gt = min(kUTiles, a.n_tiles - g.rb * kUTiles);
            prefetch_l2(item_base(g), uint32_t(gt) * KB * kUnitBytes);
          }
        }
        const int kb0 = cc * kUChunk * kUSliceKb, nkb = min(kUChunk * kUSliceKb, KB - kb0);
        uint8_t* dst = ring + (size_t)s * kURawBytes;
        mbar_arrive_expect_tx(&full_raw[s], uint32_t(nt * nkb) * kUnitBytes);
        for (int t = 0; t < nt; ++t)
          bulk_g2s(dst + (size_t)t * kUTileChunk, wm + ((uint64_t)t * KB + kb0) * kUnitBytes,
                   uint32_t(nkb) * kUnitBytes, &full_raw[s]);
        issued = c + 1;
      }
      if (*abort)   // copies still in flight land before the CTA's shared memory goes away
        for (int c = issued > kURing ? issued - kURing : 0; c < issued; ++c)
          mbar_wait(&full_raw[c % kURing], uint32_t(c / kURing) & 1u, a.status);
    }
  } else if (warp == kWMma) {
    // ---- tcgen05.mma issue -----------------------------------------------------------
    if (lane == 0) {
      uint64_t* last = nullptr;
      uint32_t last_par = 0;
      bool ok = true;
      for (int j = 0; j < n_mine && ok; ++j) {
        const Item f = item_of(j);
        const int ab = j % kUAcc;
        if (j >= kUAcc && !uwait(&acc_empty[ab], uint32_t(j / kUAcc - 1) & 1u, abort, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + uint32_t(ab * kUCols);
        const uint32_t idesc = umma_idesc_bf16(kURows, f.nmma);
        for (int sl = 0; sl < ns; ++sl) {
          const int p = j * ns + sl, st = p % kUStages;
          const uint32_t par = uint32_t(p / kUStages) & 1u;
          if (!uwait(&a_full[st], par, abort, a.status) || !uwait(&b_full[st], par, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nkb = min(kUSliceKb, KB - sl * kUSliceKb);
          const uint32_t as = smem_addr(abuf + (size_t)st * kUABytes);
          const uint32_t bs = smem_addr(bbuf + (size_t)st * kUBBytes);
          for (int kk = 0; kk < nkb * 2; ++kk)   // K = 16 steps: 32 bytes into the swizzle atoms
            umma_bf16(d, umma_desc_sw128(as + 32 * kk), umma_desc_sw128(bs + 32 * kk), idesc, sl > 0 || kk > 0);
          umma_commit(&op_empty[st]);
          last = &op_empty[st];
          last_par = par;
          if (sl == ns - 1) umma_commit(&acc_full[ab]);
        }
      }
      // every MMA has finished before tensor memory is freed
      if (last) mbar_wait(last, last_par, a.status);
    }
  } else if (warp < kWLoad) {
    // ---- epilogue: accumulator -> outputs --------------------------------------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // TMEM lane = weight row of the item
    for (int j = 0; j < n_mine; ++j) {
      const int ab = j % kUAcc;
      if (!uwait(&acc_full[ab], uint32_t(j / kUAcc) & 1u, abort, a.status)) break;
      tc_fence_after();
      const Item f = item_of(j);
      const uint32_t trow = tmem + uint32_t(ab * kUCols) + ((uint32_t)(quarter * 32) << 16);
      if (MODE == kModeGateUp) {
        // rows 16t .. 16t+7: gate of features 8 (rb*8 + t) + 0..7; rows +8: up.
        // h goes out as bf16 terms: hi = bf16(h), lo = bf16(h - hi)
        __nv_bfloat16* hhi = reinterpret_cast<__nv_bfloat16*>(a.out);
        __nv_bfloat16* hlo = hhi + (size_t)a.n_rows * a.out_ld;
        const int t = row >> 4, r16 = row & 15, tile = f.rb * kUTiles + t;
        const int fe = tile * 8 + (r16 & 7);
        const bool st_ok = r16 < 8 && tile < a.n_tiles;
        for (int c0 = 0; c0 < f.nmma; c0 += 8) {
          uint32_t v[8];
          tmem_ld8(trow + c0, v);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float gv = __uint_as_float(v[jj]);
            const float uv = __shfl_down_sync(0xFFFFFFFFu, gv, 8);
            if (st_ok && c0 + jj < f.ntok) {
              const float h = silu_f(gv) * uv;
              const __nv_bfloat16 hb = __float2bfloat16_rn(h);
              const size_t o = (size_t)(f.pos0 + c0 + jj) * a.out_ld + fe;
              hhi[o] = hb;
              hlo[o] = __float2bfloat16_rn(h - __bfloat162float(hb));
            }
          }
        }
      } else {
        const int r = f.rb * kURows + row;   // output feature
        const bool st_ok = r < a.n_tiles * kTileRows;
        for (int c0 = 0; c0 < f.n16; c0 += 8) {
          uint32_t vh[8], vl[8];
          tmem_ld8(trow + c0, vh);
          tmem_ld8(trow + f.n16 + c0, vl);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (st_ok && c0 + jj < f.ntok)
              a.out[(size_t)(f.pos0 + c0 + jj) * a.out_ld + r] = __uint_as_float(vh[jj]) + __uint_as_float(vl[jj]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  } else if (warp < kWDec) {
    // ---- activation rows -> operand stage (cp.async) --------------------------------
    // Thread lt copies 16-byte column c = lt % 8 of rows lt / 8 + 16 m. Gate/up:
    // the rows are tokens (x rows gathered through perm). Down: the rows are
    // sorted slots, hi terms to B rows r and lo terms to B rows n16 + r.
    const int lt = tid - kWLoad * 32, c = lt & 7, rr = lt >> 3;
    constexpr int kRows = MODE == kModeGateUp ? kUCols / 16 : kUCols / 32;   // rows per thread
    const __nv_bfloat16* src0 = static_cast<const __nv_bfloat16*>(a.act_raw);
    const __nv_bfloat16* src1 = static_cast<const __nv_bfloat16*>(a.act_raw2);
    int b_row[kRows], nb_row[kRows];   // source rows of this item and of the next one
    int pend = 0;                       // first slice not yet announced
    Item f{};
    // rows of item j (requested one item ahead, so the loads are in flight meanwhile)
    auto rows_of = [&](int j, int (&rows)[kRows]) {
      const Item h = item_of(j);
#pragma unroll
      for (int m = 0; m < kRows; ++m) {
        const int r = rr + 16 * m;
        rows[m] = r < h.ntok ? (MODE == kModeGateUp ? a.perm[h.pos0 + r] / a.k : h.pos0 + r) : 0;
      }
    };
    if (n_mine > 0) rows_of(0, nb_row);
    for (int p = 0; p < n_stream; ++p) {
      const int j = p / ns, sl = p - j * ns, st = p % kUStages;
      if (p >= kUStages && !uwait(&op_empty[st], uint32_t(p / kUStages - 1) & 1u, abort, a.status)) break;
      if (sl == 0) {
        f = item_of(j);
#pragma unroll
        for (int m = 0; m < kRows; ++m) b_row[m] = nb_row[m];
        if (j + 1 < n_mine) rows_of(j + 1, nb_row);
      }
      const int kb0 = sl * kUSliceKb, nc = min(kUSliceKb, KB - kb0) * (kMxBlock / 8);
      uint8_t* bb = bbuf + (size_t)st * kUBBytes;
      const int nrow = MODE == kModeGateUp ? f.nmma : f.n16;
      if (c < nc) {
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
          const int r = rr + 16 * m;
          if (r < nrow) {
            const bool valid = r < f.ntok;
            const size_t o = (size_t)b_row[m] * K + kb0 * kMxBlock + c * 8;
            cp_async16(bb + sw128_off(r, c * 8), src0 + o, valid);
            if (MODE == kModeDown) cp_async16(bb + sw128_off(f.n16 + r, c * 8), src1 + o, valid);
          }
        }
      }
      cp_async_commit();
      // announce slice p - kULag once its copies (not the later ones) have landed
      if (p - pend >= kULag) {
        cp_async_wait<kULag>();
        fence_async_smem();   // generic-proxy writes -> visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_full[pend % kUStages]);
        ++pend;
      }
    }
    cp_async_wait<0>();   // nothing lands after the CTA's shared memory goes away
    if (!*abort) {
      fence_async_smem();
      __syncwarp();
      for (; pend < n_stream; ++pend)
        if (lane == 0) mbar_arrive(&b_full[pend % kUStages]);
    }
  } else {
    // ---- raw ring -> bf16 weights (decode warp dw: tile dw % 8 of the item, the
    // slice's 32-wide K-blocks u = dw / 8, dw / 8 + 2, ...) ----------------------------
    const int dw = warp - kWDec, t = dw % kUTiles;
    const int g = lane >> 2, q = lane & 3;
    int tile = 0;
    for (int p = 0; p < n_stream; ++p) {
      const int j = p / ns, sl = p - j * ns, st = p % kUStages;
      const int cc = sl / kUChunk, sub = sl - cc * kUChunk, c = j * nch + cc, s = c % kURing;
      if (sub == 0 && !uwait(&full_raw[s], uint32_t(c / kURing) & 1u, abort, a.status)) break;
      if (p >= kUStages && !uwait(&op_empty[st], uint32_t(p / kUStages - 1) & 1u, abort, a.status)) break;
      if (sl == 0) {
        tile = item_of(j).rb * kUTiles + t;
      }
      const int nkb = min(kUSliceKb, KB - sl * kUSliceKb);
      const uint8_t* raw = ring + (size_t)s * kURawBytes + (size_t)t * kUTileChunk + (size_t)sub * kUSliceKb * kUnitBytes;
      uint8_t* ab = abuf + (size_t)st * kUABytes;
#pragma unroll
      for (int u = dw / kUTiles; u < kUSliceKb; u += kDecPerTile) {
        const int r0 = t * kTileRows + g, r1 = r0 + 8;
        uint2 c0 = make_uint2(0u, 0u), c1 = c0, c2 = c0, c3 = c0;
        if (u < nkb && tile < a.n_tiles) {
          const uint8_t* unit = raw + (size_t)u * kUnitBytes;
          const uint2 wv = *reinterpret_cast<const uint2*>(unit + lane * 8);
          const uint32_t sc16 = *reinterpret_cast<const uint16_t*>(unit + kUnitCodeBytes + 2 * g);
          const uint32_t slo = sc16 & 0xFFu, shi = sc16 >> 8;   // block scales of rows g and g+8
          const bool big = __any_sync(0xFFFFFFFFu, (slo | shi) > 128u);
          const uint32_t f1lo = scale_f1(slo), f2lo = scale_f2(slo), f1hi = scale_f1(shi), f2hi = scale_f2(shi);
          c0 = e2m1x4_to_bf16x4(decode_rowlo(wv.x), f1lo, f2lo, big);   // row g,   k 4q .. 4q+3
          c1 = e2m1x4_to_bf16x4(decode_rowhi(wv.x), f1hi, f2hi, big);   // row g+8
          c2 = e2m1x4_to_bf16x4(decode_rowlo(wv.y), f1lo, f2lo, big);   // row g,   k 16+4q ..
          c3 = e2m1x4_to_bf16x4(decode_rowhi(wv.y), f1hi, f2hi, big);   // row g+8
        }
        const int k0 = u * kMxBlock + 4 * q;
        *reinterpret_cast<uint2*>(ab + sw128_off(r0, k0)) = c0;
        *reinterpret_cast<uint2*>(ab + sw128_off(r1, k0)) = c1;
        *reinterpret_cast<uint2*>(ab + sw128_off(r0, k0 + 16)) = c2;
        *reinterpret_cast<uint2*>(ab + sw128_off(r1, k0 + 16)) = c3;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[st]);
        if (sub == kUChunk - 1 || sl == ns - 1) mbar_arrive(&empty_raw[s]);   // chunk consumed
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWProducer) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUAcc * kUCols);
  }
}

}  // namespace

int launch_umma_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s) {
  const UmmaSmem L = umma_smem();
  if (L.total > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int grid = di.sm_count;
  if (mode == kModeGateUp) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(L.total)));
    umma_routed_kernel<kModeGateUp><<<grid, kUBlock, L.total, s>>>(a, L);
  } else {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(L.total)));
    umma_routed_kernel<kModeDown><<<grid, kUBlock, L.total, s>>>(a, L);
  }
  return launch_status();
}

}  // namespace moe
