// Routed-expert GEMMs on the 5th-generation tensor cores (tcgen05) with
// block-scaled MMAs, from 5 tokens up to prefill: gate/up with SwiGLU, and
// down. The experts are the MXFP4 (W4) experts of page "3 ways to speed up
// MoE inference on NVIDIA DGX Spark", §2-§3, run with bf16 activations or, in
// the W4A8 configuration of §2, 8-bit ones; each expert runs once over the
// tokens that chose it, after they are sorted by expert (page "MoE-SpeQ ...",
// §4.2).
//
// Every MMA is tcgen05.mma.kind::mxf8f6f4.block_scale: A = 128 weight rows x
// K 32 as E2M1 codes, B = activation rows x K 32 as E4M3 codes, each with one
// E8M0 scale per row and 32-wide K-block, read by the tensor core from tensor
// memory; fp32 accumulation in tensor memory. The MXFP4 weights enter as they
// are stored: the tensor cores read E2M1 from 16-byte chunks whose low 8 bytes
// hold 16 codes (the packed layout's half-rows), and the A scale bytes are the
// packed E8M0 bytes. The activations arrive pre-quantised (quant.cu): MXFP8
// for the 8-bit-activation call, or two E4M3 terms sharing one E8M0 scale
// (bf16 precision), which the MMA reads as separate B rows and the epilogue
// adds.
//
// Work items are (active expert, block of 128 weight rows = 8 packed 16-row
// tiles, block of up to 128 B rows of that expert's tokens / slots), ordered
// by row block then token block, split into contiguous ranges per CTA (one
// CTA per SM, persistent). Along K an
// item goes in slices of four 32-wide K-blocks (one 128-byte swizzle row).
// The CTA is a pipeline of warp roles that meet only at mbarriers:
//   * producer (one thread): 1-D bulk copies of the packed MXFP4 bytes of a
//     chunk of 2 slices (one copy per tile) into a ring of raw slots; whole
//     items are also prefetched into L2 about 8 chunks ahead;
//   * 16 placement warps (two per tile): raw slot -> the half-rows of codes
//     in the K-major 128-byte-swizzled layout the MMA reads (one 8-byte load
//     and store per lane and unit, no arithmetic), and the A scale bytes in
//     the layout tcgen05.cp copies;
//   * 4 loader warps: the slice of the activation rows (x gathered by token,
//     or h by slot; each term a block of B rows) copied with cp.async, and
//     their B scale bytes; every loader thread's copies arrive on the stage
//     barrier by themselves when they land (cp.async.mbarrier.arrive.noinc),
//     so a loader never waits for its own copies;
//   * MMA (one thread): after the stage's barriers, a proxy fence (the
//     loaders' copies and scale bytes are generic-proxy writes), tcgen05.cp of
//     the slice's A and B scales into tensor memory, then one MMA per K-block (M = 128, N = the item's B rows) into
//     one of two accumulators; each slice's work is committed to the barrier
//     that frees its stage, the item's last slice also to the accumulator's;
//   * 4 epilogue warps (one per 32-lane quarter of tensor memory): tcgen05.ld,
//     the terms of a row added, then SwiGLU of the gate and up rows of a tile
//     (8 lanes apart) to fp32 h, or for the down pass the fp32 outputs per slot.
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
constexpr int kUTiles = kURows / kTileRows;  // packed tiles per item (one per placement warp pair)
constexpr int kUSliceKb = 4;                 // 32-wide K-blocks per slice: one 128-byte swizzle row
constexpr int kUSliceK = kUSliceKb * kMxBlock;
constexpr int kUStages = 4;                  // operand stages (weights + activations + scales)
constexpr int kUChunk = 2;                   // slices per raw weight copy
constexpr int kUPrefetchChunks = 8;          // weights prefetched into L2 about this many chunks ahead
constexpr int kUAcc = 2;                     // accumulators in tensor memory
constexpr int kUSfCols = 8;                  // tensor-memory columns of one stage's scales (A: 4, B: 4)
constexpr uint32_t kUTmemCols = 512;         // 2 x 128 accumulator + 4 x 8 scale columns, as a power of two
constexpr int kUMaxActive = 1024;
constexpr int kUTable = 256;                 // items per CTA with a precomputed table entry
constexpr uint32_t kUTileChunk = kUChunk * kUSliceKb * kUnitBytes;   // one tile's part of a chunk
constexpr uint32_t kURawBytes = kUTiles * kUTileChunk;                  // one chunk of packed weights
constexpr uint32_t kUABytes = kURows * kUSliceK;                     // one slice of weights (E2M1 chunks)
constexpr uint32_t kUSfBytes = 512;                                  // scales of 128 rows x 4 K-blocks

// warp roles
constexpr int kWProducer = 0, kWMma = 1, kWEpi = 2, kNEpi = 4, kWLoad = kWEpi + kNEpi, kNLoad = 4,
              kWDec = kWLoad + kNLoad, kDecPerTile = 2, kNDec = kUTiles * kDecPerTile;
constexpr int kUBlock = (kWDec + kNDec) * 32;
constexpr int kScanThreads = 256;

struct UmmaSmem {
  uint32_t ring, a, b, sfa, sfb, iofs, itab, bars, misc, total;
};
// Two configurations (template arguments COLS, RING of the kernel and of its
// shared-memory plan): wide items of up to 128 B rows with a 3-chunk raw
// ring, for many tokens per expert; narrow items of up to 64 B rows, whose
// smaller activation stages leave room for a 5-chunk raw ring (more weight
// bytes in flight), for few tokens per expert.
constexpr int kUColsWide = 128, kURingWide = 3, kUColsNarrow = 64, kURingNarrow = 5;
template <int COLS, int RING>
__host__ __device__ inline UmmaSmem umma_smem() {
  UmmaSmem m{};
  uint32_t at = 0;
  auto take = [&](uint32_t bytes, uint32_t align) {
    at = (at + align - 1) / align * align;
    const uint32_t here = at;
    at += bytes;
    return here;
  };
  m.ring = take(RING * kURawBytes, 128);
  m.a = take(kUStages * kUABytes, 1024);
  m.b = take(kUStages * uint32_t(COLS) * kUSliceK, 1024);
  m.sfa = take(kUStages * kUSfBytes, 128);
  m.sfb = take(kUStages * kUSfBytes, 128);
  m.iofs = take((kUMaxActive + 1) * 4, 16);
  m.itab = take(kUTable * 16, 16);
  m.bars = take((2 * RING + 3 * kUStages + 2 * kUAcc) * 8, 8);
  m.misc = take(16, 16);   // tensor-memory address, abort flag
  m.total = at + 1024;     // slack: the swizzled buffers are aligned to 1024 in the shared window
  return m;
}

// byte offset of the byte element (row r, k < 128) in a K-major operand with
// 128-byte swizzle: row r in atom r / 8 (1024 bytes each), line r % 8 (128
// bytes), its 16-byte chunk k / 16 stored at chunk (k / 16) ^ (r % 8)
__device__ __forceinline__ uint32_t sw128_off8(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 4) ^ (r & 7)) << 4) + (k & 15));
}
// byte offset of the scale of row r (< 128) and K-block kb (< 4) of a slice in
// the 512-byte block that tcgen05.cp .32x128b.warpx4 copies: 32 lines of 16
// bytes, line r % 32 holding rows r % 32 + 32 j (j = 0..3) at bytes 4 j + kb.
// The tensor core reads the scale of row r from column r / 32, byte kb.
__device__ __forceinline__ uint32_t sf_off(int r, int kb) { return (uint32_t)((r & 31) * 16 + (r >> 5) * 4 + kb); }

// 16-byte asynchronous global -> shared copy; zero-filled when !valid
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int MODE, int COLS, int RING>
__global__ void __launch_bounds__(kUBlock, 1) umma_routed_kernel(RoutedArgs a, UmmaSmem L) {
  constexpr int kUCols = COLS;                                    // B rows per item = largest MMA N
  constexpr int kURing = RING;                                    // raw weight chunks in flight
  constexpr uint32_t kUBBytes = uint32_t(kUCols) * kUSliceK;      // one slice of E4M3 activations
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle is a function of the shared address: align the plan's base to 1024
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem + L.ring;
  uint8_t* abuf = smem + L.a;
  uint8_t* bbuf = smem + L.b;
  uint8_t* sfabuf = smem + L.sfa;
  uint8_t* sfbbuf = smem + L.sfb;
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
  // B rows per item: every term of a token (gate/up) or slot (down) is a B row
  const int nterms = a.act_terms;
  const int kNTok = kUCols / nterms;
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
  // my item j: expert, row block, first row (sorted slot), rows, MMA N, and
  // the B rows of one term (term t occupies B rows [t n16, t n16 + ntok))
  struct Item {
    int e, rb, pos0, ntok, nmma, n16;
  };
  auto geometry = [&](Item& f) {
    f.n16 = nterms == 2 ? (f.ntok + 7) & ~7 : (f.ntok + 15) & ~15;
    f.nmma = nterms * f.n16;
  };
  auto item_slow = [&](int j) {
    Item f;
    const int it = lo + j, ai = expert_of(it), rem = it - iofs[ai];
    f.e = a.active[ai];
    const int n_e = a.offsets[f.e + 1] - a.offsets[f.e];
    // row block major, token block minor: the token blocks of one row block
    // follow each other, so the second one reads the weights from L2
    const int ntb = (n_e + kNTok - 1) / kNTok;
    f.rb = rem / ntb;
    const int tb = rem - f.rb * ntb;
    f.pos0 = a.offsets[f.e] + tb * kNTok;
    f.ntok = min(kNTok, n_e - tb * kNTok);
    geometry(f);
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
    geometry(f);
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
      mbar_init(&b_full[i], kNLoad * 32);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < kUAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kNEpi);
    }
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == kWProducer) tmem_alloc(tslot, kUTmemCols);
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
      // One thread issues every tensor-core operation of the CTA, so its own
      // instruction stream sets the pace: descriptors of stage st are the
      // stage-0 ones plus a constant (the 14-bit address field is the byte
      // address / 16 and never carries), the instruction descriptors are
      // built once per item, and the K-blocks of a slice are unrolled.
      const uint64_t a_desc0 = umma_desc_sw128(smem_addr(abuf)), b_desc0 = umma_desc_sw128(smem_addr(bbuf));
      const uint64_t sfa_desc0 = umma_desc_sf(smem_addr(sfabuf)), sfb_desc0 = umma_desc_sf(smem_addr(sfbbuf));
      const uint32_t sf_tmem0 = tmem + uint32_t(kUAcc * kUCols);
      int st = 0;
      uint32_t par = 0;
      for (int j = 0; j < n_mine && ok; ++j) {
        const Item f = item_of(j);
        const int ab = j % kUAcc;
        if (j >= kUAcc && !uwait(&acc_empty[ab], uint32_t(j / kUAcc - 1) & 1u, abort, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + uint32_t(ab * kUCols);
        uint32_t idesc[kUSliceKb];
#pragma unroll
        for (int kb = 0; kb < kUSliceKb; ++kb) idesc[kb] = umma_idesc_mx(kURows, f.nmma, kFmtE2M1, kb, kb);
        for (int sl = 0; sl < ns; ++sl) {
          if (!uwait(&a_full[st], par, abort, a.status) || !uwait(&b_full[st], par, abort, a.status)) {
            ok = false;
            break;
          }
          fence_async_smem();
          tc_fence_after();
          const int nkb = min(kUSliceKb, KB - sl * kUSliceKb);
          const uint64_t ad = a_desc0 + uint64_t(st * (kUABytes >> 4)), bd = b_desc0 + uint64_t(st * (kUBBytes >> 4));
          // this slice's scales into tensor memory (in issue order before its MMAs)
          const uint32_t sfa = sf_tmem0 + uint32_t(st * kUSfCols), sfb = sfa + 4;
          tmem_cp_sf(sfa, sfa_desc0 + uint64_t(st * (kUSfBytes >> 4)));
          tmem_cp_sf(sfb, sfb_desc0 + uint64_t(st * (kUSfBytes >> 4)));
#pragma unroll
          for (int kb = 0; kb < kUSliceKb; ++kb)   // K = 32 steps: 32 bytes into the swizzle rows
            if (kb < nkb) umma_mx(d, ad + uint64_t(2 * kb), bd + uint64_t(2 * kb), idesc[kb], sfa, sfb, sl > 0 || kb > 0);
          umma_commit(&op_empty[st]);
          last = &op_empty[st];
          last_par = par;
          if (sl == ns - 1) umma_commit(&acc_full[ab]);
          if (++st == kUStages) {
            st = 0;
            par ^= 1u;
          }
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
        // h goes out as fp32 [slot][I] (row = sorted slot)
        const int t = row >> 4, r16 = row & 15, tile = f.rb * kUTiles + t;
        const int fe = tile * 8 + (r16 & 7);
        const bool st_ok = r16 < 8 && tile < a.n_tiles;
        for (int c0 = 0; c0 < f.n16; c0 += 8) {
          uint32_t v[8], v2[8];
          tmem_ld8(trow + c0, v);
          if (nterms == 2) tmem_ld8(trow + f.n16 + c0, v2);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float gv = __uint_as_float(v[jj]) + (nterms == 2 ? __uint_as_float(v2[jj]) : 0.0f);
            const float uv = __shfl_down_sync(0xFFFFFFFFu, gv, 8);
            if (st_ok && c0 + jj < f.ntok) a.out[(size_t)(f.pos0 + c0 + jj) * a.out_ld + fe] = silu_f(gv) * uv;
          }
        }
      } else {
        const int r = f.rb * kURows + row;   // output feature
        const bool st_ok = r < a.n_tiles * kTileRows;
        for (int c0 = 0; c0 < f.n16; c0 += 8) {
          // output row of column c0 + l at lane l < 8: the sorted slot, or its
          // (token, choice) pair t k + j
          int orow = f.pos0 + c0 + (lane & 7);
          if (a.out_by_pair && lane < 8 && c0 + lane < f.ntok) orow = __ldg(a.perm + orow);
          uint32_t vh[8], vl[8];
          tmem_ld8(trow + c0, vh);
          if (nterms == 2) tmem_ld8(trow + f.n16 + c0, vl);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int o = __shfl_sync(0xFFFFFFFFu, orow, jj);
            if (st_ok && c0 + jj < f.ntok)
              a.out[(size_t)o * a.out_ld + r] =
                  __uint_as_float(vh[jj]) + (nterms == 2 ? __uint_as_float(vl[jj]) : 0.0f);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  } else if (warp < kWDec) {
    // ---- activation rows -> operand stage (cp.async), and their scales -------------
    // B row r of an item is term r / n16 of its activation row r % n16 (gate/up:
    // the token of sorted slot pos0 + r % n16; down: the slot itself). Thread lt
    // copies 16-byte chunk c = lt % 8 of B rows lt / 8 + 16 m, and writes the
    // scale bytes of B row lt.
    const int lt = tid - kWLoad * 32, c = lt & 7, rr = lt >> 3;
    constexpr int kRows = kUCols / 16;   // B rows per thread
    int b_src[kRows], nb_src[kRows];     // (activation row * nterms + term), or -1 for padding
    int s_src = -1, ns_src = -1;         // activation row of B row lt, or -1
    Item f{};
    // rows of item j (requested one item ahead, so the loads are in flight meanwhile)
    auto rows_of = [&](int j, int (&src)[kRows], int& ssrc) {
      const Item h = item_of(j);
      auto act_row = [&](int r) -> int {
        if (r >= h.nmma) return -1;
        const int tt = r / h.n16, jj = r - tt * h.n16;
        if (jj >= h.ntok) return -1;
        const int ar = MODE == kModeGateUp ? a.perm[h.pos0 + jj] / a.k : h.pos0 + jj;
        return ar * nterms + tt;
      };
#pragma unroll
      for (int m = 0; m < kRows; ++m) src[m] = act_row(rr + 16 * m);
      const int v = act_row(lt);
      ssrc = v < 0 ? -1 : v / nterms;
    };
    if (n_mine > 0) rows_of(0, nb_src, ns_src);
    for (int p = 0; p < n_stream; ++p) {
      const int j = p / ns, sl = p - j * ns, st = p % kUStages;
      if (p >= kUStages && !uwait(&op_empty[st], uint32_t(p / kUStages - 1) & 1u, abort, a.status)) break;
      if (sl == 0) {
        f = item_of(j);
#pragma unroll
        for (int m = 0; m < kRows; ++m) b_src[m] = nb_src[m];
        s_src = ns_src;
        if (j + 1 < n_mine) rows_of(j + 1, nb_src, ns_src);
      }
      const int kb0 = sl * kUSliceKb, nkb = min(kUSliceKb, KB - kb0), nc = nkb * (kMxBlock / 16);
      uint8_t* bb = bbuf + (size_t)st * kUBBytes;
      if (c < nc) {
#pragma unroll
        for (int m = 0; m < kRows; ++m) {
          const int r = rr + 16 * m;
          if (r < f.nmma) {
            const bool valid = b_src[m] >= 0;
            const size_t o = (size_t)(valid ? b_src[m] : 0) * K + kb0 * kMxBlock + c * 16;
            cp_async16(bb + sw128_off8(r, c * 16), a.act_q + o, valid);
          }
        }
      }
      uint8_t* sb = sfbbuf + (size_t)st * kUSfBytes;
#pragma unroll
      for (int i = 0; i < kUSliceKb; ++i)
        sb[sf_off(lt, i)] = (s_src >= 0 && i < nkb) ? a.act_s[(size_t)s_src * KB + kb0 + i] : uint8_t(127);
      // this thread's arrival on the stage barrier, made when its copies land
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&b_full[st])) : "memory");
    }
    cp_async_wait<0>();   // nothing lands after the CTA's shared memory goes away
  } else {
    // ---- raw ring -> the tensor cores' E2M1 operand form and A scales
    // (placement warp dw: tile dw % 8 of the item, the slice's 32-wide
    // K-blocks u = dw / 8, dw / 8 + 2). Lane l moves half-row l % 2 of row
    // l / 2 of a unit (16 codes, 8 bytes) into the low half of its 16-byte
    // chunk of the swizzled A slice; the high half is never read.
    const int dw = warp - kWDec, t = dw % kUTiles;
    const int rr = lane >> 1, hh = lane & 1;
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
      uint8_t* sa = sfabuf + (size_t)st * kUSfBytes;
#pragma unroll
      for (int u = dw / kUTiles; u < kUSliceKb; u += kDecPerTile) {
        const bool ok = u < nkb && tile < a.n_tiles;
        const uint8_t* unit = raw + (size_t)u * kUnitBytes;
        const uint2 v = ok ? *reinterpret_cast<const uint2*>(unit + rr * 16 + hh * 8) : make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(ab + sw128_off8(t * kTileRows + rr, u * kMxBlock + hh * 16)) = v;
        if (lane < 16) {   // scale byte 2g + h is row g + 8h
          const uint8_t sc = ok ? unit[kUnitCodeBytes + lane] : uint8_t(0);
          sa[sf_off(t * kTileRows + (lane >> 1) + 8 * (lane & 1), u)] = sc;
        }
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
    tmem_dealloc(tmem, kUTmemCols);
  }
}

template <int COLS, int RING>
int launch_umma_cfg(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s) {
  const UmmaSmem L = umma_smem<COLS, RING>();
  if (L.total > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int grid = di.sm_count;
  if (mode == kModeGateUp) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeGateUp, COLS, RING>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)));
    umma_routed_kernel<kModeGateUp, COLS, RING><<<grid, kUBlock, L.total, s>>>(a, L);
  } else {
    MOE_CUDA_TRY(cudaFuncSetAttribute(umma_routed_kernel<kModeDown, COLS, RING>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total)));
    umma_routed_kernel<kModeDown, COLS, RING><<<grid, kUBlock, L.total, s>>>(a, L);
  }
  return launch_status();
}

}  // namespace

int launch_umma_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s) {
  return a.narrow ? launch_umma_cfg<kUColsNarrow, kURingNarrow>(mode, a, di, s)
                  : launch_umma_cfg<kUColsWide, kURingWide>(mode, a, di, s);
}

}  // namespace moe
