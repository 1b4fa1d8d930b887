// Dense bf16 GEMMs of the per-stage path on the 5th-generation tensor cores,
// for many tokens. The router and the shared expert stay in bf16 (page
// "MoE-SpeQ ...", §2.1-§2.2: routing is sensitive to quantisation, and the
// shared expert acts on every token):
//   * front: the router logits and the shared expert's gate/up projections
//     with SwiGLU, h_sh going out as two bf16 terms (hi = bf16(h), lo =
//     bf16(h - hi));
//   * combine: the shared expert's down projection of h_sh (both terms into
//     one accumulator, so h keeps about 16 significant bits) plus the
//     routing-weighted sum of the routed experts' outputs, rounded to bf16.
//
// Every MMA is tcgen05.mma.kind::f16: A = 128 weight rows x K 16, B = 128
// tokens x K 16, both bf16 and K-major in shared memory with the 128-byte
// swizzle, fp32 accumulator in tensor memory (lane = weight row, column =
// token). The operand tiles are 128-row x 64-column boxes brought in by the
// tensor memory accelerator (cp.async.bulk.tensor with 2-D tensor maps); the
// rows and columns of a box past the end of a matrix read as zero, which is
// how ragged T, E, I, d and K are handled.
//
// Items are (block of 128 weight rows, block of 128 tokens). A router or
// combine item has one accumulator; a shared gate/up item has two, the gate
// rows and the up rows of the same 128 features, so the epilogue thread of
// feature f holds both; it costs twice as much. One CTA per SM, persistent;
// the two-cost items are dealt longest first (the costly ones round-robin,
// then the cheap ones to the CTAs with less work first), so no CTA holds
// much more than the mean.
//
// Warp roles, meeting only at mbarriers:
//   * producer (one thread): per 64-wide K step, the step's boxes into one of
//     the operand stages (48 KB: up to three boxes), completion in bytes;
//   * MMA (one thread): 4 MMAs per box pair and K step into one of two
//     accumulators (256 columns each), each step committed to the barrier
//     that frees its stage, an item's last also to the accumulator's;
//   * combine only, part producer (one thread): the routed outputs of the
//     item's tokens, rows t k + j of part (one token's k rows are adjacent),
//     columns = the item's 128 output features, as 2-D boxes of kpt tokens
//     (512-byte row pieces) into a ring of four 32 KB slots;
//   * 8 epilogue warps (two per 32-lane quarter of tensor memory): tcgen05.ld,
//     then the outputs. In the combine the two warps of a quarter take the
//     two halves of each part box's tokens and read the part values from
//     shared memory (lane = feature: conflict-free).
// Every wait is bounded; a timeout sets MOE_DEV_TIMEOUT and an abort flag
// that ends the other roles' waits, and the CTA drains its own copies and
// MMAs before it frees tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"
#include "tma.cuh"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int kTM = 128;                   // weight rows per item (MMA M)
constexpr int kTN = 128;                   // tokens per item (MMA N)
constexpr int kTK = 64;                    // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kTBox = kTM * kTK * 2;  // one operand box, 16 KB
constexpr uint32_t kTStageBytes = 3 * kTBox;
constexpr int kTAcc = 2;
constexpr uint32_t kTAccCols = 2 * kTN;    // two accumulators per item
constexpr uint32_t kTTmemCols = kTAcc * kTAccCols;
constexpr int kTWProd = 0, kTWMma = 1, kTWPart = 2, kTWEpi = 4, kTNEpi = 8;
constexpr int kTBlock = (kTWEpi + kTNEpi) * 32;
constexpr int kPartRing = 4;                    // combine: part box slots
constexpr int kPartRows = 64;                   // rows (token, choice pairs) per part box, at most
constexpr uint32_t kPartBox = kPartRows * kTM * 4;   // 32 KB

static_assert(kTM == 128 && kTN % 16 == 0 && kTN <= 256, "MMA shape");
static_assert(kTTmemCols <= 512, "tensor memory");

// Shared-memory plan of the front (MODE 0: 4 operand stages) and of the
// combine (MODE 1: 2 operand stages + the part ring).
template <int MODE>
struct TcdPlan {
  static constexpr int kStages = MODE == 0 ? 4 : 2;
  static constexpr uint32_t kPart = kStages * kTStageBytes;                       // part ring (MODE 1)
  static constexpr uint32_t kBars = kPart + (MODE == 1 ? kPartRing * kPartBox : 0);
  static constexpr int kNBars = 2 * kStages + 2 * kTAcc + (MODE == 1 ? 2 * kPartRing : 0);
  static constexpr uint32_t kTotal = kBars + kNBars * 8 + 16 + 1024;   // + slack for the 1024 alignment
};

// Operands of one kernel. Front: map 0 = x [T][d], 1 = router [E][d], 2 =
// shared gate [I][d], 3 = shared up [I][d] (bf16, 128 x 64 boxes, 128-byte
// swizzle). Combine: map 0 = h_sh hi [T][I], 1 = shared down [d][I], 2 =
// h_sh lo [T][I] (the same), 3 = part [T k][d] (fp32, kpt k x 128 boxes, no
// swizzle).
struct TcdParams {
  CUtensorMap map[4];
  int T, K, E, I, d, k;
  int kpt;              // combine: tokens per part box (kpt k <= 64, kpt a power of two >= 8)
  int n_big, n_small;   // items of cost 2 (gate/up) and of cost 1 (router, combine)
  int n_fb, n_mb;       // row blocks of the big and of the small items
  float* logits;        // [T][E]
  __nv_bfloat16* hh;    // [T][I]
  __nv_bfloat16* hl;    // [T][I]
  const float* w;       // [T][k]
  __nv_bfloat16* y;     // [T][d]
  int* status;
};

// Dealing of n_big items of cost 2 and n_small of cost 1 to G CTAs: the big
// ones round-robin (CTA b gets b, b + G, ...), so CTAs [r, G) hold one fewer
// (r = n_big % G); the first small ones go to those CTAs, up to two each
// (which evens them out), the rest round-robin over all CTAs. Item ids: big
// items [0, n_big), small ones n_big + s.
struct TcdSched {
  int G, n_big, n_small, q, r, nL, n1;
};
__host__ __device__ inline TcdSched tcd_sched(int G, int n_big, int n_small) {
  TcdSched s;
  s.G = G;
  s.n_big = n_big;
  s.n_small = n_small;
  s.q = n_big / G;
  s.r = n_big % G;
  s.nL = G - s.r;
  s.n1 = n_small < 2 * s.nL ? n_small : 2 * s.nL;
  return s;
}
__host__ __device__ inline int tcd_first_small(const TcdSched& s, int b) {
  if (b < s.r) return 0;
  const int i0 = b - s.r;
  return (i0 < s.n1 ? 1 : 0) + (i0 + s.nL < s.n1 ? 1 : 0);
}
__host__ __device__ inline int tcd_count(const TcdSched& s, int b) {
  const int rest = s.n_small - s.n1 - b;
  return s.q + (b < s.r ? 1 : 0) + tcd_first_small(s, b) + (rest > 0 ? (rest + s.G - 1) / s.G : 0);
}
__host__ __device__ inline int tcd_item(const TcdSched& s, int b, int j) {
  const int nb = s.q + (b < s.r ? 1 : 0);
  if (j < nb) return b + j * s.G;
  j -= nb;
  const int n1 = tcd_first_small(s, b);
  if (j < n1) return s.n_big + (b - s.r) + j * s.nL;
  j -= n1;
  return s.n_big + s.n1 + b + j * s.G;
}

// MODE 0: front; MODE 1: combine.
template <int MODE>
__global__ void __launch_bounds__(kTBlock, 1) tc_dense_kernel(const __grid_constant__ TcdParams P) {
  using Plan = TcdPlan<MODE>;
  constexpr int kStages = Plan::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle is a function of the shared address: align the stages to 1024
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Plan::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + kTAcc;
  uint64_t* part_full = acc_empty + kTAcc;            // MODE 1
  uint64_t* part_empty = part_full + kPartRing;       // MODE 1
  uint32_t* tslot = reinterpret_cast<uint32_t*>(full + Plan::kNBars);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  const float* part_smem = reinterpret_cast<const float*>(smem + Plan::kPart);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const TcdSched S = tcd_sched(int(gridDim.x), P.n_big, P.n_small);
  const int n_mine = tcd_count(S, int(blockIdx.x));
  if (n_mine == 0) return;
  const int nk = (P.K + kTK - 1) / kTK;

  struct Item {
    int big, m0, t0;   // two accumulators?, first weight row, first token
  };
  auto item = [&](int j) {
    const int id = tcd_item(S, int(blockIdx.x), j);
    Item f;
    if (id < P.n_big) {
      f.big = 1;
      f.m0 = (id % P.n_fb) * kTM;
      f.t0 = (id / P.n_fb) * kTN;
    } else {
      const int s = id - P.n_big;
      f.big = 0;
      f.m0 = (s % P.n_mb) * kTM;
      f.t0 = (s / P.n_mb) * kTN;
    }
    return f;
  };
  // combine: part boxes of an item (those with at least one token < T)
  auto n_boxes = [&](const Item& f) {
    const int nt = min(kTN, P.T - f.t0);
    return (nt + P.kpt - 1) / P.kpt;
  };

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kTAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kTNEpi);
    }
    if (MODE == 1)
      for (int i = 0; i < kPartRing; ++i) {
        mbar_init(&part_full[i], 1);
        mbar_init(&part_empty[i], kTNEpi);
      }
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == kTWMma) tmem_alloc(tslot, kTTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t stage0 = smem_addr(smem);

  if (warp == kTWProd) {
    // ---- operand boxes -> stages ----------------------------------------------------
    if (lane == 0) {
      for (int i = 0; i < (MODE == 0 ? 4 : 3); ++i) tma_prefetch_map(&P.map[i]);
      int p = 0, issued = 0;
      bool ok = true;
      for (int j = 0; j < n_mine && ok; ++j) {
        const Item f = item(j);
        for (int ks = 0; ks < nk; ++ks, ++p) {
          const int s = p % kStages;
          if (p >= kStages && !uwait(&empty[s], uint32_t(p / kStages - 1) & 1u, abort, P.status)) {
            ok = false;
            break;
          }
          const uint32_t st = stage0 + uint32_t(s) * kTStageBytes;
          const int kx = ks * kTK;
          if (MODE == 0) {
            // box 0: router or gate rows, box 1: up rows, box 2: x
            mbar_arrive_expect_tx(&full[s], (f.big ? 3u : 2u) * kTBox);
            if (f.big) {
              tma_load_2d(st, &P.map[2], kx, f.m0, &full[s]);
              tma_load_2d(st + kTBox, &P.map[3], kx, f.m0, &full[s]);
            } else {
              tma_load_2d(st, &P.map[1], kx, f.m0, &full[s]);
            }
            tma_load_2d(st + 2 * kTBox, &P.map[0], kx, f.t0, &full[s]);
          } else {
            // box 0: shared down rows, box 1: h_sh lo, box 2: h_sh hi
            mbar_arrive_expect_tx(&full[s], 3u * kTBox);
            tma_load_2d(st, &P.map[1], kx, f.m0, &full[s]);
            tma_load_2d(st + kTBox, &P.map[2], kx, f.t0, &full[s]);
            tma_load_2d(st + 2 * kTBox, &P.map[0], kx, f.t0, &full[s]);
          }
          issued = p + 1;
        }
      }
      if (*abort)   // copies still in flight land before the CTA's shared memory goes away
        for (int c = issued > kStages ? issued - kStages : 0; c < issued; ++c)
          mbar_wait(&full[c % kStages], uint32_t(c / kStages) & 1u, P.status);
    }
  } else if (warp == kTWMma) {
    // ---- tcgen05.mma issue -----------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTM, kTN);
      uint64_t* last = nullptr;
      uint32_t last_par = 0;
      int p = 0;
      bool ok = true;
      for (int j = 0; j < n_mine && ok; ++j) {
        const Item f = item(j);
        const int ab = j % kTAcc;
        if (j >= kTAcc && !uwait(&acc_empty[ab], uint32_t(j / kTAcc - 1) & 1u, abort, P.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + uint32_t(ab) * kTAccCols, d1 = d0 + kTN;
        for (int ks = 0; ks < nk; ++ks, ++p) {
          const int s = p % kStages;
          const uint32_t par = uint32_t(p / kStages) & 1u;
          if (!uwait(&full[s], par, abort, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = stage0 + uint32_t(s) * kTStageBytes, a1 = a0 + kTBox, b0 = a0 + 2 * kTBox;
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk) {   // K = 16 steps: 32 bytes into the swizzle rows
            const bool acc = ks > 0 || kk > 0;
            const uint64_t da = umma_desc_sw128(a0 + 32 * kk), db = umma_desc_sw128(b0 + 32 * kk);
            umma_bf16(d0, da, db, idesc, acc);
            if (MODE == 0) {
              if (f.big) umma_bf16(d1, umma_desc_sw128(a1 + 32 * kk), db, idesc, acc);
            } else {
              umma_bf16(d0, da, umma_desc_sw128(a1 + 32 * kk), idesc, true);
            }
          }
          umma_commit(&empty[s]);
          last = &empty[s];
          last_par = par;
          if (ks == nk - 1) umma_commit(&acc_full[ab]);
        }
      }
      // every MMA has finished before tensor memory is freed
      if (last) mbar_wait(last, last_par, P.status);
    }
  } else if (MODE == 1 && warp == kTWPart) {
    // ---- combine: part boxes -> ring ------------------------------------------------
    if (lane == 0) {
      tma_prefetch_map(&P.map[3]);
      const uint32_t ring = stage0 + Plan::kPart;
      const uint32_t box_bytes = uint32_t(P.kpt * P.k) * kTM * 4;
      int q = 0, issued = 0;
      bool ok = true;
      for (int j = 0; j < n_mine && ok; ++j) {
        const Item f = item(j);
        const int nb = n_boxes(f);
        for (int u = 0; u < nb; ++u, ++q) {
          const int s = q % kPartRing;
          if (q >= kPartRing && !uwait(&part_empty[s], uint32_t(q / kPartRing - 1) & 1u, abort, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&part_full[s], box_bytes);
          tma_load_2d(ring + uint32_t(s) * kPartBox, &P.map[3], f.m0, (f.t0 + u * P.kpt) * P.k, &part_full[s]);
          issued = q + 1;
        }
      }
      if (*abort)
        for (int c = issued > kPartRing ? issued - kPartRing : 0; c < issued; ++c)
          mbar_wait(&part_full[c % kPartRing], uint32_t(c / kPartRing) & 1u, P.status);
    }
  } else if (warp >= kTWEpi) {
    // ---- epilogue: accumulators -> outputs --------------------------------------------
    const int quarter = warp & 3, half = (warp - kTWEpi) >> 2;
    const int row = quarter * 32 + lane;   // TMEM lane = weight row of the item
    int q = 0;                             // combine: part boxes consumed
    for (int j = 0; j < n_mine; ++j) {
      const int ab = j % kTAcc;
      if (!uwait(&acc_full[ab], uint32_t(j / kTAcc) & 1u, abort, P.status)) break;
      tc_fence_after();
      const Item f = item(j);
      const uint32_t tq = tmem + uint32_t(ab) * kTAccCols + ((uint32_t)(quarter * 32) << 16);
      bool ok = true;
      if (MODE == 0) {
        const int t0 = f.t0 + half * (kTN / 2);
        const uint32_t ta = tq + uint32_t(half * (kTN / 2));
        if (f.big) {
          // feature fe: gate in the first accumulator, up in the second
          const int fe = f.m0 + row;
          const bool fok = fe < P.I;
          for (int c0 = 0; c0 < kTN / 2; c0 += 16) {
            uint32_t g[16], u[16];
            tmem_ld16x2(ta + c0, ta + kTN + c0, g, u);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const int t = t0 + c0 + cc;
              if (fok && t < P.T) {
                const float h = silu_f(__uint_as_float(g[cc])) * __uint_as_float(u[cc]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(h);
                P.hh[(size_t)t * P.I + fe] = hi;
                P.hl[(size_t)t * P.I + fe] = __float2bfloat16_rn(h - __bfloat162float(hi));
              }
            }
          }
        } else {
          const int m = f.m0 + row;   // expert
          const bool mok = m < P.E;
          for (int c0 = 0; c0 < kTN / 2; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(ta + c0, v);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const int t = t0 + c0 + cc;
              if (mok && t < P.T) P.logits[(size_t)t * P.E + m] = __uint_as_float(v[cc]);
            }
          }
        }
      } else {
        // y[t][r] = shared down + sum_j w[t][j] part[t k + j][r], j ascending.
        // Part box u holds tokens f.t0 + u kpt + [0, kpt); this warp takes the
        // half [half kpt / 2, (half + 1) kpt / 2), 4 at a time. The weights of
        // a chunk of 4 tokens are one load per lane (token l / 8, choice l %
        // 8), requested one chunk ahead and handed round by shuffles.
        const int r = f.m0 + row;   // output feature
        const bool rok = r < P.d;
        const int k = P.k, kpt = P.kpt, hp = kpt / 2, nb = n_boxes(f);
        const int jl = lane & 7, il = lane >> 3;
        auto load_w = [&](int u, int c0) {
          const int t = f.t0 + u * kpt + half * hp + c0 + il;
          return (u < nb && jl < k && t < P.T) ? __ldg(P.w + (size_t)t * k + jl) : 0.0f;
        };
        float wn = load_w(0, 0);
        for (int u = 0; u < nb; ++u, ++q) {
          const int s = q % kPartRing;
          if (!uwait(&part_full[s], uint32_t(q / kPartRing) & 1u, abort, P.status)) {
            ok = false;
            break;
          }
          const float* pb = part_smem + (size_t)s * (kPartBox / 4) + row;
          for (int c0 = 0; c0 < hp; c0 += 4) {
            const float wc = wn;
            wn = c0 + 4 < hp ? load_w(u, c0 + 4) : load_w(u + 1, 0);
            const int tl0 = half * hp + c0;    // first token of the 4 within the box
            const int col = u * kpt + tl0;     // its accumulator column
            uint32_t v[4];
            tmem_ld4(tq + uint32_t(col), v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float y = __uint_as_float(v[i]);
              const float* pt = pb + (size_t)(tl0 + i) * k * kTM;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const float wv = __shfl_sync(0xFFFFFFFFu, wc, (i << 3) | jj);
                if (jj < k) y = fmaf(wv, pt[jj * kTM], y);
              }
              const int t = f.t0 + col + i;
              if (rok && t < P.T) P.y[(size_t)t * P.d + r] = __float2bfloat16_rn(y);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&part_empty[s]);
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTWMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTTmemCols);
  }
}

// Tensor map of a row-major matrix [rows][cols] (row stride cols) of bf16
// (box_rows x 64 boxes, 128-byte swizzle) or fp32 (box_rows x 128 boxes, no
// swizzle); zero fill outside the matrix.
int encode_map(CUtensorMap* m, const void* base, int rows, int cols, bool fp32, int box_rows) {
  const uint64_t dims[2] = {uint64_t(cols), uint64_t(rows)};
  const uint64_t strides[1] = {uint64_t(cols) * (fp32 ? 4 : 2)};
  const uint32_t box[2] = {uint32_t(fp32 ? kTM : kTK), uint32_t(box_rows)};
  return tma_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                    strides, box, fp32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE>
int launch_tcd(const TcdParams& P, const DeviceInfo& di, cudaStream_t s) {
  constexpr uint32_t smem = TcdPlan<MODE>::kTotal;
  if (smem > di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int n = P.n_big + P.n_small;
  if (n == 0) return MOE_OK;
  const int grid = n < di.sm_count ? n : di.sm_count;
  MOE_CUDA_TRY(cudaFuncSetAttribute(tc_dense_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
  tc_dense_kernel<MODE><<<grid, kTBlock, smem, s>>>(P);
  return launch_status();
}

}  // namespace

bool tc_dense_supported(int T, int d, int I, int k, bool has_shared, const DeviceInfo& di) {
  return has_shared && T >= 1 && k >= 1 && k <= 8 && d % 8 == 0 && I % 8 == 0 &&
         TcdPlan<0>::kTotal <= di.smem_optin && TcdPlan<1>::kTotal <= di.smem_optin && tma_available();
}

int launch_tc_front(const FrontArgs& a, __nv_bfloat16* h_hi, __nv_bfloat16* h_lo, int* status,
                    const DeviceInfo& di, cudaStream_t s) {
  if (!a.sh_gate || !a.sh_up) return MOE_ERR_INVALID_ARG;
  TcdParams P{};
  int st;
  if ((st = encode_map(&P.map[0], a.x, a.T, a.d, false, kTN))) return st;
  if ((st = encode_map(&P.map[1], a.router_w, a.E, a.d, false, kTM))) return st;
  if ((st = encode_map(&P.map[2], a.sh_gate, a.I, a.d, false, kTM))) return st;
  if ((st = encode_map(&P.map[3], a.sh_up, a.I, a.d, false, kTM))) return st;
  P.T = a.T;
  P.K = a.d;
  P.E = a.E;
  P.I = a.I;
  P.d = a.d;
  const int n_tb = (a.T + kTN - 1) / kTN;
  P.n_fb = (a.I + kTM - 1) / kTM;
  P.n_mb = (a.E + kTM - 1) / kTM;
  P.n_big = P.n_fb * n_tb;
  P.n_small = P.n_mb * n_tb;
  P.logits = a.logits;
  P.hh = h_hi;
  P.hl = h_lo;
  P.status = status;
  return launch_tcd<0>(P, di, s);
}

int launch_tc_combine(const CombineArgs& a, const __nv_bfloat16* h_hi, const __nv_bfloat16* h_lo, int* status,
                      const DeviceInfo& di, cudaStream_t s) {
  if (!a.sh_down || a.k < 1 || a.k > 8) return MOE_ERR_INVALID_ARG;
  TcdParams P{};
  // tokens per part box: the largest power of two with kpt k <= 64 (8 .. 64 for k <= 8)
  int kpt = kTN;
  while (kpt * a.k > kPartRows) kpt >>= 1;
  int st;
  if ((st = encode_map(&P.map[0], h_hi, a.T, a.I, false, kTN))) return st;
  if ((st = encode_map(&P.map[1], a.sh_down, a.d, a.I, false, kTM))) return st;
  if ((st = encode_map(&P.map[2], h_lo, a.T, a.I, false, kTN))) return st;
  if ((st = encode_map(&P.map[3], a.part, a.T * a.k, a.d, true, kpt * a.k))) return st;
  P.T = a.T;
  P.K = a.I;
  P.I = a.I;
  P.d = a.d;
  P.k = a.k;
  P.kpt = kpt;
  const int n_tb = (a.T + kTN - 1) / kTN;
  P.n_fb = 1;
  P.n_mb = (a.d + kTM - 1) / kTM;
  P.n_big = 0;
  P.n_small = P.n_mb * n_tb;
  P.w = a.w;
  P.y = a.y;
  P.status = status;
  return launch_tcd<1>(P, di, s);
}

}  // namespace moe
