// Routing: top-k selection with renormalised softmax weights (one warp per
// token, warp-wide max/min reductions), and the stable token->expert sort used
// for T > 1 (page "MoE-SpeQ ...", §4.2: gather the verify tokens' expert
// assignments, sort them by expert id, run each expert once over its tokens).
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "kernels.h"

namespace moe {

// Order-preserving map fp32 -> uint32 for ranking: larger key = larger value.
// -0 ranks as +0; NaN ranks as -inf; 0 is reserved for "no candidate".
__device__ __forceinline__ uint32_t rank_key(float v) {
  if (isnan(v)) return 0x007FFFFFu;                 // same as -inf
  if (v == 0.0f) v = 0.0f;                         // -0 -> +0
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float rank_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of token t by one warp: the best k keys (logit + bias), equal keys to
// the lower expert index, and their softmax weights; to idx/w (and, if sidx
// is set, idx to sidx too). PL = 32-expert groups per lane.
template <int PL>
__device__ __forceinline__ void topk_token(const float* __restrict__ logits, int t, int E, int k,
                                           const float* __restrict__ bias, int bias_stride, int lane,
                                           int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                           int32_t* sidx) {
  const float* row = logits + (size_t)t * E;
  const float* brow = bias ? bias + (size_t)t * bias_stride : nullptr;
  uint32_t key[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = i * 32 + lane;
    if (e < E) {
      float v = row[e];
      if (brow) v = __fadd_rn(v, brow[e]);
      key[i] = rank_key(v);
    } else {
      key[i] = 0u;
    }
  }
  auto local_best = [&](uint32_t& bk, uint32_t& be) {
    bk = 0u;
    be = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < PL; ++i)
      if (key[i] > bk) { bk = key[i]; be = uint32_t(i * 32 + lane); }   // strict: lowest index wins ties
  };
  uint32_t bk, be;
  local_best(bk, be);
  uint32_t my_e = 0, my_key = 0;
  for (int r = 0; r < k; ++r) {
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, bk == wmax ? be : 0xFFFFFFFFu);
    if (lane == r) { my_e = emin; my_key = wmax; }
    if (lane == int(emin & 31u)) {
      const int slot = int(emin >> 5);
#pragma unroll
      for (int i = 0; i < PL; ++i)
        if (i == slot) key[i] = 0u;
      local_best(bk, be);
    }
  }
  const float v = rank_value(my_key);
  const float v0 = __shfl_sync(0xFFFFFFFFu, v, 0);
  float ex = lane < k ? expf(v - v0) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane < k) {
    idx_out[(size_t)t * k + lane] = int32_t(my_e);
    w_out[(size_t)t * k + lane] = ex / sum;
    if (sidx) sidx[t * k + lane] = int32_t(my_e);
  }
}

template <int PL>
__global__ void __launch_bounds__(128)
topk_kernel(const float* __restrict__ logits, int T, int E, int k, const float* __restrict__ bias,
            int bias_stride, int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_token<PL>(logits, t, E, k, bias, bias_stride, lane, idx_out, w_out, nullptr);
}

// ---- stable sort by expert: counts per token chunk, scan, scatter ----------

constexpr int kSortChunk = 128;   // tokens per chunk (4 mask words)

// True if idx[t][j] is a valid, first occurrence within token t.
__device__ __forceinline__ bool entry_valid(const int32_t* idx, int t, int j, int k, int E) {
  const int e = idx[(size_t)t * k + j];
  if (e < 0 || e >= E) return false;
  for (int jj = 0; jj < j; ++jj)
    if (idx[(size_t)t * k + jj] == e) return false;
  return true;
}

__global__ void __launch_bounds__(256)
sort_count_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ chunk_counts,
                  int* status) {
  extern __shared__ int32_t hist[];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t0 = c * kSortChunk, t1 = min(T, t0 + kSortChunk);
  const int n = (t1 - t0) * k;
  bool bad = false;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int t = t0 + i / k, j = i % k;
    if (entry_valid(idx, t, j, k, E)) atomicAdd(&hist[idx[(size_t)t * k + j]], 1);
    else bad = true;
  }
  if (bad && status) atomicOr(status, MOE_DEV_INDEX_OOB);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)c * E + e] = hist[e];
}

// One block of 1024 threads; E <= 1024.
__global__ void __launch_bounds__(1024)
sort_scan_kernel(const int32_t* __restrict__ chunk_counts, int n_chunks, int E,
                 int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                 int32_t* __restrict__ n_active) {
  __shared__ int32_t warp_sum[2][32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int32_t total = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const int32_t v = chunk_counts[(size_t)c * E + e];
      chunk_base[(size_t)c * E + e] = total;
      total += v;
    }
    counts[e] = total;
  }
  // block-wide exclusive scans of total (-> offsets) and of (total > 0) (-> active slots)
  int32_t a = total, b = total > 0 ? 1 : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, a, o), yb = __shfl_up_sync(0xFFFFFFFFu, b, o);
    if (lane >= o) { a += ya; b += yb; }
  }
  if (lane == 31) { warp_sum[0][warp] = a; warp_sum[1][warp] = b; }
  __syncthreads();
  if (warp == 0) {
    int32_t sa = warp_sum[0][lane], sb = warp_sum[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, sa, o), yb = __shfl_up_sync(0xFFFFFFFFu, sb, o);
      if (lane >= o) { sa += ya; sb += yb; }
    }
    warp_sum[0][lane] = sa;
    warp_sum[1][lane] = sb;
  }
  __syncthreads();
  const int32_t pa = (warp ? warp_sum[0][warp - 1] : 0) + a - total;       // exclusive
  const int32_t pb = (warp ? warp_sum[1][warp - 1] : 0) + b - (total > 0 ? 1 : 0);
  if (e < E) {
    offsets[e] = pa;
    if (total > 0) active[pb] = e;
    for (int c = 0; c < n_chunks; ++c) chunk_base[(size_t)c * E + e] += pa;
  }
  if (e == E - 1) {
    offsets[E] = pa + total;
    *n_active = pb + (total > 0 ? 1 : 0);
  }
}

__global__ void __launch_bounds__(256)
sort_scatter_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm,
                    int32_t* __restrict__ inv) {
  extern __shared__ uint32_t mask[];   // [E][4]: tokens of this chunk that chose e
  const int c = blockIdx.x;
  for (int i = threadIdx.x; i < E * 4; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int t0 = c * kSortChunk, t1 = min(T, t0 + kSortChunk);
  const int n = (t1 - t0) * k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int tl = i / k, j = i % k;
    if (entry_valid(idx, t0 + tl, j, k, E))
      atomicOr(&mask[idx[(size_t)(t0 + tl) * k + j] * 4 + (tl >> 5)], 1u << (tl & 31));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int tl = i / k, j = i % k;
    const int p = (t0 + tl) * k + j;
    if (!entry_valid(idx, t0 + tl, j, k, E)) { inv[p] = -1; continue; }
    const int e = idx[p];
    const uint32_t* m = mask + e * 4;
    int rank = 0;
    for (int wv = 0; wv < (tl >> 5); ++wv) rank += __popc(m[wv]);
    rank += __popc(m[tl >> 5] & ((1u << (tl & 31)) - 1u));
    const int pos = chunk_base[(size_t)c * E + e] + rank;
    perm[pos] = p;
    inv[p] = pos;
  }
}

// ---- the sort of one chunk (T <= kSortChunk) in one block, with or without
// the top-k before it ------------------------------------------------------------
// The same steps as the three sort kernels for one chunk: thread e < E owns
// expert e for the counts and the scans (offsets, active list); the scatter
// ranks each entry among the chunk's tokens that chose its expert (bit
// masks). With TOPK (T <= 32) warp w first ranks tokens w, w + 32, ... as
// topk_kernel does: one launch instead of four; without it the entries come
// from idx: one launch instead of three.
template <int PL, bool TOPK>
__global__ void __launch_bounds__(1024)
route_small_kernel(const float* __restrict__ logits, int T, int E, int k, const float* __restrict__ bias,
                   int bias_stride, int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                   int32_t* __restrict__ active, int32_t* __restrict__ n_active, int* status) {
  extern __shared__ uint32_t rs[];
  int32_t* base = reinterpret_cast<int32_t*>(rs);        // [E]: counts, then first sorted slot
  uint32_t* mask = rs + E;                               // [E][4]: tokens that chose e
  int32_t* sidx = reinterpret_cast<int32_t*>(mask + 4 * E);   // [T k]
  __shared__ int32_t warp_sum[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 5 * E; i += blockDim.x) rs[i] = 0u;
  if constexpr (TOPK) {
    for (int t = warp; t < T; t += 32) topk_token<PL>(logits, t, E, k, bias, bias_stride, lane, idx, w, sidx);
  } else {
    for (int i = tid; i < T * k; i += blockDim.x) sidx[i] = idx[i];
  }
  __syncthreads();
  const int n = T * k;
  auto valid = [&](int t, int j) {   // in range, and the token's first entry of its expert
    const int e = sidx[t * k + j];
    if (e < 0 || e >= E) return false;
    for (int jj = 0; jj < j; ++jj)
      if (sidx[t * k + jj] == e) return false;
    return true;
  };
  bool bad = false;
  for (int i = tid; i < n; i += blockDim.x) {
    const int t = i / k, j = i - t * k;
    if (valid(t, j)) {
      const int e = sidx[i];
      atomicAdd(&base[e], 1);
      atomicOr(&mask[e * 4 + (t >> 5)], 1u << (t & 31));
    } else {
      bad = true;
    }
  }
  if (bad && status) atomicOr(status, MOE_DEV_INDEX_OOB);
  __syncthreads();
  // exclusive scans of the counts (-> offsets) and of (count > 0) (-> active)
  const int e = tid;
  const int32_t total = e < E ? base[e] : 0;
  int32_t a = total, b = total > 0 ? 1 : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, a, o), yb = __shfl_up_sync(0xFFFFFFFFu, b, o);
    if (lane >= o) { a += ya; b += yb; }
  }
  if (lane == 31) { warp_sum[0][warp] = a; warp_sum[1][warp] = b; }
  __syncthreads();
  if (warp == 0) {
    int32_t sa = warp_sum[0][lane], sb = warp_sum[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, sa, o), yb = __shfl_up_sync(0xFFFFFFFFu, sb, o);
      if (lane >= o) { sa += ya; sb += yb; }
    }
    warp_sum[0][lane] = sa;
    warp_sum[1][lane] = sb;
  }
  __syncthreads();
  const int32_t pa = (warp ? warp_sum[0][warp - 1] : 0) + a - total;
  const int32_t pb = (warp ? warp_sum[1][warp - 1] : 0) + b - (total > 0 ? 1 : 0);
  if (e < E) {
    counts[e] = total;
    offsets[e] = pa;
    if (total > 0) active[pb] = e;
    base[e] = pa;
  }
  if (e == E - 1) {
    offsets[E] = pa + total;
    *n_active = pb + (total > 0 ? 1 : 0);
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const int t = i / k, j = i - t * k;
    if (!valid(t, j)) {
      inv[i] = -1;
      continue;
    }
    const uint32_t* m = mask + sidx[i] * 4;
    int rank = 0;
    for (int wv = 0; wv < (t >> 5); ++wv) rank += __popc(m[wv]);
    rank += __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
    const int pos = base[sidx[i]] + rank;
    perm[pos] = i;
    inv[i] = pos;
  }
}

// ---- launchers --------------------------------------------------------------

int launch_topk(const float* logits, int T, int E, int k, const float* bias, int bias_stride,
                int32_t* idx, float* w, cudaStream_t s) {
  const int grid = (T + 3) / 4;
  const int pl = (E + 31) / 32;
#define MOE_TOPK_CASE(P)                                                               \
  topk_kernel<P><<<grid, 128, 0, s>>>(logits, T, E, k, bias, bias_stride, idx, w); \
  break;
  switch (pl <= 1 ? 1 : pl <= 2 ? 2 : pl <= 4 ? 4 : pl <= 8 ? 8 : pl <= 16 ? 16 : 32) {
    case 1: MOE_TOPK_CASE(1)
    case 2: MOE_TOPK_CASE(2)
    case 4: MOE_TOPK_CASE(4)
    case 8: MOE_TOPK_CASE(8)
    case 16: MOE_TOPK_CASE(16)
    default: MOE_TOPK_CASE(32)
  }
#undef MOE_TOPK_CASE
  return launch_status();
}

// One warp per token: beyond 32 tokens a warp would rank several in turn,
// slower than the separate top-k kernel's one warp per token across the GPU.
bool route_fused_ok(int T, int E, int k) { return T <= 32 && E <= 1024 && k <= 32; }

int launch_route_fused(const float* logits, int T, int E, int k, const float* bias, int bias_stride,
                       int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                       int32_t* active, int32_t* n_active, int* status, cudaStream_t s) {
  if (!route_fused_ok(T, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const size_t smem = (size_t)5 * E * 4 + (size_t)T * k * 4;
  const int pl = (E + 31) / 32;
#define MOE_ROUTE_CASE(P)                                                                                         \
  route_small_kernel<P, true><<<1, 1024, smem, s>>>(logits, T, E, k, bias, bias_stride, idx, w, counts, offsets, \
                                                    perm, inv, active, n_active, status);                        \
  break;
  switch (pl <= 1 ? 1 : pl <= 2 ? 2 : pl <= 4 ? 4 : pl <= 8 ? 8 : pl <= 16 ? 16 : 32) {
    case 1: MOE_ROUTE_CASE(1)
    case 2: MOE_ROUTE_CASE(2)
    case 4: MOE_ROUTE_CASE(4)
    case 8: MOE_ROUTE_CASE(8)
    case 16: MOE_ROUTE_CASE(16)
    default: MOE_ROUTE_CASE(32)
  }
#undef MOE_ROUTE_CASE
  return launch_status();
}

size_t sort_workspace_bytes(int T, int E) {
  const size_t chunks = (size_t)(T + kSortChunk - 1) / kSortChunk;
  return 2 * round_up(chunks * E * sizeof(int32_t), 256);
}

int launch_sort(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                int32_t* perm, int32_t* inv, int32_t* active, int32_t* n_active, void* ws,
                int* status, cudaStream_t s) {
  const int chunks = (T + kSortChunk - 1) / kSortChunk;
  if (chunks == 1 && E <= 1024 && k <= 32) {   // one chunk: one block, one launch
    const size_t smem = (size_t)5 * E * 4 + (size_t)T * k * 4;
    route_small_kernel<1, false><<<1, 1024, smem, s>>>(nullptr, T, E, k, nullptr, 0, const_cast<int32_t*>(idx),
                                                       nullptr, counts, offsets, perm, inv, active, n_active, status);
    return launch_status();
  }
  int32_t* chunk_counts = static_cast<int32_t*>(ws);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                                   round_up((size_t)chunks * E * sizeof(int32_t), 256));
  sort_count_kernel<<<chunks, 256, E * sizeof(int32_t), s>>>(idx, T, k, E, chunk_counts, status);
  sort_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, chunks, E, chunk_base, counts, offsets, active,
                                      n_active);
  sort_scatter_kernel<<<chunks, 256, E * 4 * sizeof(uint32_t), s>>>(idx, T, k, E, chunk_base, perm,
                                                                    inv);
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route_topk(const float* logits_dev, int T, int E, int k, const float* bias_dev,
                              int bias_row_stride, int32_t* idx_dev, float* w_dev,
                              moe_stream_t stream) {
  MOE_CHECK_ARG(logits_dev && idx_dev && w_dev, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(T >= 1 && E >= 1 && k >= 1, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(E <= 1024 && k <= 32 && k <= E, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK_ARG(bias_row_stride == 0 || bias_row_stride >= E, MOE_ERR_INVALID_ARG);
  DeviceInfo di;
  int st = current_device(&di);
  if (st != MOE_OK) return st;
  return launch_topk(logits_dev, T, E, k, bias_dev, bias_row_stride, idx_dev, w_dev,
                     (cudaStream_t)stream);
}

extern "C" size_t moe_sort_workspace_bytes(int T, int k, int E) {
  (void)k;
  if (T < 1 || E < 1 || E > 1024) return 0;
  return sort_workspace_bytes(T, E);
}

extern "C" int moe_sort_by_expert(const int32_t* idx_dev, int T, int k, int E, int32_t* counts_dev,
                                  int32_t* offsets_dev, int32_t* perm_dev, int32_t* inv_dev,
                                  int32_t* active_dev, int32_t* n_active_dev, void* workspace_dev,
                                  size_t workspace_bytes, int* dev_status, moe_stream_t stream) {
  MOE_CHECK_ARG(idx_dev && counts_dev && offsets_dev && perm_dev && inv_dev && active_dev &&
                    n_active_dev && workspace_dev,
                MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(T >= 1 && k >= 1 && E >= 1, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(E <= 1024 && k <= 32, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK_ARG(workspace_bytes >= sort_workspace_bytes(T, E), MOE_ERR_WORKSPACE_TOO_SMALL);
  DeviceInfo di;
  int st = current_device(&di);
  if (st != MOE_OK) return st;
  return launch_sort(idx_dev, T, k, E, counts_dev, offsets_dev, perm_dev, inv_dev, active_dev,
                     n_active_dev, workspace_dev, dev_status, (cudaStream_t)stream);
}
