// C-ABI entry points for the layer: argument and descriptor checks, workspace
// carving, and the kernel sequence of one forward call.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "host_util.h"
#include "kernels.h"

namespace moe {

int current_device(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& c = cache[dev];
  if (c.device != dev) {
    DeviceInfo d;
    d.device = dev;
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev));
    int optin = 0;
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    d.smem_optin = size_t(optin);
    c = d;
  }
  if (c.major != 10 || c.minor != 3) return MOE_ERR_NO_DEVICE;
  *out = c;
  return MOE_OK;
}

namespace {

// Tokens from which the routed experts run as tcgen05 grouped GEMMs (below
// it, and only where the single-launch kernel cannot take the shape, they
// run as warp-MMA GEMVs): measured faster than the warp-MMA path from 5.
constexpr int kPrefillMinT = 5;
// Tensor-core path: the combine (shared down + weighted sum) always runs as a
// tcgen05 GEMM; the router + shared gate/up do from this many tokens (below
// it their 10 or so 128-row blocks leave most SMs idle).
constexpr int kFrontTcMinT = 128;
// Tensor-core routed GEMMs: items of up to 64 B rows (32 tokens with two
// activation terms, 64 with one) while the mean tokens per expert, T k / E,
// stays below 3/4 of that, else of up to 128 B rows. Graph-timed at the Ling
// shape: 64-row items 896 against 968 us at T=1024, 128-row items 1,063
// against 1,291 us at T=2048.
constexpr int kNarrowRowsPerExpert = 48;   // T k terms < this x E: 64-row items

// Workspace sections of one forward call (byte offsets from the base).
struct Workspace {
  size_t state, logits, idx, w, sort_ws, counts, offsets, perm, inv, active, n_active, status;
  size_t x_b, x_e, h_sh, h, h_b, h_e, part, xq, xs, hq, hs, total;
};

Workspace plan(const moe_shape& sh, int T) {
  Workspace o{};
  const size_t d = size_t(sh.d_model), I = size_t(sh.d_ff), E = size_t(sh.n_experts),
               k = size_t(sh.top_k), slots = size_t(T) * k;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at += round_up(bytes, 256);
    return here;
  };
  o.state = take(decode_state_bytes(T, int(E)));   // persists across calls
  o.logits = take(size_t(T) * E * 4);
  o.idx = take(slots * 4);
  o.w = take(slots * 4);
  o.sort_ws = take(sort_workspace_bytes(T, int(E)));
  o.counts = take(E * 4);
  o.offsets = take((E + 1) * 4);
  o.perm = take(slots * 4);
  o.inv = take(slots * 4);
  o.active = take(E * 4);
  o.n_active = take(4);
  o.status = take(4);
  o.x_b = take(size_t(T) * (d / 32) * kActRowKbBytes);
  o.x_e = take(size_t(T) * (d / 32) * 2);
  o.h_sh = take(size_t(T) * I * 4);
  o.h = take(slots * I * 4);
  o.h_b = take(slots * (I / 32) * kActRowKbBytes);
  o.h_e = take(slots * decode_he_stride(int(I)) * 2);
  o.part = take(slots * d * 4);
  // activations of the tcgen05 path as E4M3 terms (up to 2) + E8M0 scales
  o.xq = take(size_t(T) * 2 * d);
  o.xs = take(size_t(T) * (d / 32));
  o.hq = take(slots * 2 * I);
  o.hs = take(slots * (I / 32));
  o.total = at;
  return o;
}

int check_shape(const moe_shape* sh, int T) {
  if (!sh) return MOE_ERR_INVALID_ARG;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if (sh->d_model < 32 || sh->d_ff < 32 || sh->n_experts < 1 || sh->top_k < 1) return MOE_ERR_INVALID_ARG;
  if (sh->d_model % 32 || sh->d_ff % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (sh->n_experts > 1024 || sh->top_k > 32 || sh->top_k > sh->n_experts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (sh->has_shared != 0 && sh->has_shared != 1) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool desc_matches(const moe_packed_desc& d, int layout, int n_mat, int N, int K) {
  return d.magic == MOE_PACK_MAGIC && d.version == MOE_PACK_VERSION && d.layout == layout &&
         d.n_mat == n_mat && d.N == N && d.K == K &&
         d.bytes_per_mat == (uint64_t)N * K / 2 + (uint64_t)N * K / 32 &&
         d.total_bytes == d.bytes_per_mat * (uint64_t)n_mat;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_workspace_bytes(const moe_shape* shape, int T) {
  if (check_shape(shape, T) != MOE_OK) return 0;
  return plan(*shape, T).total;
}

// Path for (shape, T) on the current device: the single-launch decode kernel
// when T <= 4 and the shape fits it; the per-stage kernels with tcgen05
// routed GEMMs from kPrefillMinT tokens; else the per-stage kernels.
static int select_path(const moe_shape& sh, int T, const DeviceInfo& di) {
  DecodeArgs probe{};
  probe.T = T;
  probe.d = sh.d_model;
  probe.I = sh.d_ff;
  probe.E = sh.n_experts;
  probe.k = sh.top_k;
  uint32_t smem;
  if (T <= kDecodeMaxT && decode_plan(probe, di, &smem) == MOE_OK) return MOE_PATH_DECODE_FUSED;
  if (T >= kPrefillMinT) return MOE_PATH_PREFILL_TC;
  return MOE_PATH_DECODE_MMA;
}

extern "C" int moe_query_path(const moe_shape* shape, int T) {
  const int st = check_shape(shape, T);
  if (st != MOE_OK) return st;
  DeviceInfo di;
  const int dst = current_device(&di);
  if (dst != MOE_OK) return dst;
  return select_path(*shape, T, di);
}

namespace moe {
namespace {

// Every argument check of a forward call, done before anything is enqueued.
// On MOE_OK, *ws holds the workspace plan and *di the current device.
int validate_forward(const moe_layer* L, const void* x_dev, int T, const void* y_dev, int bias_row_stride,
                     const void* workspace_dev, size_t workspace_bytes, Workspace* ws, DeviceInfo* di) {
  MOE_CHECK_ARG(L && x_dev && y_dev && workspace_dev, MOE_ERR_INVALID_ARG);
  int st = check_shape(&L->shape, T);
  if (st != MOE_OK) return st;
  const moe_shape& sh = L->shape;
  const int d = sh.d_model, I = sh.d_ff, E = sh.n_experts;
  MOE_CHECK_ARG(L->router_w && L->gate_up && L->down, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(!sh.has_shared || (L->shared_gate && L->shared_up && L->shared_down), MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(bias_row_stride == 0 || bias_row_stride >= E, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(x_dev != y_dev, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(desc_matches(L->gate_up_desc, MOE_LAYOUT_TILE16_GATEUP, E, 2 * I, d), MOE_ERR_BAD_DESCRIPTOR);
  MOE_CHECK_ARG(desc_matches(L->down_desc, MOE_LAYOUT_TILE16, E, d, I), MOE_ERR_BAD_DESCRIPTOR);
  MOE_CHECK_ARG(aligned(L->gate_up, 16) && aligned(L->down, 16) && aligned(L->router_w, 16) &&
                    aligned(x_dev, 16) && aligned(workspace_dev, 256),
                MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(!sh.has_shared || (aligned(L->shared_gate, 16) && aligned(L->shared_up, 16) &&
                                   aligned(L->shared_down, 16)),
                MOE_ERR_INVALID_ARG);
  *ws = plan(sh, T);
  MOE_CHECK_ARG(workspace_bytes >= ws->total, MOE_ERR_WORKSPACE_TOO_SMALL);
  return current_device(di);
}

// The kernel sequence of one validated forward call on `stream`; stage_events
// as in moe_forward_profiled (n_stage_events 0: none).
int enqueue_forward(const moe_layer* L, const void* x_dev, int T, void* y_dev, const float* bias_dev,
                    int bias_row_stride, float* logits_out, int32_t* idx_out, float* w_out, void* workspace_dev,
                    int* dev_status, void* const* stage_events, int n_stage_events, moe_stream_t stream,
                    const Workspace& ws, const DeviceInfo& di, bool act_mxfp8 = false) {
  int st = MOE_OK;
  const moe_shape& sh = L->shape;
  const int d = sh.d_model, I = sh.d_ff, E = sh.n_experts, k = sh.top_k;
  cudaStream_t s = (cudaStream_t)stream;
  void* B = workspace_dev;
  float* logits = logits_out ? logits_out : at<float>(B, ws.logits);
  int32_t* idx = idx_out ? idx_out : at<int32_t>(B, ws.idx);
  float* w = w_out ? w_out : at<float>(B, ws.w);
  int* status = dev_status ? dev_status : at<int>(B, ws.status);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(x_dev);
  // Under stream capture an event record must be an external node to be
  // timed on replay; outside capture the flag records as usual.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (n_stage_events > 0) MOE_CUDA_TRY(cudaStreamIsCapturing(s, &cap));
  const unsigned ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  int mark_i = 0;
  auto mark = [&]() -> int {
    if (mark_i < n_stage_events && stage_events[mark_i]) {
      if (cudaEventRecordWithFlags((cudaEvent_t)stage_events[mark_i], s, ev_flags) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
      }
    }
    ++mark_i;
    return MOE_OK;
  };
  if ((st = mark())) return st;

  const int path = act_mxfp8 ? MOE_PATH_PREFILL_TC : select_path(sh, T, di);
  if (path == MOE_PATH_DECODE_FUSED) {
    DecodeArgs da{};
    da.T = T;
    da.d = d;
    da.I = I;
    da.E = E;
    da.k = k;
    da.has_shared = sh.has_shared;
    da.x = x;
    da.router_w = static_cast<const __nv_bfloat16*>(L->router_w);
    da.sh_gate = sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_gate) : nullptr;
    da.sh_up = sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_up) : nullptr;
    da.sh_down = sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_down) : nullptr;
    da.gate_up = static_cast<const uint8_t*>(L->gate_up);
    da.down = static_cast<const uint8_t*>(L->down);
    da.gu_mat = L->gate_up_desc.bytes_per_mat;
    da.dn_mat = L->down_desc.bytes_per_mat;
    da.bias = bias_dev;
    da.bias_stride = bias_row_stride;
    da.logits = logits;
    da.idx_out = idx_out;
    da.w_out = w_out;
    da.y = static_cast<__nv_bfloat16*>(y_dev);
    da.state = at<DecodeState>(B, ws.state);
    da.h = at<uint8_t>(B, ws.h);   // decode_h_bytes(T, k, I) <= slots * I * 4
    da.h_sh = at<float>(B, ws.h_sh);
    da.status = status;
    if ((st = launch_decode(da, di, s))) return st;
    return mark();
  }

  const bool tc = path == MOE_PATH_PREFILL_TC;
  // 1. activations -> e4m3 B-operand terms (the tcgen05 path reads x as bf16)
  if (!tc) {
    if ((st = launch_act_split(x, true, T, d, at<uint8_t>(B, ws.x_b), at<int16_t>(B, ws.x_e), di, s))) return st;
    if ((st = mark())) return st;
  }
  // 2. router logits and shared gate/up (routing-independent)
  FrontArgs fa{x, T, d, E, I, static_cast<const __nv_bfloat16*>(L->router_w),
               sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_gate) : nullptr,
               sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_up) : nullptr, logits,
               at<float>(B, ws.h_sh)};
  // tcgen05 dense stages: h_sh as bf16 hi and lo terms in the fp32 h_sh section
  const bool tcd = tc && tc_dense_supported(T, d, I, k, sh.has_shared != 0, di);
  __nv_bfloat16* h_hi = at<__nv_bfloat16>(B, ws.h_sh);
  __nv_bfloat16* h_lo = h_hi + (size_t)T * I;
  if (tcd) {
    fa.h_hi = h_hi;
    fa.h_lo = h_lo;
  }
  if ((st = tcd && T >= kFrontTcMinT ? launch_tc_front(fa, h_hi, h_lo, status, di, s) : launch_front(fa, di, s)))
    return st;
  if ((st = mark())) return st;
  // 3. top-k + weights, 4. sort by expert (one launch for up to 32 tokens;
  // the sort stage is then empty)
  int32_t* offsets = at<int32_t>(B, ws.offsets);
  int32_t* perm = at<int32_t>(B, ws.perm);
  int32_t* inv = at<int32_t>(B, ws.inv);
  int32_t* active = at<int32_t>(B, ws.active);
  int32_t* n_active = at<int32_t>(B, ws.n_active);
  if (route_fused_ok(T, E, k)) {
    if ((st = launch_route_fused(logits, T, E, k, bias_dev, bias_row_stride, idx, w, at<int32_t>(B, ws.counts),
                                 offsets, perm, inv, active, n_active, status, s)))
      return st;
    if ((st = mark())) return st;
  } else {
    if ((st = launch_topk(logits, T, E, k, bias_dev, bias_row_stride, idx, w, s))) return st;
    if ((st = mark())) return st;
    if ((st = launch_sort(idx, T, k, E, at<int32_t>(B, ws.counts), offsets, perm, inv, active, n_active,
                          at<void>(B, ws.sort_ws), status, s)))
      return st;
  }
  if ((st = mark())) return st;
  const int max_active = T * k < E ? T * k : E;
  if (tc) {
    // x -> E4M3 terms with E8M0 scales per 32 (MXFP8 for the 8-bit-activation
    // call, else two terms of bf16 precision); routed gate/up on block-scaled
    // tcgen05 MMAs -> h fp32 [slots][I]; h -> E4M3 terms; routed down -> part
    // [slots][d]; shared down + combine
    const int qmode = act_mxfp8 ? kQuantMxfp8 : kQuantSplit2;
    const int nterms = act_mxfp8 ? 1 : 2;
    if ((st = launch_act_quant(x, true, T, d, qmode, at<uint8_t>(B, ws.xq), at<uint8_t>(B, ws.xs), s))) return st;
    if ((st = mark())) return st;
    RoutedArgs ua{};
    ua.w = static_cast<const uint8_t*>(L->gate_up);
    ua.mat_bytes = L->gate_up_desc.bytes_per_mat;
    ua.n_tiles = 2 * I / kTileRows;
    ua.KB = d / kMxBlock;
    ua.active = active;
    ua.n_active = n_active;
    ua.offsets = offsets;
    ua.perm = perm;
    ua.k = k;
    ua.act_q = at<uint8_t>(B, ws.xq);
    ua.act_s = at<uint8_t>(B, ws.xs);
    ua.act_terms = nterms;
    ua.narrow = (int64_t)T * k * nterms < (int64_t)kNarrowRowsPerExpert * E ? 1 : 0;
    ua.out = at<float>(B, ws.h);
    ua.out_ld = I;
    ua.status = status;
    if ((st = launch_umma_routed(kModeGateUp, ua, di, s))) return st;
    if ((st = mark())) return st;
    if ((st = launch_act_quant(at<float>(B, ws.h), false, T * k, I, qmode, at<uint8_t>(B, ws.hq),
                               at<uint8_t>(B, ws.hs), s)))
      return st;
    if ((st = mark())) return st;
    RoutedArgs ud = ua;
    ud.w = static_cast<const uint8_t*>(L->down);
    ud.mat_bytes = L->down_desc.bytes_per_mat;
    ud.n_tiles = d / kTileRows;
    ud.KB = I / kMxBlock;
    ud.act_q = at<uint8_t>(B, ws.hq);
    ud.act_s = at<uint8_t>(B, ws.hs);
    ud.out = at<float>(B, ws.part);
    ud.out_ld = d;
    ud.out_by_pair = tcd ? 1 : 0;   // the tcgen05 combine reads part in (token, choice) order
    if ((st = launch_umma_routed(kModeDown, ud, di, s))) return st;
    if ((st = mark())) return st;
    CombineArgs ca{T, d, I, k,
                   sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_down) : nullptr,
                   at<float>(B, ws.h_sh), w, inv, at<float>(B, ws.part),
                   static_cast<__nv_bfloat16*>(y_dev)};
    if ((st = tcd ? launch_tc_combine(ca, h_hi, h_lo, status, di, s) : launch_combine(ca, di, s))) return st;
    return mark();
  }
  // 5. routed gate/up + SwiGLU -> h [slots][I]
  RoutedArgs ra{};
  ra.w = static_cast<const uint8_t*>(L->gate_up);
  ra.mat_bytes = L->gate_up_desc.bytes_per_mat;
  ra.n_tiles = 2 * I / kTileRows;
  ra.KB = d / kMxBlock;
  ra.active = active;
  ra.n_active = n_active;
  ra.offsets = offsets;
  ra.perm = perm;
  ra.k = k;
  ra.act_b = at<uint8_t>(B, ws.x_b);
  ra.act_e = at<int16_t>(B, ws.x_e);
  ra.act_by_token = 1;
  ra.max_items = (max_active + (T * k + 7) / 8) * ra.n_tiles;   // (expert, 8-row chunk, tile) items
  ra.out = at<float>(B, ws.h);
  ra.out_ld = I;
  ra.status = status;
  if ((st = launch_routed(kModeGateUp, ra, di, s))) return st;
  if ((st = mark())) return st;
  // 6. h -> e4m3 terms
  const int slots = T * k;
  if ((st = launch_act_split(at<float>(B, ws.h), false, slots, I, at<uint8_t>(B, ws.h_b),
                             at<int16_t>(B, ws.h_e), di, s)))
    return st;
  if ((st = mark())) return st;
  // 7. routed down -> part [slots][d]
  RoutedArgs rd = ra;
  rd.w = static_cast<const uint8_t*>(L->down);
  rd.mat_bytes = L->down_desc.bytes_per_mat;
  rd.n_tiles = d / kTileRows;
  rd.KB = I / kMxBlock;
  rd.act_b = at<uint8_t>(B, ws.h_b);
  rd.act_e = at<int16_t>(B, ws.h_e);
  rd.act_by_token = 0;
  rd.max_items = (max_active + (T * k + 7) / 8) * rd.n_tiles;
  rd.out = at<float>(B, ws.part);
  rd.out_ld = d;
  if ((st = launch_routed(kModeDown, rd, di, s))) return st;
  if ((st = mark())) return st;
  // 8. shared down + weighted combine -> y bf16
  CombineArgs ca{T, d, I, k,
                 sh.has_shared ? static_cast<const __nv_bfloat16*>(L->shared_down) : nullptr,
                 at<float>(B, ws.h_sh), w, inv, at<float>(B, ws.part),
                 static_cast<__nv_bfloat16*>(y_dev)};
  if ((st = launch_combine(ca, di, s))) return st;
  return mark();
}

}  // namespace
}  // namespace moe

extern "C" int moe_forward(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                           const float* bias_dev, int bias_row_stride, float* logits_out,
                           int32_t* idx_out, float* w_out, void* workspace_dev,
                           size_t workspace_bytes, int* dev_status, moe_stream_t stream) {
  Workspace ws;
  DeviceInfo di;
  const int st = validate_forward(L, x_dev, T, y_dev, bias_row_stride, workspace_dev, workspace_bytes, &ws, &di);
  if (st != MOE_OK) return st;
  return enqueue_forward(L, x_dev, T, y_dev, bias_dev, bias_row_stride, logits_out, idx_out, w_out, workspace_dev,
                         dev_status, nullptr, 0, stream, ws, di);
}

extern "C" int moe_forward_profiled(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                                    const float* bias_dev, int bias_row_stride, float* logits_out,
                                    int32_t* idx_out, float* w_out, void* workspace_dev,
                                    size_t workspace_bytes, int* dev_status, void* const* stage_events,
                                    int n_stage_events, moe_stream_t stream) {
  MOE_CHECK_ARG(n_stage_events >= 0 && (stage_events || n_stage_events == 0), MOE_ERR_INVALID_ARG);
  Workspace ws;
  DeviceInfo di;
  const int st = validate_forward(L, x_dev, T, y_dev, bias_row_stride, workspace_dev, workspace_bytes, &ws, &di);
  if (st != MOE_OK) return st;
  return enqueue_forward(L, x_dev, T, y_dev, bias_dev, bias_row_stride, logits_out, idx_out, w_out, workspace_dev,
                         dev_status, stage_events, n_stage_events, stream, ws, di);
}

extern "C" int moe_forward_w4a8(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                                const float* bias_dev, int bias_row_stride, float* logits_out,
                                int32_t* idx_out, float* w_out, void* workspace_dev,
                                size_t workspace_bytes, int* dev_status, moe_stream_t stream) {
  Workspace ws;
  DeviceInfo di;
  const int st = validate_forward(L, x_dev, T, y_dev, bias_row_stride, workspace_dev, workspace_bytes, &ws, &di);
  if (st != MOE_OK) return st;
  return enqueue_forward(L, x_dev, T, y_dev, bias_dev, bias_row_stride, logits_out, idx_out, w_out, workspace_dev,
                         dev_status, nullptr, 0, stream, ws, di, true);
}

namespace moe {
namespace {
// Scratch of moe_forward_static_scratch: part of this library's device image,
// one copy per device, so that entry point needs no allocation. Every call on
// a device uses the same bytes.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

// Identity of the calling thread's current CUDA context (0 if it has none).
// A device's primary context gets a new identity when it is destroyed and
// created again (cudaDeviceReset), which invalidates device addresses.
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);                  // cuCtxGetCurrent
  using GetId = int (*)(void*, unsigned long long*);   // cuCtxGetId
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    (void)cudaGetLastError();
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of g_static_scratch on device `dev` (the current device).
// It is looked up with cudaGetSymbolAddress the first time the device calls,
// and again whenever the device's context has changed since (after a
// cudaDeviceReset the old address is no longer valid).
int static_scratch_address(int dev, void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  static unsigned long long cache_ctx[64] = {};
  if (dev < 0 || dev >= 64) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (!cache[dev] || ctx == 0 || ctx != cache_ctx[dev]) {
    void* p = nullptr;
    MOE_CUDA_TRY(cudaGetSymbolAddress(&p, g_static_scratch));
    if (!p) return MOE_ERR_CUDA;
    cache[dev] = p;
    cache_ctx[dev] = current_context_id();   // the lookup made the context current if it was not
  }
  *out = cache[dev];
  return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" int moe_forward_static_scratch(const moe_layer* L, const void* x_dev, int T, void* y_dev,
                                          const float* bias_dev, int bias_row_stride, float* logits_out,
                                          int32_t* idx_out, float* w_out, int* dev_status,
                                          moe_stream_t stream) {
  MOE_CHECK_ARG(L && x_dev && y_dev, MOE_ERR_INVALID_ARG);
  int st = check_shape(&L->shape, T);
  if (st != MOE_OK) return st;
  if (plan(L->shape, T).total > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo di;
  if ((st = current_device(&di))) return st;
  void* scratch = nullptr;
  if ((st = static_scratch_address(di.device, &scratch))) return st;
  // every check of moe_forward, before anything is enqueued
  Workspace ws;
  st = validate_forward(L, x_dev, T, y_dev, bias_row_stride, scratch, MOE_STATIC_SCRATCH_BYTES, &ws, &di);
  if (st != MOE_OK) return st;
  // The synchronisation counters at the head of the workspace must read zero
  // when the call's kernels start; clear them on the call's own stream so a
  // call never depends on how an earlier one ended.
  MOE_CUDA_TRY(cudaMemsetAsync(static_cast<char*>(scratch) + ws.state, 0,
                               decode_state_bytes(T, L->shape.n_experts), (cudaStream_t)stream));
  return enqueue_forward(L, x_dev, T, y_dev, bias_dev, bias_row_stride, logits_out, idx_out, w_out, scratch,
                         dev_status, nullptr, 0, stream, ws, di);
}

extern "C" int moe_quant_mxfp8(const void* src_dev, int src_is_bf16, int rows, int K, uint8_t* codes_dev,
                               uint8_t* scales_dev, moe_stream_t stream) {
  MOE_CHECK_ARG(src_dev && codes_dev && scales_dev && rows >= 0 && K > 0, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(src_is_bf16 == 0 || src_is_bf16 == 1, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(K % 32 == 0, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK_ARG(aligned(src_dev, 16) && aligned(codes_dev, 16), MOE_ERR_INVALID_ARG);
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != MOE_OK) return st;
  return launch_act_quant(src_dev, src_is_bf16 != 0, rows, K, kQuantMxfp8, codes_dev, scales_dev,
                          (cudaStream_t)stream);
}

extern "C" int moe_lmhead_pack_fp8(const void* w_dev, int V, int d, uint8_t* codes_dev, float* scales_dev,
                                   moe_stream_t stream) {
  MOE_CHECK_ARG(w_dev && codes_dev && scales_dev && V > 0 && d > 0, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(d % 2 == 0 && aligned(codes_dev, 2), MOE_ERR_UNSUPPORTED_SHAPE);
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != MOE_OK) return st;
  return launch_lm_pack(w_dev, V, d, codes_dev, scales_dev, (cudaStream_t)stream);
}

extern "C" int moe_lmhead_fp8(const uint8_t* codes_dev, const float* scales_dev, int V, int d, const void* x_dev,
                              int T, float* logits_dev, moe_stream_t stream) {
  MOE_CHECK_ARG(codes_dev && scales_dev && x_dev && logits_dev && V > 0 && d > 0 && T >= 1, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(V % 16 == 0 && d % 64 == 0 && T <= 8, MOE_ERR_UNSUPPORTED_SHAPE);
  MOE_CHECK_ARG(aligned(codes_dev, 8) && aligned(x_dev, 16), MOE_ERR_INVALID_ARG);
  DeviceInfo di;
  const int st = current_device(&di);
  if (st != MOE_OK) return st;
  return launch_lm_gemv(codes_dev, scales_dev, V, d, x_dev, T, logits_dev, di, (cudaStream_t)stream);
}

extern "C" const char* moe_stage_names(int path) {
  if (path == MOE_PATH_DECODE_FUSED) return "decode_fused";
  if (path == MOE_PATH_DECODE_MMA)
    return "act_split_x,router_shared_gateup,topk,sort,routed_gateup,act_split_h,routed_down,combine";
  if (path == MOE_PATH_PREFILL_TC)
    return "router_shared_gateup,topk,sort,quant_x,routed_gateup,quant_h,routed_down,combine";
  return nullptr;
}

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_BAD_DESCRIPTOR: return "packed-weight descriptor does not match";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_BUFFER_TOO_SMALL: return "buffer too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_NO_DEVICE: return "current device is not an sm_103 GPU";
    default: return "unknown status";
  }
}

extern "C" const char* moe_version(void) { return "moe_mxfp4 1.2 sm_103a"; }

namespace moe {
namespace {
// One thread waits, with the same bounded helper the decode kernel uses, for
// *flag == want; on expiry MOE_DEV_TIMEOUT is set and the kernel returns.
__global__ void wait_selftest_kernel(const uint32_t* flag, uint32_t want, long long budget, int* status) {
  if (threadIdx.x == 0 && blockIdx.x == 0) wait_eq_u32(flag, want, status, budget);
}
}  // namespace
}  // namespace moe

extern "C" int moe_selftest_bounded_wait(const uint32_t* flag_dev, uint32_t want, long long budget_cycles,
                                         int* dev_status, moe_stream_t stream) {
  MOE_CHECK_ARG(flag_dev && dev_status, MOE_ERR_INVALID_ARG);
  MOE_CHECK_ARG(budget_cycles > 0 && budget_cycles <= kSpinBudget, MOE_ERR_INVALID_ARG);
  DeviceInfo di;
  int st = current_device(&di);
  if (st != MOE_OK) return st;
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(flag_dev, want, budget_cycles, dev_status);
  return launch_status();
}
