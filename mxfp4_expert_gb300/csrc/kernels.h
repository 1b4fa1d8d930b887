// Launchers shared between the translation units of libmoe_mxfp4.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "host_util.h"

namespace moe {

// route.cu
int launch_topk(const float* logits, int T, int E, int k, const float* bias, int bias_stride,
                int32_t* idx, float* w, cudaStream_t s);
size_t sort_workspace_bytes(int T, int E);
// top-k and the sort in one launch (one block), for T <= 32 tokens
bool route_fused_ok(int T, int E, int k);
int launch_route_fused(const float* logits, int T, int E, int k, const float* bias, int bias_stride,
                       int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                       int32_t* active, int32_t* n_active, int* status, cudaStream_t s);
int launch_sort(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                int32_t* perm, int32_t* inv, int32_t* active, int32_t* n_active, void* ws,
                int* status, cudaStream_t s);

// experts.cu
// Activation rows [rows][K] (bf16 if src_bf16, else fp32) -> B-operand terms
// act_b [rows][K/32][128] and block exponents act_e [rows][K/32].
int launch_act_split(const void* src, bool src_bf16, int rows, int K, uint8_t* act_b,
                     int16_t* act_e, const DeviceInfo& di, cudaStream_t s);

// quant.cu: activation rows (bf16 or fp32) [rows][K] -> E4M3 terms
// q [rows][nterms][K] and E8M0 scales [rows][K/32] (see quant.cu).
enum QuantMode { kQuantMxfp8 = 0, kQuantSplit2 = 1 };
int launch_act_quant(const void* src, bool src_bf16, int rows, int K, int mode, uint8_t* q, uint8_t* scales,
                     cudaStream_t s);

// lmhead.cu: FP8 LM head (E4M3 rows with an fp32 scale per row)
int launch_lm_pack(const void* w_bf16, int V, int d, uint8_t* codes, float* scales, cudaStream_t s);
int launch_lm_gemv(const uint8_t* codes, const float* scales, int V, int d, const void* x_bf16, int T,
                   float* logits, const DeviceInfo& di, cudaStream_t s);

enum RoutedMode { kModeGateUp = 0, kModeDown = 1 };

struct RoutedArgs {
  const uint8_t* w;         // packed matrices, expert e at w + e * mat_bytes
  uint64_t mat_bytes;
  int n_tiles;              // N / 16
  int KB;                   // K / 32
  const int32_t* active;    // [E] active experts (ascending)
  const int32_t* n_active;  // [1]
  const int32_t* offsets;   // [E+1] sorted-slot offsets per expert
  const int32_t* perm;      // sorted slot -> p = t*k + j
  int k;
  const uint8_t* act_b;     // B-operand rows (e4m3 terms)
  const int16_t* act_e;
  const uint8_t* act_q;     // tensor-core path: activation rows as E4M3 terms [rows][act_terms][K]
                            // (gate/up: x rows by token; down: h rows by sorted slot)
  const uint8_t* act_s;     // tensor-core path: their E8M0 scales [rows][K/32]
  int act_terms;            // tensor-core path: 1 (MXFP8) or 2 (two-term split)
  int act_by_token;         // 1: activation row = perm[slot] / k; 0: = slot
  int max_items;            // upper bound on n_active * n_tiles (grid sizing)
  float* out;               // gate/up: h [slots][N/2]; down: part [slots][N]
  int out_ld;
  int out_by_pair;          // tensor-core down pass: part row = perm[slot] (t k + j), not the slot
  int narrow;               // tensor-core path: items of up to 64 B rows (few tokens per expert), else 128
  int* status;
};
int launch_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s);

// umma.cu: the same routed GEMMs on tcgen05 block-scaled MMAs (E4M3-coded
// MXFP4 weights x E4M3 activation terms, E8M0 scales in tensor memory, fp32
// accumulator in tensor memory), for large T.
int launch_umma_routed(RoutedMode mode, const RoutedArgs& a, const DeviceInfo& di, cudaStream_t s);

// dense.cu
struct FrontArgs {
  const __nv_bfloat16* x;   // [T][d]
  int T, d, E, I;
  const __nv_bfloat16* router_w;   // [E][d]
  const __nv_bfloat16* sh_gate;    // [I][d] or null
  const __nv_bfloat16* sh_up;      // [I][d]
  float* logits;                   // [T][E]
  float* h_sh;                     // [T][I]
  __nv_bfloat16* h_hi = nullptr;   // if set: h_sh goes out as two bf16 terms [T][I] here
  __nv_bfloat16* h_lo = nullptr;   //   (hi = bf16(h), lo = bf16(h - hi)) instead of fp32
};
int launch_front(const FrontArgs& a, const DeviceInfo& di, cudaStream_t s);

struct CombineArgs {
  int T, d, I, k;
  const __nv_bfloat16* sh_down;    // [d][I] or null
  const float* h_sh;               // [T][I]
  const float* w;                  // [T][k]
  const int32_t* inv;              // [T*k] p -> sorted slot
  const float* part;               // [slots][d]
  __nv_bfloat16* y;                // [T][d]
};
int launch_combine(const CombineArgs& a, const DeviceInfo& di, cudaStream_t s);

// tcdense.cu: the same two dense stages on tcgen05 bf16 MMAs with TMA-tiled
// operands (shared expert and k <= 8 required). h_sh passes between them as
// two bf16 terms h_hi, h_lo [T][I] (hi = bf16(h), lo = bf16(h - hi)); a.h_sh
// is unused by both (launch_front writes the same terms when a.h_hi is set).
// The combine reads part in (token, choice) order: part row t k + j (a.inv
// unused).
bool tc_dense_supported(int T, int d, int I, int k, bool has_shared, const DeviceInfo& di);
int launch_tc_front(const FrontArgs& a, __nv_bfloat16* h_hi, __nv_bfloat16* h_lo, int* status,
                    const DeviceInfo& di, cudaStream_t s);
int launch_tc_combine(const CombineArgs& a, const __nv_bfloat16* h_hi, const __nv_bfloat16* h_lo, int* status,
                      const DeviceInfo& di, cudaStream_t s);

}  // namespace moe
