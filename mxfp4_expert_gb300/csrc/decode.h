// Single-launch decode path (see decode.cu).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "host_util.h"

namespace moe {

constexpr int kDecodeMaxT = 4;        // tokens per call on this path
constexpr int kDecodeMaxTiles = 4;    // 16-row output tiles per CTA
constexpr int kDecodeStateWords = 16; // synchronisation words at the head of the workspace

// Synchronisation words at the start of the workspace (zero before the
// first call; the last CTA of every call puts them back to zero).
struct DecodeState {
  uint32_t routed;   // CTAs whose router logits and shared gate/up features are written
  uint32_t done;     // CTAs finished (compared modulo the grid size; never reset)
  uint32_t gudone;   // CTAs whose routed gate/up features are written
  uint32_t pad[13];
};
static_assert(sizeof(DecodeState) == kDecodeStateWords * 4, "state header size");

struct DecodeArgs {
  int T, d, I, E, k, has_shared;
  const __nv_bfloat16* x;
  const __nv_bfloat16* router_w;
  const __nv_bfloat16* sh_gate;
  const __nv_bfloat16* sh_up;
  const __nv_bfloat16* sh_down;
  const uint8_t* gate_up;
  const uint8_t* down;
  uint64_t gu_mat, dn_mat;
  const float* bias;
  int bias_stride;
  float* logits;        // [T][E]
  int32_t* idx_out;     // [T][k] or null
  float* w_out;         // [T][k] or null
  __nv_bfloat16* y;     // [T][d]
  DecodeState* state;
  uint8_t* h;           // routed SwiGLU outputs as e4m3 terms + group factors, exchanged between CTAs
  float* h_sh;          // [T][I]
  int* status;
};

// Bytes of the cross-call state (the counters above).
size_t decode_state_bytes(int T, int E);
// Row stride (elements) of the per-stage path's h exponent array: I/32 rounded up to 8.
uint32_t decode_he_stride(int I);
// Bytes of the routed-h exchange area the single-launch kernel uses.
size_t decode_h_bytes(int T, int k, int I);
// MOE_OK if the shape/T can take this path on this device; *smem_bytes is the
// dynamic shared memory of the launch.
int decode_plan(const DecodeArgs& a, const DeviceInfo& di, uint32_t* smem_bytes);
int launch_decode(const DecodeArgs& a, const DeviceInfo& di, cudaStream_t s);

}  // namespace moe
