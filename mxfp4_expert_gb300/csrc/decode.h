// Single-launch decode path (see decode.cu).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "host_util.h"

namespace moe {

constexpr int kDecodeMaxT = 4;        // tokens per call on this path
constexpr int kDecodeMaxTiles = 4;    // 16-row output tiles per CTA
constexpr int kDecodeMaxStages = 16;
constexpr int kDecodeStateWords = 16; // header words before the per-block counters

// Synchronisation words at the start of the workspace (zero before the
// first call; the last CTA of every call puts them back to zero).
struct DecodeState {
  unsigned long long bar;  // CTAs past their router rows
  uint32_t done;           // CTAs finished (compared modulo the grid size; never reset)
  uint32_t shcnt;          // CTAs whose shared gate/up slice is written
  uint32_t gudone;         // CTAs whose routed gate/up items are written
  uint32_t pad[11];
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
  float* h;             // [T*k][I] routed SwiGLU outputs, exchanged between CTAs
  float* h_sh;          // [T][I]
  int* status;
  int stages;           // set by launch_decode
  uint32_t slot_bytes;  // set by launch_decode
};

size_t decode_state_bytes(int E, int I);
// Row stride (elements) of the h exponent array: I/32 rounded up to 8.
uint32_t decode_he_stride(int I);
// MOE_OK if the shape/T can take this path on this device.
int decode_plan(const DecodeArgs& a, const DeviceInfo& di, int* stages, uint32_t* slot_bytes,
                uint32_t* smem_bytes);
int launch_decode(DecodeArgs a, const DeviceInfo& di, cudaStream_t s);

}  // namespace moe
