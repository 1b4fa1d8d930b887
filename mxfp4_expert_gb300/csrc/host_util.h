// Host-side helpers shared by the C-ABI entry points: argument checks, CUDA
// error mapping, per-device properties.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

#define MOE_CHECK_ARG(cond, code) \
  do {                            \
    if (!(cond)) return (code);   \
  } while (0)

#define MOE_CUDA_TRY(expr)                    \
  do {                                        \
    cudaError_t _e = (expr);                  \
    if (_e != cudaSuccess) {                  \
      (void)cudaGetLastError();               \
      return MOE_ERR_CUDA;                    \
    }                                         \
  } while (0)

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
};

// Properties of the current device (queried once per device, then cached).
// Returns MOE_OK, MOE_ERR_CUDA or MOE_ERR_NO_DEVICE (not compute capability 10.3).
int current_device(DeviceInfo* out);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch status of the last kernel (configuration errors only; asynchronous
// faults surface at the caller's next synchronisation).
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
