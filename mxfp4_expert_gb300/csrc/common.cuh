// Shared device helpers for the sm_103a MXFP4 MoE kernels: inline-PTX wrappers
// (mbarrier, 1-D bulk copies, e4m3 warp MMA, fp8 conversions), bounded waits,
// and the constants of the packed weight format (see include/moe_mxfp4.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

constexpr int kMxBlock = 32;        // elements per E8M0 scale (OCP MX)
constexpr int kTileRows = 16;       // rows per packed tile = MMA M
constexpr int kUnitCodeBytes = 256; // 16 rows x 32 codes x 4 bits
constexpr int kUnitBytes = 272;     // codes + 16 scale bytes
constexpr int kActTerms = 3;        // e4m3 terms per activation value (MMA B columns 0..2; column 3 is zero)
constexpr int kActRowKbBytes = 96;  // 3 terms x 32 e4m3 bytes per (row, K-block)
constexpr int16_t kActZeroExp = -32768;  // marks an all-zero activation block

// Spin budget for any wait on another agent (clock64 cycles, ~1 s at 2 GHz).
constexpr long long kSpinBudget = 2000000000LL;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbarrier.try_wait with an explicit suspend-time limit: the thread sleeps in
// hardware until the phase completes or about `ns` nanoseconds pass, instead
// of spinning (a spinning warp takes issue slots from the working warps)
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and sets MOE_DEV_TIMEOUT) if the phase never
// completes within kSpinBudget cycles. Between polls the thread sleeps for
// sleep_ns, so waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, unsigned sleep_ns = 32) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kSpinBudget) {
      if (status) atomicOr(status, MOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(sleep_ns);
  }
  return true;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (no shared-memory destination).
// src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---- loads ----------------------------------------------------------------
__device__ __forceinline__ uint2 ldg_nc_u2(const void* p) {
  uint2 v;
  asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldg_nc_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---- e4m3 warp MMA: D[16x8] = A[16x32] * B[32x8], fp32 accumulate from 0 ----
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// A 4-byte word of a packed unit row (8 E2M1 codes, code 2j in the low nibble
// of byte j) -> two e4m3x4 registers, each byte worth 2^-6 times the E2M1
// value (sign to bit 7, the 3 exponent/mantissa bits to bits 2..4; the E2M1
// subnormal lands on the E4M3 subnormal). dec_even: codes 0, 2, 4, 6 of the
// word; dec_odd: codes 1, 3, 5, 7.
__device__ __forceinline__ uint32_t dec_even(uint32_t w) {
  return ((w << 4) & 0x80808080u) | ((w << 2) & 0x1C1C1C1Cu);
}
__device__ __forceinline__ uint32_t dec_odd(uint32_t w) { return (w & 0x80808080u) | ((w >> 2) & 0x1C1C1C1Cu); }

// The warp MMA's A fragment from packed unit rows. Lane (g, q) reads bytes
// [4q, 4q+4) of rows g and g+8 (codes 8q..8q+7) and hands the even codes to MMA
// K positions 4q..4q+3 and the odd ones to 16+4q..16+4q+3. K is thereby
// permuted inside each 32-block: MMA position 4q+j <-> code 8q+2j and
// 16+4q+j <-> 8q+2j+1. B operands are stored in the same permuted order
// (bfrag_pos), so every product pairs the right elements.
struct AFrag {
  uint32_t a0, a1, a2, a3;
};
__device__ __forceinline__ AFrag load_afrag(const uint8_t* unit, int g, int q) {
  const uint32_t w0 = *reinterpret_cast<const uint32_t*>(unit + g * 16 + 4 * q);
  const uint32_t w1 = *reinterpret_cast<const uint32_t*>(unit + (g + 8) * 16 + 4 * q);
  return AFrag{dec_even(w0), dec_even(w1), dec_odd(w0), dec_odd(w1)};
}
// Byte position of element e (0..31) of a 32-element B column block, so that
// lane q of a quad reads its fragment (b0, b1) as bytes [8q, 8q+8).
__device__ __forceinline__ int bfrag_pos(int e) { return (e & 24) + ((e & 1) << 2) + ((e >> 1) & 3); }

// fp32 pair -> e4m3x2 (round to nearest even, saturating to +-448); low byte = lo.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// e4m3 byte (low 8 bits of c) -> fp32, exact, through the hardware
// fp8 -> f16x2 conversion (every finite e4m3 value is an f16 value).
__device__ __forceinline__ float e4m3_to_f32_hw(uint32_t c) {
  uint32_t h2;
  asm("{\n .reg .b16 lo;\n cvt.u16.u32 lo, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}\n" : "=r"(h2) : "r"(c));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
// Exact e4m3 -> fp32 (finite codes).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : float(m) * 0.001953125f;
  return (c & 0x80u) ? -mag : mag;
}

// 2^ex as fp32 for an unbiased exponent, including the subnormal/overflow ends.
__device__ __forceinline__ float exp2i(int ex) {
  const int f = ex + 127;
  if (f >= 1 && f <= 254) return __uint_as_float(uint32_t(f) << 23);
  return ldexpf(1.0f, ex);
}
// v * 2^ex, exact whenever the result is a normal fp32 number.
__device__ __forceinline__ float scale2(float v, int ex) {
  if (ex >= -126 && ex <= 127) return v * __uint_as_float(uint32_t(ex + 127) << 23);
  return ldexpf(v, ex);
}

// Combined factor of one (weight row, K-block) x (activation row, K-block):
// weights were decoded as 2^-6 * value, activations stored as value * 2^-e.
// factor = 2^(s - 127) * 2^6 * 2^e.
__device__ __forceinline__ float block_factor(uint32_t s, int e) {
  if (e == kActZeroExp) return 0.0f;
  return exp2i(int(s) - 121 + e);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ---- acquire/release accesses and bounded waits on global flags ----------
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint2 ld_cg_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Bounded spins (acquire). Return false on timeout.
__device__ __forceinline__ bool wait_geq_u64(const unsigned long long* p, unsigned long long target, int* status) {
  if (ld_acquire_u64(p) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_u64(p) < target) {
    if (clock64() - t0 > kSpinBudget) {
      if (status) atomicOr(status, MOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ bool wait_geq_u32(const uint32_t* p, uint32_t target, int* status) {
  if (ld_acquire_u32(p) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_u32(p) < target) {
    if (clock64() - t0 > kSpinBudget) {
      if (status) atomicOr(status, MOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ bool wait_eq_u32(const uint32_t* p, uint32_t want, int* status,
                                            long long budget = kSpinBudget) {
  if (ld_acquire_u32(p) == want) return true;
  const long long t0 = clock64();
  while (ld_acquire_u32(p) != want) {
    if (clock64() - t0 > budget) {
      if (status) atomicOr(status, MOE_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

}  // namespace moe
