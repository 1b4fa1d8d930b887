// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05): tensor
// memory (TMEM) allocation, shared-memory matrix descriptors, the instruction
// descriptors of a block-scaled (E2M1 or E4M3) x E4M3 -> fp32 MMA and of a
// bf16 x bf16 -> fp32 MMA, the MMAs themselves, the copy of scale factors
// into TMEM, the completion signal, TMEM -> register loads, and the bounded
// mbarrier wait of the warp-specialised kernels.
#pragma once

#include "common.cuh"

namespace moe {

// ---- tensor memory --------------------------------------------------------
// Whole warp: allocate ncols (power of two >= 32) TMEM columns; the TMEM
// address (lane 0, first column) is written to *slot in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
// Whole warp: free the columns again (before the CTA exits).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes -> visible to the tensor cores.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- descriptors ------------------------------------------------------------
// Shared-memory matrix descriptor, K-major, no swizzle. The operand is stored
// as 8-row x 16-byte core matrices (128 contiguous bytes); lbo = byte offset
// between core matrices adjacent along K, sbo = between core matrices adjacent
// along M (or N).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version of this architecture
  return d;
}
// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row x 128-byte
// atoms stacked along M (or N) 1024 bytes apart, the 16-byte chunk j of row r
// of an atom stored at chunk j ^ (r % 8). The atoms must be 1024-byte
// aligned; a K step inside the atom advances saddr by its bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                   // leading byte offset: unused for this layout
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                   // descriptor version of this architecture
  d |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle
  return d;
}
// Shared-memory descriptor of a 512-byte scale block for tcgen05.cp: 32 lines
// of 16 bytes, no swizzle (8-line core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t umma_desc_sf(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Operand formats of kind::mxf8f6f4.
constexpr int kFmtE4M3 = 0, kFmtE2M1 = 5;
// Instruction descriptor of a block-scaled MMA (kind::mxf8f6f4): fp32
// accumulator, A of format a_fmt (bits 7-9) and E4M3 B (bits 10-12 zero), both
// K-major, E8M0 scales (bit 23), M x N, and which byte of the 32-bit scale
// words the A and B scales of this K-block are (sf_a at bits 29-30, sf_b at
// bits 4-5). An E2M1 operand sits in shared memory as 16-byte chunks whose low
// 8 bytes hold 16 codes (code 2j in the low nibble of byte j); the high 8
// bytes are not read.
__host__ __device__ constexpr uint32_t umma_idesc_mx(int M, int N, int a_fmt, int sf_a, int sf_b) {
  return ((uint32_t)(sf_b & 3) << 4) | ((uint32_t)(a_fmt & 7) << 7) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | ((uint32_t)(sf_a & 3) << 29);
}

// Instruction descriptor of a dense MMA of kind::f16 with bf16 A and B (bits
// 7-9 and 10-12 = 1), both K-major, fp32 accumulator (bits 4-5 = 1), M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- MMA ----------------------------------------------------------------------
// One thread: D[tmem] (+)= A * B^T for one K = 16 step of bf16 operands
// (kind::f16, fp32 accumulator, cta_group::1).
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// One thread: D[tmem] (+)= (A x scale_A) * (B x scale_B)^T for one K = 32 step
// (kind::mxf8f6f4, block_scale, one scale per 32 elements, cta_group::1).
__device__ __forceinline__ void umma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t tmem_sfa, uint32_t tmem_sfb, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem_sfa), "r"(tmem_sfb), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// One thread: copy a 512-byte scale block (32 lines x 16 bytes) from shared
// memory to 4 tensor-memory columns, the same in each of the 4 lane quarters.
__device__ __forceinline__ void tmem_cp_sf(uint32_t tmem_col, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem_col), "l"(sdesc) : "memory");
}
// One thread: arrive on *bar once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// ---- TMEM -> registers ----------------------------------------------------------
// Whole warp: thread t gets TMEM lane (taddr lane + t), 8 consecutive columns.
// The warp may only address its own 32-lane quarter (warp id % 4).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Whole warp: 4 consecutive columns of TMEM lane (taddr lane + t) to thread t.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
      : "r"(taddr)
      : "memory");
}
// Whole warp: 16 consecutive columns of TMEM lane (taddr lane + t) to thread t.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
// Whole warp: two such loads (columns at ta and at tb) under one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
        "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}

// ---- bounded waits of a warp-specialised CTA ------------------------------------
// mbarrier wait that gives up after kSpinBudget cycles (setting MOE_DEV_TIMEOUT
// and *abort) or as soon as another role of the CTA has set *abort (seen
// within one suspend period).
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

}  // namespace moe
