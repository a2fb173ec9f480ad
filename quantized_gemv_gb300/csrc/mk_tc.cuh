// Fifth-generation tensor core (tcgen05) wrappers for the batched verify kernel: tensor-memory
// allocation, the UMMA shared-memory and instruction descriptors, MMA issue, commit to an mbarrier,
// tensor-memory loads and the fences between them. sm_103a only.
//
// Operand layout used throughout: K-major, 128-byte swizzle. An "atom" is 8 rows x 128 bytes
// (1024 bytes, 1024-byte aligned); row r of an atom holds its 16-byte chunk c at chunk position
// c ^ (r % 8). Consecutive 8-row groups of an operand are SBO = 1024 bytes apart; one MMA consumes
// a K slice of 16 16-bit elements (32 bytes), selected by advancing the start address by 32 bytes
// inside the atom's 128-byte rows.
#pragma once
#include <cstdint>

#include "mk_device.cuh"

namespace mk {

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major operand whose rows are
// grouped in atoms of 8 (atoms 1024 bytes apart).
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor: start address, leading-dimension offset 16 bytes (unused by
// swizzled K-major operands), stride-dimension offset 1024 bytes (between 8-row groups), descriptor
// version 1, layout 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
         ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A and B both f16 (ab_bf16 = 0) or
// both bf16 (1), both K-major, M = 128, N = n (a multiple of 16).
__host__ __device__ __forceinline__ uint32_t umma_idesc_f16(int ab_bf16, int n) {
  const uint32_t t = ab_bf16 ? 1u : 0u;
  return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K slice of 16; accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every MMA this thread issued so far has completed (its shared
// memory operands may then be overwritten and its accumulator read).
__device__ __forceinline__ void umma_commit(uint64_t* mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(mbar))
               : "memory");
}

// Tensor-memory allocation by one whole warp: ncols columns (a power of two >= 32); the base
// address is written to *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Issue a load of 8 consecutive fp32 columns of this thread's tensor-memory lane into r (raw bits;
// the warp reads the 32 lanes of its quarter, warp % 4, starting at taddr's lane field); the
// registers hold the values only after tmem_wait_ld8() on them.
__device__ __forceinline__ void tmem_ld8_issue(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// Wait for this thread's tensor-memory loads; r (8 registers of one of them) is passed through, so
// the compiler cannot move its uses above the wait. Call it for every load's registers: the first
// call waits for all of them, the others return at once.
__device__ __forceinline__ void tmem_wait_ld8(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes (operands staged by threads) made visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace mk
