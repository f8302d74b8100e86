// mk_tc.cuh -- fifth-generation tensor-core helpers (tcgen05, sm_100 family):
// tensor-memory allocation, shared-memory matrix descriptors, the bf16 MMA,
// its commit to an mbarrier and the accumulator read-back.  Inline PTX only.
//
// Operand layout used throughout: K-major tiles in the 128-byte swizzle.  A
// tile of R rows x 64 bf16 (one K chunk) is R/8 atoms of 8 rows x 128 bytes,
// atom after atom (1024 bytes apart); inside an atom, 16-byte chunk j of row r
// sits at chunk slot j ^ r.  A tile starts on a 1024-byte boundary, so the
// swizzle the tensor core applies to address bits [4:6] (xor bits [7:9])
// matches the stored one.  The K = 16 slices of a chunk are addressed by
// moving the descriptor's start 32 bytes per slice.
#pragma once
#include <stdint.h>

namespace mk {

#ifndef MK_DEV
#define MK_DEV __device__ __forceinline__
#endif

// Byte offset of element (r, k), k < 64, inside a swizzled K-major tile.
MK_DEV uint32_t sw128_off(uint32_t r, uint32_t k) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((((k >> 3) ^ r) & 7u) << 4) + (k & 7u) * 2u;
}

// Shared-memory matrix descriptor of a swizzled K-major tile starting at
// shared address `addr` (1024-byte aligned, plus 32 bytes per K = 16 slice):
// start address >> 4 in bits [0, 14), leading byte offset (unused by the
// swizzled K-major form; 16 bytes) in [16, 30), stride byte offset 1024 (the
// next 8-row atom) in [32, 46), descriptor version 1 in [46, 48), base
// offset 0, swizzle mode 2 (128-byte) in [61, 64).
MK_DEV uint64_t sw128_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
         ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B, f32 accumulator,
// both operands K-major: D format (1 = f32) in [4, 6), A format (1 = bf16)
// in [7, 10), B format in [10, 13), N >> 3 in [17, 23), M >> 4 in [24, 29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Tensor-memory allocation of `ncols` columns (a power of two >= 32) by one
// whole warp; the base address is written to shared memory at `slot`.
MK_DEV void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MK_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[adesc] * B[bdesc]^T, M x N x 16, issued by the calling thread.
MK_DEV void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive (once) on the mbarrier when every MMA this thread issued so far has
// completed: their reads of shared memory and writes of tensor memory.
MK_DEV void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

MK_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

MK_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Sixteen consecutive f32 columns of this thread's tensor-memory lane: warp w
// of a warpgroup reads lanes 32 (w % 4) .. + 31, so taddr carries that lane
// base in its upper half.  The load and its wait sit in one asm statement, so
// no use of the registers can be scheduled before the data has arrived.
MK_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

}  // namespace mk
