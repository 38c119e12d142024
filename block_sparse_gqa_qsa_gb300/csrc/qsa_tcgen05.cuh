// qsa_tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores of
// sm_103a: tensor-memory (TMEM) allocation, tcgen05.mma of kind::f16 with
// shared-memory matrix descriptors, completion through an mbarrier, and
// TMEM -> register loads.
//
// Shared-memory operand layouts used by the kernels (16-bit elements):
//   SW128 K-major   rows of 128 bytes (64 elements of the contraction dim),
//                   16-byte chunk c of row r stored at chunk c ^ (r % 8); 8-row
//                   groups of 1024 bytes (SBO = 1024).  A 128-element row is two
//                   such tiles ("halves") one after the other.  The tile base is
//                   1024-byte aligned; a K step of 16 elements inside a half
//                   advances the start address by 32 bytes.
//   SW128 MN-major  the same bytes read with the contiguous 64 elements as the
//                   M (or N) dimension: LBO = stride between the 64-element
//                   halves, SBO = 1024 (8 rows of the contraction dim).
//   plain MN-major  8 x 8 core matrices of 128 contiguous bytes (8 rows of the
//                   contraction dim, 8 contiguous M/N elements each); with N = 8
//                   the next core matrix along the contraction dim is 128 bytes on.
// These layouts were checked numerically on a GB300 against a CPU product.
#pragma once

#include <stdint.h>

#include "qsa_device.cuh"

namespace qsa {

enum : uint32_t { kSmemSwizzleNone = 0, kSmemSwizzle128B = 2 };

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), the fixed version field of sm_100-family parts,
// and the swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle & 7u) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both fp16
// (or both bf16), each K-major (0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t mma_idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A * B, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// The mbarrier completes a phase once every tcgen05.mma this thread issued before has finished.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// TMEM allocation by one whole warp: `ncols` (a power of two >= 32) columns;
// the address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane (warp w of a
// warpgroup reads lanes 32w .. 32w+31; taddr carries the lane in bits 16..31).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace qsa
