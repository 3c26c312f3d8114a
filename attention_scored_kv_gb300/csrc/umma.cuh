// tcgen05 (5th-generation tensor core) helpers: TMEM allocation, shared-memory matrix
// descriptors, the kind::f16 MMA, commits to mbarriers and TMEM loads.
//
// Operand layout used here: K-major tiles with the 128-byte swizzle.  A tile of R rows
// by 128 16-bit elements is stored as two 64-element halves ("k-blocks"), each
// [R rows][128 bytes].  Within every group of 8 rows (1024 bytes) the 16-byte chunk c
// of row r sits at chunk position c ^ (r % 8).  Tiles start on 1024-byte boundaries.
// The descriptor of such a tile has the stride between 8-row groups (1024 bytes) in
// its stride field, and k-step ks (16 elements = 32 bytes) starts at
// k-block (ks / 4), byte offset 32 * (ks % 4) of the row.
#pragma once
#include <cstdint>

#include "kvs_internal.cuh"

namespace kvs {
namespace umma {

// Byte offset of element (row r, element e) of a K-major 128-byte-swizzled tile of
// `rows` rows with 16-bit elements.
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t rows, uint32_t r, uint32_t e) {
  return (e / 64) * rows * 128u + r * 128u + ((((e % 64) * 2u / 16u) ^ (r % 8u)) * 16u) + ((e % 64) * 2u) % 16u;
}

// Shared-memory matrix descriptor: start address, leading byte offset 16 (unused by
// swizzled K-major layouts), stride byte offset 1024, descriptor version 1, 128-byte
// swizzle.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: f32 accumulator, A and B both bf16 (bf16 = true)
// or both f16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[a_desc] * B[b_desc]^T; accumulate = false overwrites D.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// The mbarrier at `bar` receives one arrival when every MMA issued so far by this
// thread has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
               : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (lane = 32 * (warp % 4) + lane
// id, given in taddr's upper half), starting at taddr's column.  The load and its wait
// are one statement, so no use of the registers can be scheduled before the wait.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace umma
}  // namespace kvs
