// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors, MMA issue, commit and
// tensor-memory loads.  Written from the PTX ISA description of tcgen05.
#pragma once

#include <cstdint>

#include "flint_common.cuh"

namespace flint {
namespace tc05 {

// ---- tensor memory (TMEM) allocation: executed by one full warp
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

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// tensor core's (async proxy) operand reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- shared-memory matrix descriptor, K-major operand with the 128-byte
// swizzle: rows of 128 bytes (64 16-bit elements of K), 8-row atoms of 1024
// bytes; the tile base must be 1024-byte aligned.  Element (r, k) of a tile
// lives at byte r * 128 + (((k / 8) ^ (r % 8)) * 16) + (k % 8) * 2.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for this layout), stride byte offset >> 4 (32-45) = 1024 between
// 8-row groups, version 1 (46-47), layout type 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                 // leading byte offset (ignored): 16 B
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset: 1024 B
  d |= (uint64_t)1u << 46;                 // descriptor version
  d |= (uint64_t)2u << 61;                 // 128-byte swizzle
  return d;
}
// Byte offset of element (r, k) (16-bit elements) inside a 128B-swizzled K-major tile.
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t k) {
  return r * 128u + ((((k >> 3) ^ (r & 7u)) & 7u) << 4) + ((k & 7u) << 1);
}

// ---- instruction descriptor of kind::f16 with fp32 accumulation, both
// operands K-major.  ab_bf16: 0 = f16 operands, 1 = bf16 operands.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int ab_bf16) {
  return (1u << 4)                       // D format: f32
         | ((uint32_t)ab_bf16 << 7)      // A format
         | ((uint32_t)ab_bf16 << 10)     // B format
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (M x N x 16), issued by
// one lane of the threads in `members` (all of which must execute the call
// together, e.g. members = __activemask()): every member executes it and
// elect.sync picks the issuing lane.  With the same members it picks the same
// lane every time, which matters for commit_elect below.  The operands are
// values every member computed.
__device__ __forceinline__ void mma_f16_elect(uint32_t members, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, %5;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(members)
      : "memory");
}

// Arrives (once) on an mbarrier when all MMAs previously issued by the issuing
// thread have completed; the issuing lane is elected as in mma_f16_elect, so
// with the same members the commit tracks the MMAs issued that way.
__device__ __forceinline__ void commit_elect(uint32_t members, uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, %1;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar)),
      "r"(members)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of the warp's 32 lanes (lane i -> thread i).
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc05
}  // namespace flint
