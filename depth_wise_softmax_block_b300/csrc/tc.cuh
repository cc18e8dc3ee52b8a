// Fifth-generation tensor-core (tcgen05) helpers for sm_103a, as inline PTX: tensor-memory
// allocation, shared-memory matrix descriptors, the bf16 x bf16 -> fp32 MMA, its completion
// signal and tensor-memory loads.
#pragma once

#include <stdint.h>

#include "tma.cuh"

namespace attnres {

// Allocate `ncols` (a power of two >= 32) tensor-memory columns; the whole warp executes it and
// the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Ordering of tensor-core operations across a thread barrier.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Makes this thread's ordinary shared-memory writes visible to the async proxy (the tensor
// core reads its operands through it).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Descriptor of a K-major operand tile in shared memory laid out as the 128-byte-swizzled
// tensor copy writes it: rows of 128 bytes (64 bf16 along K), groups of 8 rows 1024 bytes
// apart, tile base aligned to 1024 bytes.  `saddr` may be advanced by 32-byte steps to select
// the 16-element K slice of one MMA.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);  // start address, bits 0-13
  d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// Descriptor of an MN-major operand tile (the M or N index runs along the 128-byte rows) laid
// out by the 128-byte-swizzled tensor copy: each row holds 64 bf16 of the MN index for one K
// index, groups of 8 K rows 1024 bytes apart; `mn_stride` bytes separate the 64-element blocks of
// the MN index (the second copy of a 128-wide operand).  Base aligned to 1024 bytes; advance
// `saddr` by 2048 bytes per K = 16 step.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3fffu) << 16;  // between 64-element MN blocks
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                    // between 8-row K groups
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Descriptor of a K-major operand without swizzle, as 8 x 8 core matrices (8 rows of 16 bytes,
// 128 bytes each): the core matrix of K chunk kc (8 elements) and row group g (8 rows) starts at
// kc * k_stride + g * row_stride bytes.  Advance `saddr` by 2 * k_stride per K = 16 step.
__device__ __forceinline__ uint64_t desc_kmajor_plain(uint32_t saddr, uint32_t k_stride,
                                                      uint32_t row_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>((k_stride >> 4) & 0x3fffu) << 16;
  d |= static_cast<uint64_t>((row_stride >> 4) & 0x3fffu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // no swizzle (layout 0)
  return d;
}

// Instruction descriptor: dense MMA, A and B bf16, K-major, D fp32, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with A MN-major (bit 15) and B K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn(int M, int N) {
  return idesc_bf16_f32(M, N) | (1u << 15);
}

// D[M x N] (+)= A[M x K=16] . B[N x K=16]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane (32x32b shape: thread i of
// the warp reads lane base+i).  Complete with tmem_ld_wait() before using the values.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 8 consecutive fp32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
// A 16-lane x 8-column block (16x256b shape): thread i gets (lane base + i / 4, columns
// 2 (i % 4) and 2 (i % 4) + 1) in r[0], r[1] and the same columns of lane base + 8 + i / 4 in
// r[2], r[3] - the accumulator-fragment layout that stmatrix takes.  The lane base is 0 or 16
// within the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace attnres
