// Thin wrappers over the sm_100-family tensor-core instructions (tcgen05.*)
// used by the tensor-core kernels: shared-memory matrix descriptors, the
// instruction descriptor of a BF16 x BF16 -> FP32 MMA, tensor-memory (TMEM)
// allocation, MMA issue / commit and TMEM loads.  Written from the PTX ISA's
// descriptions of these instructions; internal to the library.
#pragma once

#include "common.cuh"

namespace lora {
namespace tc {

// Byte offset of element (row r, column k) of a bf16 tile stored K-major with
// 64-element (128-byte) rows in the 128-byte swizzle layout: rows grouped by
// 8 into 1024-byte atoms, and within a row the 16-byte chunk c stored at
// position c ^ (r mod 8).  The tile base must be 1024-byte aligned.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) +
                    (k & 7) * 2);
}

// Shared-memory matrix descriptor of such a tile: start address (>> 4) in
// bits 0-13, leading-dimension byte offset (unused for a swizzled K-major
// operand whose K-step stays inside one 128-byte row) in bits 16-29, stride
// byte offset between 8-row atoms (1024 B >> 4) in bits 32-45, descriptor
// version 1 in bits 46-47, swizzle mode 2 (128-byte) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_byte_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with BF16 A and B, FP32
// accumulator, both operands K-major: D format in bits 4-5 (1 = F32), A and B
// formats in bits 7-9 and 10-12 (1 = BF16), N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Warp-wide: allocate `ncols` (a power of two >= 32) TMEM columns; the TMEM
// address is written to *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide: release TMEM allocated by this CTA.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one M x N x 16 step, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 TMEM lanes x 16 consecutive fp32 columns: lane t of the warp receives
// row (lane base + t), columns [col, col + 16) of `taddr`.  The warp may only
// address the 32-lane quarter (warp id mod 4) of TMEM.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace tc
}  // namespace lora
