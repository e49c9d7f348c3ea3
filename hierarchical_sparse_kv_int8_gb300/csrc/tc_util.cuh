// Fifth-generation tensor core (tcgen05) helpers in inline PTX: tensor memory
// allocation, the bf16 MMA of kind::f16 with operands in shared memory and the
// accumulator in tensor memory, its completion signal, tensor-memory loads and
// stores, and the descriptors the MMA takes.
//
// Shared-memory operand layout used throughout (no swizzle): a matrix is cut
// into core matrices of 8 rows x 16 bytes (8 bf16), each stored as 128
// contiguous bytes, row r of the core at byte 16 r.  For a K-major operand
// (the reduction index K contiguous within a row) the cores that follow along
// K are `lbo` bytes apart and the groups of 8 rows `sbo` bytes apart.  For an
// MN-major operand (the output index contiguous) a core is 8 consecutive K
// indices x 8 consecutive N elements, the cores that follow along N are
// `sbo` bytes apart and the groups of 8 K indices `lbo` bytes apart.
#pragma once
#include <stdint.h>

#include "ptx_util.cuh"

namespace dhs {

// Shared-memory matrix descriptor (64 bits): start address, leading and
// stride byte offsets (each >> 4), the descriptor version of this tensor-core
// generation (bit 46), no swizzle (layout type 0), base offset 0.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// The same for an operand in the 128-byte-swizzled layout (layout type 2):
// rows of 128 bytes, 16-byte chunk c of row r stored at chunk position
// c ^ (r mod 8) within its 1024-byte group of 8 rows (the pattern follows
// address bits 4-6 and 7-9, so the groups start on 1024-byte boundaries).
// K-major: `sbo` = bytes between groups of 8 rows, `lbo` unused (16); the K
// steps of one MMA advance the start address within the 128-byte row.
// MN-major: `lbo` = bytes between 64-element blocks along N, `sbo` = bytes
// between groups of 8 K indices.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return tc_desc(saddr, lbo, sbo) | ((uint64_t)2 << 61);
}

// Instruction descriptor of a dense kind::f16 MMA with bf16 A and B, fp32 D:
// D format (bits 4-5) = f32, A and B formats (bits 7-9, 10-12) = bf16, A and B
// major-ness (bits 15, 16; 1 = MN-major), N >> 3 (bits 17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Tensor memory: `ncols` columns (a power of two >= 32) of the SM's 128
// lanes, allocated by one whole warp; the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier receives one arrival once every MMA this thread issued before
// has completed.
__device__ __forceinline__ void tc_commit(void *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 32 consecutive 32-bit columns of the warp's 32 lanes (lane l of the warp
// reads tensor-memory lane base_lane + l): taddr = base + (lane << 16) + col.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// 2^x by the PTX ISA's approximate base-2 exponential instruction
// (ex2.approx.ftz; -inf gives +0), for softmax weights that are rounded to
// bf16 anyway.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Plain arrival on an mbarrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(void *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

}  // namespace dhs
