// Inline-PTX wrappers for the fifth-generation tensor cores (tcgen05) of
// sm_103a: tensor-memory (TMEM) allocation, shared-memory matrix descriptors,
// the single-thread MMA with a TMEM accumulator, its commit to an mbarrier,
// and the warp-wide TMEM loads and stores of the epilogue.
//
// Encodings follow the PTX ISA's tcgen05 chapter:
//  * shared-memory descriptor (64 bit): start address >> 4 in bits 0-13,
//    leading-dimension byte offset >> 4 in bits 16-29, stride-dimension byte
//    offset >> 4 in bits 32-45, descriptor version 1 in bits 46-47, base
//    offset 0 (every swizzle atom starts on its own period), swizzle mode in
//    bits 61-63 (2 = 128-byte, 4 = 64-byte);
//  * instruction descriptor of kind::f16 (32 bit): D format in bits 4-5
//    (1 = f32), A and B formats in bits 7-9 and 10-12 (1 = bf16), A and B
//    major-ness in bits 15 and 16 (0 = K-major, 1 = M/N-major), N >> 3 in
//    bits 17-22 and M >> 4 in bits 24-28.
// Canonical swizzled layouts (16-bit elements):
//  * K-major, 128-byte swizzle: rows of 64 elements (128 B) along K, 8-row
//    groups along M/N at the stride-dimension offset; a 16-element K step
//    inside the row is a 32-byte advance of the start address;
//  * M/N-major: rows of one K index, 64 (128-byte swizzle) or 32 (64-byte
//    swizzle) M/N elements wide; 8-row K groups at the stride-dimension
//    offset, further 64- or 32-element M/N atoms at the leading-dimension
//    offset.
// The swizzle is a function of the shared-memory address (16-byte chunk bits
// 4-6, or 4-5, XOR address bits 7-9, or 7-8), so buffers start on 1 KiB.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace pkv {

enum : uint32_t { kSwizzle128 = 2u, kSwizzle64 = 4u };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle) << 61);
}

// bf16 x bf16 -> f32, M x N tile; a_mn / b_mn: operand stored M/N-major
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Allocation by one whole warp; the TMEM address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
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

// Order tcgen05 operations against thread synchronisation (barriers, mbarriers).
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) = A (smem) . B (smem) [+ D when acc]; issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// D (TMEM) = A (TMEM) . B (smem) [+ D when acc]; A is K-major in TMEM: row m
// in lane m, 16-bit elements two to a 32-bit column (the lower K index in the
// low half), so a K = 16 step spans 8 columns.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp-wide TMEM load: lane i of the warp reads TMEM lane (taddr.lane + i),
// columns taddr.col .. +N-1, one 32-bit value per column.  The wait takes the
// registers as operands so that no use of them is scheduled above it.
#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_W8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                  "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define PKV_S8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                  "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
               :
               : "memory");
}

// The same load without the wait, and the wait alone (taking 32 of the
// loaded registers as operands): several loads can then share one wait.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : PKV_R8(0), PKV_R8(8)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PKV_W8(0), PKV_W8(8) : : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : PKV_R8(0)
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PKV_W8(0) : : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      PKV_S8(0), PKV_S8(8), PKV_S8(16), PKV_S8(24)
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// The store without its wait, and the wait for every store issued before.
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      PKV_S8(0), PKV_S8(8), PKV_S8(16), PKV_S8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      PKV_S8(0), PKV_S8(8)
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               PKV_S8(0)
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef PKV_R8
#undef PKV_W8
#undef PKV_S8

}  // namespace pkv
