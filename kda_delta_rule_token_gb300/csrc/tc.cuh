// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05) and
// tensor memory (TMEM), written from the PTX ISA: TMEM allocation, kind::tf32
// and kind::f16 (bf16) MMAs with operands in shared memory or TMEM, commits
// to an mbarrier, and 32-lane x 32-bit TMEM loads/stores.
//
// Shared-memory operands use the K-major, 128-byte-swizzled layout: rows of
// 128 bytes (32 fp32/tf32 or 64 bf16 elements of K), 8-row atoms of 1024 bytes, the
// 16-byte chunk index XOR-ed with (row % 8); K beyond 32 elements continues
// in further blocks of rows x 128 bytes.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace kda {
namespace tc {

// fp32 -> tf32 (bits of a 32-bit word, low 13 bits zero), rounded to
// nearest with ties to even.  Measured on the prefill: 3.4 % faster than the
// ties-away-from-zero form (cvt.rna) with the same accuracy.
__device__ __forceinline__ uint32_t f2tf32(float x) {
    uint32_t r;
    asm("cvt.rn.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// Byte offset of element (row, k) in a K-major SW128 operand of `rows` rows.
__device__ __forceinline__ uint32_t sw128(int row, int k, int rows) {
    const int kb = k >> 5, kk = k & 31;
    return (uint32_t)(kb * rows * 128 + row * 128 + ((((kk >> 2) ^ (row & 7))) << 4) + ((kk & 3) << 2));
}

// Shared-memory matrix descriptor: K-major, SWIZZLE_128B, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The descriptor of the operand `off` bytes (a multiple of 16) past the one
// `d` describes.  The start-address field holds bits 4..17 of the
// shared-memory address and every operand lies below 256 KiB, so the sum
// never carries out of the field.  Issue loops that add constant offsets to
// one base descriptor and are fully unrolled issue an MMA every 45-64 cycles
// (the tensor pipe's own rate for tf32 at N = 64..128); the same loop kept
// rolled, or rebuilding the descriptor from the address each time, issues
// one every 87-127 cycles, and a single issuing thread then sets the pace.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }

// Instruction descriptor: kind::tf32, D = f32, A = B = tf32, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor: kind::f16 with bf16 A and B, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Whole-warp TMEM allocation; the base address is written to *dst (shared).
__device__ __forceinline__ void alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(ptx::smem_u32(dst)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 operands (kind::f16, K = 16 per instruction)
__device__ __forceinline__ void mma_ss_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n"
        ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Arrive once on mbarrier m when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void commit(uint64_t* m) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(ptx::smem_u32(m)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#define KDA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
#define KDA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), \
                  "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : KDA_R8(0), KDA_R8(8), KDA_R8(16), KDA_R8(24)
        : "r"(taddr));
}

__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), KDA_W8(0), KDA_W8(8), KDA_W8(16), KDA_W8(24)
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : KDA_R8(0), KDA_R8(8)
                 : "r"(taddr));
}

__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), KDA_W8(0), KDA_W8(8)
                 : "memory");
}

// 8 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : KDA_R8(0)
                 : "r"(taddr));
}

__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), KDA_W8(0)
                 : "memory");
}

#undef KDA_R8
#undef KDA_W8

// TMEM address of (lane base of this warp's quadrant, column col).
__device__ __forceinline__ uint32_t taddr(uint32_t base, int warp, int col) {
    return base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col;
}

}  // namespace tc
}  // namespace kda
