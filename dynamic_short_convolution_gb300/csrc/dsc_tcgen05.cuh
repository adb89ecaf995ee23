// dsc_tcgen05.cuh -- 5th-generation tensor core (tcgen05) building blocks for
// sm_100-family GPUs, as inline PTX: tensor-memory (TMEM) allocation, the
// shared-memory matrix descriptor, the instruction descriptor of
// kind::f16 (bf16 inputs, fp32 accumulation), MMA issue and commit, and
// TMEM -> register loads.
#pragma once

#include <stdint.h>

#include "dsc_device.cuh"

namespace dsc {

// ------------------------------------------------------------------ TMEM allocation (one full warp)

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations across thread synchronisation.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor of a K-major operand tile in the canonical
// 128-byte-swizzled layout: rows of 128 bytes (64 bf16 of K), 8-row groups
// 1024 bytes apart, the tile 1024-byte aligned.  A K step inside the 128-byte
// row advances the start address by 32 bytes (16 bf16).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address, 16-byte units
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused when swizzled)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version of the tcgen05 family
    d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128-byte
    return d;
}

// General shared-memory matrix descriptor: start address, leading and stride
// byte offsets, swizzle mode (0 none, 2 128-byte, 4 64-byte, 6 32-byte).
// K-major swizzled: SBO = distance between 8-row groups (LBO unused).
// MN-major swizzled: rows are K indices holding 64 MN elements (128 B), SBO =
// distance between groups of 8 K rows, LBO = distance between 64-wide MN blocks.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swizzle & 7u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: A and B bf16, D fp32,
// shape M x N; a_mn / b_mn select the MN-major (transposed) operand layouts.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn = false, bool b_mn = false)
{
    return (1u << 4)                                  // D format: fp32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | ((a_mn ? 1u : 0u) << 15)                 // A major-ness: 0 K-major, 1 MN-major
           | ((b_mn ? 1u : 0u) << 16)                 // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ------------------------------------------------------------------ MMA

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA, issued by a single thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA without a compiler memory clobber, for long issue sequences whose
// operands sit in registers: volatile asm statements keep their relative order, so
// the MMA still follows the mbarrier waits and precedes the commit that tracks it.
__device__ __forceinline__ void umma_bf16_nc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]^T: the A operand (M = 128 lanes, K along
// columns, two bf16 per 32-bit column) read from tensor memory.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------------ TMEM -> registers

// 32 TMEM lanes x N consecutive 32-bit columns: thread i of the warp receives
// lane (lane base + i), columns col .. col+N-1.  Completes at tmem_ld_wait().
__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// N = 8 * W columns (W = 1..8) as a sum of x32 / x16 / x8 loads.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N])
{
    static_assert(N % 8 == 0 && N >= 8 && N <= 64, "8..64 columns");
    constexpr int n32 = N / 32, rem = N % 32;
    if constexpr (n32 >= 1) tmem_ld_x32(taddr, r);
    if constexpr (n32 >= 2) tmem_ld_x32(taddr + 32, r + 32);
    if constexpr (rem >= 16) tmem_ld_x16(taddr + n32 * 32, r + n32 * 32);
    if constexpr (rem % 16 == 8) tmem_ld_x8(taddr + n32 * 32 + (rem >= 16 ? 16 : 0), r + n32 * 32 + (rem >= 16 ? 16 : 0));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ registers -> TMEM

// 32 TMEM lanes x 4 consecutive 32-bit columns from each thread's registers
// (thread i -> lane base+i).  Complete at tmem_st_wait().
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_bar(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the OR of `pred` over every participating
// thread, so a group of warps takes one common decision (e.g. to abort).
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace dsc
