// dsc_lowrank_common.cuh -- device helpers shared by the low-rank kernels:
// an event-driven bounded mbarrier wait, packed bf16 arithmetic for the exact
// hi + lo split of the filter gradient, swizzled tile addressing and TMEM
// stores / loads of any column count.
#pragma once

#include <stdint.h>

#include "dsc_device.cuh"
#include "dsc_tcgen05.cuh"

namespace dsc {

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `hint_ns` passes, so a waiting warp costs no issue
// slots and wakes as soon as the barrier flips.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity: false after limit_ns of
// wall time.  Each poll suspends in hardware for up to 20 us.
__device__ __forceinline__ bool mbar_wait_ev(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

#ifndef DSC_WAIT_MODE
#define DSC_WAIT_MODE 0
#endif

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded spin on a non-blocking test of the phase (the clock is read every 64 polls).
__device__ __forceinline__ bool mbar_spin(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 63) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ bool mbar_try_nohint(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Warp-wide bounded wait for a barrier phase; returns the same outcome in every lane.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
#if DSC_WAIT_MODE == 0
    return __all_sync(0xffffffffu, mbar_wait_ev(bar, parity, limit_ns));
#elif DSC_WAIT_MODE == 1
    return __all_sync(0xffffffffu, mbar_try_nohint(bar, parity, limit_ns));
#elif DSC_WAIT_MODE == 4
    return __all_sync(0xffffffffu, mbar_spin(bar, parity, limit_ns));
#else
    int ok = 1;
#if DSC_WAIT_MODE == 2
    if ((threadIdx.x & 31) == 0) ok = mbar_spin(bar, parity, limit_ns) ? 1 : 0;
#else
    if ((threadIdx.x & 31) == 0) ok = mbar_try_nohint(bar, parity, limit_ns) ? 1 : 0;
#endif
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
#endif
}

// Record a timeout in the device status word and raise the CTA's abort flag.
__device__ __forceinline__ void lr_abort(int *status, volatile int *abort_flag)
{
    record_status(status, kStatusTimeout);
    *abort_flag = 1;
}

// ------------------------------------------------------------------ packed bf16 (two lanes per register)

// Round-to-nearest-even product of two bf16 pairs.
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// a * b + c with a single rounding to bf16 (fused).
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The product of two bf16 values has at most 16 significant bits.  hi is that
// product rounded to bf16, lo = product - hi computed by one fused
// multiply-add; lo has at most 8 significant bits, so it is exact in bf16 and
// hi + lo equals the product exactly (both pairs at once).
__device__ __forceinline__ void exact_product_split(uint32_t a, uint32_t b, uint32_t &hi, uint32_t &lo)
{
    hi = bmul2(a, b);
    lo = bfma2(a, b, hi ^ 0x80008000u);
}

// __byte_perm selector taking bf16 half `h0` (0 low, 1 high) of the first word
// into the low half of the result and half `h1` of the second word into the high half.
__host__ __device__ constexpr uint32_t half_sel(int h0, int h1)
{
    return ((h1 ? 0x76u : 0x54u) << 8) | (h0 ? 0x32u : 0x10u);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ------------------------------------------------------------------ swizzled tiles

// Byte offset of 16-byte chunk `c` of row `row` in a TMA tile whose rows are RB
// bytes (16: no swizzle; 32, 64, 128: the matching swizzle mode, which XORs the
// chunk index with address bits 7 and up).  The tile is 1024-byte aligned.
template <int RB>
__device__ __forceinline__ uint32_t swzt(int row, int c)
{
    static_assert(RB == 16 || RB == 32 || RB == 64 || RB == 128, "row bytes");
    if constexpr (RB == 16) return static_cast<uint32_t>(row) * 16u;
    else {
        const uint32_t lin = static_cast<uint32_t>(row) * RB;
        return lin + ((static_cast<uint32_t>(c) ^ ((lin >> 7) & (RB / 16 - 1))) << 4);
    }
}

__host__ __device__ constexpr CUtensorMapSwizzle_enum swizzle_for(int RB)
{
    return RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                     : RB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : RB == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// ------------------------------------------------------------------ TMEM of any multiple-of-4 column count

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// N consecutive 32-bit columns (N a multiple of 4, at most 64) from registers.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t *v)
{
    static_assert(N % 4 == 0 && N >= 4 && N <= 64, "4..64 columns");
    int o = 0;
    if constexpr (N >= 32) { tmem_st_x32(taddr, v); o = 32; }
    if constexpr (N >= 64) { tmem_st_x32(taddr + 32, v + 32); o = 64; }
    if constexpr ((N % 32) >= 16) { tmem_st_x16(taddr + o, v + o); o += 16; }
    if constexpr ((N % 16) >= 8) { tmem_st_x8(taddr + o, v + o); o += 8; }
    if constexpr ((N % 8) >= 4) { tmem_st_x4(taddr + o, v + o); }
}

// N consecutive 32-bit columns (N a multiple of 4, at most 64) into registers.
template <int N>
__device__ __forceinline__ void tmem_ld_any(uint32_t taddr, uint32_t *r)
{
    static_assert(N % 4 == 0 && N >= 4 && N <= 64, "4..64 columns");
    int o = 0;
    if constexpr (N >= 32) { tmem_ld_x32(taddr, r); o = 32; }
    if constexpr (N >= 64) { tmem_ld_x32(taddr + 32, r + 32); o = 64; }
    if constexpr ((N % 32) >= 16) { tmem_ld_x16(taddr + o, r + o); o += 16; }
    if constexpr ((N % 16) >= 8) { tmem_ld_x8(taddr + o, r + o); o += 8; }
    if constexpr ((N % 8) >= 4) { tmem_ld_x4(taddr + o, r + o); }
}

// Channels per step of the low-rank backward kernels: a power of two from 8 to
// 64 (the x / dy tile rows are then 16..128 bytes, one TMA swizzle mode each)
// with at most `max_cols` filter columns per step.
__host__ __device__ constexpr int lr_step_channels(int W, int max_cols)
{
    return (64 * W <= max_cols) ? 64 : (32 * W <= max_cols) ? 32 : (16 * W <= max_cols) ? 16 : 8;
}

}  // namespace dsc
