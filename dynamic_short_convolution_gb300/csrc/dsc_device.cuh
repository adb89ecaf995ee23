// dsc_device.cuh -- device-side building blocks shared by the libdsc kernels:
// mbarriers with bounded waits, TMA tile loads/stores, vector loads and stores
// of bf16 / fp32 channel groups.  Inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

namespace dsc {

// Device status codes (mirror dsc_status in dsc.h).
constexpr int kStatusTimeout = 4;
constexpr int kStatusInvalid = 1;

// Wait limit used while draining in-flight copies after an abort: always the
// fixed default, never the (possibly tiny) limit a test asked for.
constexpr unsigned long long kDrainLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record the first error of a launch in the device status word.
__device__ __forceinline__ void record_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns of wall time (and a bounded number of polls).  Returns false on
// timeout; never spins forever.  After a miss the thread backs off with a short
// sleep, so a waiting warp leaves the issue slots to the warps doing the work,
// and it reads the wall clock only every 32 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        __nanosleep(it < 4 ? 20 : 100);
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load global -> shared, completion counted on `bar` in bytes.
// c0 is the innermost (contiguous) coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Contiguous bulk copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte aligned),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 2-D tiled store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, const void *src, int c0, int c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void tma_store_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void tma_store_wait_all()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch.  grid_dependency_wait(): wait until the grids this one was allowed to
// overlap have completed and their memory operations are visible (returns at once when there are none).
// grid_dependents_launch(): let the grids that may overlap this one begin launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ element groups

template <typename E>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Load 8 consecutive elements (16 B of bf16, 32 B of fp32) as fp32; p is 16-B aligned.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void load8(const float *p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 8 consecutive elements as 4 channel pairs (fp32x2), for packed fp32 math.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ void load8x2(const __nv_bfloat16 *p, float2 (&v)[4])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    v[0] = bf16x2_to_f2(u.x);
    v[1] = bf16x2_to_f2(u.y);
    v[2] = bf16x2_to_f2(u.z);
    v[3] = bf16x2_to_f2(u.w);
}

__device__ __forceinline__ void load8x2(const float *p, float2 (&v)[4])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = make_float2(a.x, a.y);
    v[1] = make_float2(a.z, a.w);
    v[2] = make_float2(b.x, b.y);
    v[3] = make_float2(b.z, b.w);
}

__device__ __forceinline__ void store8x2(__nv_bfloat16 *p, const float2 (&v)[4])
{
    uint4 u;
    __nv_bfloat162 h0 = __float22bfloat162_rn(v[0]), h1 = __float22bfloat162_rn(v[1]);
    __nv_bfloat162 h2 = __float22bfloat162_rn(v[2]), h3 = __float22bfloat162_rn(v[3]);
    u.x = *reinterpret_cast<uint32_t *>(&h0);
    u.y = *reinterpret_cast<uint32_t *>(&h1);
    u.z = *reinterpret_cast<uint32_t *>(&h2);
    u.w = *reinterpret_cast<uint32_t *>(&h3);
    *reinterpret_cast<uint4 *>(p) = u;
}

__device__ __forceinline__ void store8x2(float *p, const float2 (&v)[4])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0].x, v[0].y, v[1].x, v[1].y);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[2].x, v[2].y, v[3].x, v[3].y);
}

// Packed fp32 fused multiply-add / multiply (two lanes per instruction on sm_100+).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// Compile-time slot of a W-slot ring: ((i % W) + W) % W.
__host__ __device__ constexpr int ring(int i, int W) { return ((i % W) + W) % W; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Store 8 fp32 values as 8 consecutive elements; p is 16-B aligned.
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8])
{
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(p) = u;
}

__device__ __forceinline__ void store8(float *p, const float (&v)[8])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Largest power of two (<= 16) dividing n.
__host__ __device__ constexpr int pow2_align(int n) { return (n % 16 == 0) ? 16 : (n % 8 == 0) ? 8 : (n % 4 == 0) ? 4 : (n % 2 == 0) ? 2 : 1; }

// Load N consecutive elements from a pointer whose byte address is a multiple
// of pow2_align(N * sizeof(E)) (the widest vector that alignment allows).
template <typename E, int N>
__device__ __forceinline__ void load_n(const E *p, float (&v)[N])
{
    constexpr int kEB = Elem<E>::kBytes;
    constexpr int kVB = pow2_align(N * kEB);      // bytes per vector access
    constexpr int kPer = kVB / kEB > 0 ? kVB / kEB : 1;
    static_assert(kVB >= kEB, "element-aligned at least");
    if constexpr (kVB == 16 || kVB == 8 || kVB == 4) {
        using V = typename std::conditional<kVB == 16, uint4, typename std::conditional<kVB == 8, uint2, uint32_t>::type>::type;
        constexpr int kWords = kVB / 4;
#pragma unroll
        for (int i = 0; i < N / kPer; ++i) {
            const V u = reinterpret_cast<const V *>(p)[i];
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&u);
#pragma unroll
            for (int j = 0; j < kWords; ++j) {
                if constexpr (sizeof(E) == 2) {
                    v[i * kPer + 2 * j] = __uint_as_float(w[j] << 16);
                    v[i * kPer + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                } else {
                    v[i * kPer + j] = __uint_as_float(w[j]);
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = Elem<E>::to_f(p[i]);
    }
}

// Store N consecutive fp32 values as elements, same alignment contract as load_n.
template <typename E, int N>
__device__ __forceinline__ void store_n(E *p, const float (&v)[N])
{
    constexpr int kEB = Elem<E>::kBytes;
    constexpr int kVB = pow2_align(N * kEB);
    if constexpr (sizeof(E) == 2 && kVB >= 4) {
        uint32_t w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        constexpr int kWordsPerVec = kVB / 4;
#pragma unroll
        for (int i = 0; i < (N / 2) / kWordsPerVec; ++i) {
            if constexpr (kWordsPerVec == 4)
                reinterpret_cast<uint4 *>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            else if constexpr (kWordsPerVec == 2)
                reinterpret_cast<uint2 *>(p)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
            else
                reinterpret_cast<uint32_t *>(p)[i] = w[i];
        }
    } else if constexpr (sizeof(E) == 4 && kVB == 16) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i)
            reinterpret_cast<float4 *>(p)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else if constexpr (sizeof(E) == 4 && kVB == 8) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) reinterpret_cast<float2 *>(p)[i] = make_float2(v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) p[i] = Elem<E>::from_f(v[i]);
    }
}

// ------------------------------------------------------------------ documents

// Number of valid taps of token t (1..W): taps k with t-k inside t's document.
// cu: packed-document offsets (n_docs + 1 entries) or nullptr.  Any content of
// cu gives an in-range result, so malformed offsets cannot cause an
// out-of-bounds access.  (Token indices are < 2^31: 32-bit arithmetic.)
__device__ __forceinline__ int valid_taps(int t, int T, int W, const int32_t *cu, int n_docs)
{
    int ds = t - t % T;  // start of t's sequence
    if (cu != nullptr) {
        int lo = 0, hi = n_docs;
        while (lo < hi) {  // largest i with cu[i] <= t
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
        }
        const int c = __ldg(cu + lo);
        if (c <= t && c > ds) ds = c;
    }
    const int nv = t - ds + 1;
    return nv < 1 ? 1 : (nv > W ? W : nv);
}

// valid_taps for a thread that asks about increasing tokens: it keeps the
// index of the last document offset <= t and walks it forward (usually zero
// or one step per token) instead of searching cu from scratch.  reset() when
// the tokens jump backwards.  Same in-range guarantee for malformed offsets.
struct DocCursor {
    int ci = -1;
    int last_t = -1, last_ds = 0;  // last token asked about and the start of its sequence
    __device__ __forceinline__ void reset()
    {
        ci = -1;
        last_t = -1;
    }
    __device__ __forceinline__ int taps(int t, int T, int W, const int32_t *cu, int n_docs)
    {
        // start of t's sequence: walked forward from the previous token (no division per call)
        int ds;
        if (last_t >= 0 && t >= last_t) {
            ds = last_ds;
            while (t - ds >= T) ds += T;
        } else {
            ds = t - t % T;
        }
        last_t = t;
        last_ds = ds;
        if (cu != nullptr) {
            if (ci < 0) {
                int lo = 0, hi = n_docs;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
                }
                ci = lo;
            }
            while (ci < n_docs && __ldg(cu + ci + 1) <= t) ++ci;
            const int c = __ldg(cu + ci);
            if (c <= t && c > ds) ds = c;
        }
        const int nv = t - ds + 1;
        return nv < 1 ? 1 : (nv > W ? W : nv);
    }
};

}  // namespace dsc
