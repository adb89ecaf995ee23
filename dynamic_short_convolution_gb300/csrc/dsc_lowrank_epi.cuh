// dsc_lowrank_epi.cuh -- the epilogue arithmetic shared by the low-rank
// forward kernels (the low-rank form of "Parameterization", eq. 2 with the
// residual of eq. 3): y of one token's group of 8 channels from its filter
// row, held in TMEM, and its causal x window, held in a swizzled x tile in
// shared memory.
#pragma once

#include <cuda_bf16.h>

#include "dsc_lowrank_common.cuh"

namespace dsc {

// y[t, c] = x[t, c] + sum_k acc[c*W + k] * x~[t-k, c] for the 8 channels c of group g, as packed bf16 pairs.
// tcol: TMEM address of the group's 8W filter columns for this thread's lane (tap k of channel c at c*W + k);
// xs: the x tile (rows of RB bytes, token row r + W-1 holds the tile's token r); row: this thread's token in
// the tile.  When the warp is not clear of a document start (full_taps false), taps k >= nv read zero.  For
// W > 4 the group is formed in two halves of four channels, so that a half's filter (4W registers) and x window
// (2W registers) fit beside the rest of the kernel without spilling.
template <int W, int RB>
__device__ __forceinline__ uint4 lr_group_y(uint32_t tcol, const uint8_t *xs, int row, int g, bool full_taps, int nv)
{
    constexpr int NH = W > 4 ? 2 : 1;  // halves
    constexpr int EH = 4 / NH;         // channel pairs per half
    constexpr int NC = 8 * W / NH;     // filter columns per half
    uint32_t packed[4];
#pragma unroll
    for (int hv = 0; hv < NH; ++hv) {
        uint32_t acc[NC];  // acc[c*W + k]: tap k of the half's channel c
        tmem_ld_any<NC>(tcol + hv * NC, acc);
        uint32_t xw[W][EH];  // x~ rows row-k of the half's channels, bf16 pairs
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const uint8_t *src = xs + swzt<RB>(row + (W - 1) - k, g) + hv * (4 * EH);
            if constexpr (EH == 4) {
                const uint4 r = *reinterpret_cast<const uint4 *>(src);
                xw[k][0] = r.x;
                xw[k][1] = r.y;
                xw[k][2] = r.z;
                xw[k][3] = r.w;
            } else {
                const uint2 r = *reinterpret_cast<const uint2 *>(src);
                xw[k][0] = r.x;
                xw[k][1] = r.y;
            }
        }
        if (!full_taps) {  // x~ is zero before the document start (warp-uniform branch)
#pragma unroll
            for (int k = 1; k < W; ++k)
#pragma unroll
                for (int e = 0; e < EH; ++e) xw[k][e] = k < nv ? xw[k][e] : 0u;
        }
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < EH; ++e) {
            float y2[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {  // the half's channel c = 2e + h2
                const int c = 2 * e + h2;
                auto xv = [&](int k) {
                    const uint32_t w2 = xw[k][e];
                    return __uint_as_float(h2 ? (w2 & 0xffff0000u) : (w2 << 16));
                };
                // residual + sum_k acc_k * x~_k, taps paired for packed fp32x2 arithmetic
                float2 sum = make_float2(xv(0), 0.f);
#pragma unroll
                for (int k = 0; k + 1 < W; k += 2)
                    sum = fma2(make_float2(__uint_as_float(acc[c * W + k]), __uint_as_float(acc[c * W + k + 1])),
                               make_float2(xv(k), xv(k + 1)), sum);
                if constexpr (W % 2 == 1) sum.x = fmaf(__uint_as_float(acc[c * W + W - 1]), xv(W - 1), sum.x);
                y2[h2] = sum.x + sum.y;
            }
            __nv_bfloat162 hv2 = __float22bfloat162_rn(make_float2(y2[0], y2[1]));
            packed[hv * EH + e] = *reinterpret_cast<uint32_t *>(&hv2);
        }
    }
    return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace dsc
