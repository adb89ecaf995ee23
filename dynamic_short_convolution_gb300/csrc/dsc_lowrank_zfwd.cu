// dsc_lowrank_zfwd.cu -- forward pass of the low-rank dynamic short
// convolution with both projections of the filter generator on chip
// ("Parameterization": the generator maps the layer input through
// D -> R -> W*D; "Placement": its first projection runs beside the Q/K/V
// projection; "Efficient training": the generated filter never reaches HBM):
//
//   z[t, r]      = sum_i h[t, i] W1[r, i] + b1[r]               (tensor cores, per token tile)
//   Wt[t, d*W+k] = sum_r z[t, r] U[r, d*W+k] + bias[d*W+k]       (tensor cores, per unit)
//   y[t, d]      = x[t, d] + sum_k Wt[t, d*W+k] * x~[t-k, d]      (epilogue)
//
// The code z is never stored: it lives in TMEM, then in shared memory as an
// exact pair of bf16 halves (z_hi = bf16(z), z_lo = bf16(z - z_hi), together
// z to about 16 significant bits) that is the A operand of the second
// projection for every channel block of its token tile: [z_hi | z_lo] against
// [U ; U], then an all-ones tile against the bias rows [b_hi ; b_lo ; 0..].
//
// Work unit: 128 tokens x one block of CB channels, ordered token-major; a
// CTA takes a contiguous run of units, which covers one or two token tiles,
// and computes z once for each tile it touches.  (Whole tiles per CTA read h
// once but leave SMs idle when there are fewer tiles than SMs: measured
// slower.)  One ring of shared-memory slots carries two kinds of items in the
// order the CTA needs them: "z items" (two 64-wide K chunks of the h tile and
// of W1) when a token tile starts, and one "unit item" per unit (the block's
// U rows with the bias as 16 extra rows, and the x tile with its (W-1)-token
// causal halo).
//   warp 0      producer: TMA loads of every item; writes the bias rows of
//               each unit item (bf16 hi and lo, 14 zero rows after them) from
//               the bias it loaded during the previous item
//   warp 1      TMEM owner; lane 0 issues the z MMAs (M=128, N=R, K=16) into
//               the accumulator the tile's first unit will use, then per unit
//               the filter MMAs [z_hi | z_lo | 1] . [U ; U ; b_hi + b_lo]
//   warps 2..17 epilogue: at a token tile's start they read z from TMEM, add
//               b1 and write it as the bf16 hi + lo z tile; per unit, as the
//               low-rank forward: the accumulator row of a token times its x
//               window, plus the residual, staged and TMA-stored per warp
#include <type_traits>

#include "dsc_internal.h"
#include "dsc_lowrank_common.cuh"
#include "dsc_lowrank_epi.cuh"

namespace dsc {

// A 2-D tiled TMA load with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// L2 policy for data read once: its lines leave L2 first.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

namespace lrz {

constexpr int kM = 128;            // tokens per tile (MMA M, TMEM lanes)
constexpr int kEpiWarps = 16;      // four per TMEM lane quadrant
constexpr int kEpiWarp0 = 2;       // warps 0, 1: producer, MMA issuer
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kMaxSlots = 6;
constexpr int kTmemCols = 512;     // two accumulators of up to 256 columns

struct Params {
    const float *b1;               // the first projection's bias [R], or null
    const float *bias;
    const int32_t *cu;
    int n_docs;
    int BT, T, D, Dm, R, N;        // N = D * W filter columns
    int rp;                        // R rounded up to 16: MMA N of the z product, K of the filter product
    int n_nb, n_mt, n_units, n_zitems;  // channel blocks, token tiles, units, z items per token tile
    unsigned ublk;                 // bytes of one 64-column block of a unit item's U rows: (rp + 16) rows x 128 B
    unsigned zt_off, one_off, y_off, ring_off, slot_bytes, x_in_slot, w1_in_slot;
    unsigned u_bytes, x_bytes, z_item_bytes;  // TMA bytes of a unit item's U rows and x tile, of a z item
    int nslots;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t z_full, z_ready, drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct RingPos {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void step(int n)
    {
        if (++s == n) {
            s = 0;
            ph ^= 1u;
        }
    }
};

}  // namespace lrz

template <int W, int CB>
__global__ void __launch_bounds__(lrz::kThreads, 1)
    lowrank_zfwd_tc(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_y, const lrz::Params p)
{
    using namespace lrz;
    constexpr int NB = CB * W;         // filter columns per block (MMA N of the filter product)
    constexpr int RB = CB * 2;         // bytes per x / y tile row
    constexpr int GROUPS = CB / 8;     // 8-channel groups per block
    constexpr int NCW = GROUPS < 4 ? GROUPS : 4;  // epilogue warps with work per lane quadrant
    constexpr int GPW = GROUPS / NCW;  // groups per working epilogue warp
    constexpr int YB = RB / NCW;       // bytes of a warp's y staging row
    constexpr int NBLK = (NB + 63) / 64;  // 64-column blocks of the U rows (the last may be partial)
    static_assert(NB % 16 == 0 && NB <= 256 && GROUPS % NCW == 0, "MMA N, channel groups");
    constexpr uint32_t IDESC_F = idesc_bf16_f32(kM, NB, false, true);  // A z tile K-major, B U rows MN-major

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *zt = base + p.zt_off;       // z tile: [128 tokens][2 rp] bf16, K-major, 64-column chunks of 16 KB
    uint8_t *one_s = base + p.one_off;   // all-ones A tile [128 rows][16 K], no swizzle: meets the bias rows
    uint8_t *y_s = base + p.y_off;       // per working epilogue warp: [32 rows][YB] staging for its own stores
    uint8_t *ring = base + p.ring_off;   // nslots slots of slot_bytes

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1 + 4 * NCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->tmem_full[b], 1);
            mbar_init(&hdr->tmem_empty[b], 4 * NCW);
        }
        mbar_init(&hdr->z_full, 1);
        mbar_init(&hdr->z_ready, 4 * NCW);
        mbar_init(&hdr->drain, 1);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kM * 16 / 2; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(&hdr->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // this launch may overlap the end of the stream's previous kernel: every access to global memory
    // comes after the wait; the next kernel may begin its own prologue as soon as this one runs
    grid_dependents_launch();
    grid_dependency_wait();
    const uint32_t tmem = hdr->tmem_base;
    volatile int *abort_flag = &hdr->abort_flag;

    const int u_begin = static_cast<int>(static_cast<long long>(blockIdx.x) * p.n_units / gridDim.x);
    const int u_end = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.n_units / gridDim.x);

    int issued_last[kMaxSlots];  // producer: last item index loaded into each slot
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s) issued_last[s] = -1;
    bool mma_issued = false;     // MMA thread: some MMA may still be in flight

    if (warp == 0) {
        // ---------------- producer
        RingPos rs;
        int item = 0;
        int cur_mt = -1;
        bool ok = true;
        // x is read once: its lines may leave L2 first
        const uint64_t pol_once = l2_policy_evict_first();
        float bv[8];  // this lane's 8 bias columns (chunk `lane`) of the next unit item's block
        auto load_bias = [&](int nbx) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int gn = nbx * NB + lane * 8 + e;
                bv[e] = (lane < NB / 8 && gn < p.N) ? __ldg(p.bias + gn) : 0.f;
            }
        };
        if (u_begin < u_end) load_bias(u_begin % p.n_nb);
        for (int v = u_begin; v < u_end && ok; ++v) {
            const int mt = v / p.n_nb, nb = v - mt * p.n_nb;
            if (mt != cur_mt) {
                for (int zi = 0; zi < p.n_zitems && ok; ++zi, ++item, rs.step(p.nslots)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&hdr->empty[rs.s], rs.ph ^ 1, p.wait_ns)) &&
                         (*abort_flag == 0);
                    if (ok && lane == 0) {
                        uint8_t *sl = ring + rs.s * p.slot_bytes;
                        mbar_arrive_expect_tx(&hdr->full[rs.s], p.z_item_bytes);
                        for (int c = 0; c < 2; ++c) {
                            const int k0 = (2 * zi + c) * 64;
                            tma_load_2d(sl + c * 16384, &tm_h, &hdr->full[rs.s], k0, mt * kM);
                            tma_load_2d(sl + p.w1_in_slot + c * (p.rp * 128), &tm_w1, &hdr->full[rs.s], k0, 0);
                        }
                        issued_last[rs.s] = item;
                    }
                }
                cur_mt = mt;
            }
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(&hdr->empty[rs.s], rs.ph ^ 1, p.wait_ns)) && (*abort_flag == 0);
            if (!ok) break;
            uint8_t *sl = ring + rs.s * p.slot_bytes;
            // the bias rows rp .. rp+15 of each 64-column block (128-byte swizzled, MN-major like the U rows):
            // row rp = bf16(b), row rp+1 = bf16(b - bf16(b)) from this lane's 8 columns, the rest zero
            if (lane < NB / 8) {
                uint32_t whi[4], wlo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 hv = __float22bfloat162_rn(make_float2(bv[2 * e], bv[2 * e + 1]));
                    __nv_bfloat162 lv = __float22bfloat162_rn(
                        make_float2(bv[2 * e] - __low2float(hv), bv[2 * e + 1] - __high2float(hv)));
                    whi[e] = *reinterpret_cast<uint32_t *>(&hv);
                    wlo[e] = *reinterpret_cast<uint32_t *>(&lv);
                }
                const int blk = lane >> 3, c8 = lane & 7;
                *reinterpret_cast<uint4 *>(sl + blk * p.ublk + p.rp * 128 + ((c8 ^ (p.rp & 7)) << 4)) =
                    make_uint4(whi[0], whi[1], whi[2], whi[3]);
                *reinterpret_cast<uint4 *>(sl + blk * p.ublk + (p.rp + 1) * 128 + ((c8 ^ ((p.rp + 1) & 7)) << 4)) =
                    make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
            }
            for (int q = lane; q < (NB / 8) * 14; q += 32) {
                const int kr = p.rp + 2 + q / (NB / 8), cc = q % (NB / 8);
                *reinterpret_cast<uint4 *>(sl + (cc >> 3) * p.ublk + kr * 128 + (((cc & 7) ^ (kr & 7)) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&hdr->full[rs.s], p.u_bytes + p.x_bytes);
                for (int blk = 0; blk < NBLK; ++blk)
                    tma_load_2d(sl + blk * p.ublk, &tm_u, &hdr->full[rs.s], nb * NB + blk * 64, 0);
                tma_load_2d_hint(sl + p.x_in_slot, &tm_x, &hdr->full[rs.s], nb * CB, mt * kM - (W - 1), pol_once);
                issued_last[rs.s] = item;
            }
            ++item;
            rs.step(p.nslots);
            if (v + 1 < u_end) load_bias((v + 1) % p.n_nb);  // the next item's bias, loaded while this one flies
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
    } else if (warp == 1) {
        // ---------------- MMA issuer
        RingPos rs;
        int cur_mt = -1;
        uint32_t zc = 0;  // token tiles started (z phases)
        bool ok = true;
        for (int v = u_begin, i = 0; v < u_end && ok; ++v, ++i) {
            const int mt = v / p.n_nb;
            const int b = i & 1;
            const uint32_t tph = (i >> 1) & 1;
            bool have_tmem = false;
            if (mt != cur_mt) {
                // z = h W1^T into this unit's accumulator (its first rp columns)
                ok = __all_sync(0xffffffffu, mbar_wait(&hdr->tmem_empty[b], tph ^ 1, p.wait_ns)) &&
                     (*abort_flag == 0);
                have_tmem = true;
                const uint32_t idesc_z = idesc_bf16_f32(kM, p.rp, false, false);
                for (int zi = 0; zi < p.n_zitems && ok; ++zi, rs.step(p.nslots)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&hdr->full[rs.s], rs.ph, p.wait_ns)) && (*abort_flag == 0);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sl = smem_u32(ring + rs.s * p.slot_bytes);
                        for (int c = 0; c < 2; ++c)
                            for (int kk = 0; kk < 4; ++kk)
                                umma_bf16(tmem + b * 256, sdesc_kmajor_sw128(sl + c * 16384 + kk * 32),
                                          sdesc_kmajor_sw128(sl + p.w1_in_slot + c * (p.rp * 128) + kk * 32),
                                          idesc_z, (zi | c | kk) ? 1u : 0u);
                        umma_commit(&hdr->empty[rs.s]);
                        mma_issued = true;
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) umma_commit(&hdr->z_full);
                __syncwarp();
                // the epilogue turns z into the bf16 z tile
                ok = __all_sync(0xffffffffu, mbar_wait(&hdr->z_ready, zc & 1, p.wait_ns)) && (*abort_flag == 0);
                ++zc;
                cur_mt = mt;
                if (!ok) break;
            }
            ok = mbar_wait(&hdr->full[rs.s], rs.ph, p.wait_ns) &&
                 (have_tmem || mbar_wait(&hdr->tmem_empty[b], tph ^ 1, p.wait_ns));
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                // [z_hi | z_lo] . [U ; U]: rp/16 K steps of each half of the code against the same U rows; then
                // ones . [b_hi ; b_lo ; 0 ..], the bias rows after the U rows
                const uint32_t sl = smem_u32(ring + rs.s * p.slot_bytes);
                const uint32_t zs = smem_u32(zt);
                const int nks = p.rp / 16;
                for (int ks = 0; ks < 2 * nks; ++ks)
                    umma_bf16(tmem + b * 256, sdesc_kmajor_sw128(zs + (ks >> 2) * 16384 + (ks & 3) * 32),
                              sdesc(sl + (ks < nks ? ks : ks - nks) * 2048, p.ublk, 1024, 2), IDESC_F,
                              ks > 0 ? 1u : 0u);
                umma_bf16(tmem + b * 256, sdesc(smem_u32(one_s), 128, 256, 0), sdesc(sl + nks * 2048, p.ublk, 1024, 2),
                          IDESC_F, 1u);
                umma_commit(&hdr->empty[rs.s]);
                umma_commit(&hdr->tmem_full[b]);
                mma_issued = true;
            }
            __syncwarp();
            rs.step(p.nslots);
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
    } else if (((warp - kEpiWarp0) >> 2) < NCW) {
        // ---------------- epilogue
        const int q = warp & 3;                          // TMEM lane quadrant
        const int h = (warp - kEpiWarp0) >> 2;           // which share of the channel groups (and of z's columns)
        const int row = q * 32 + lane;                   // token within the tile
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        uint8_t *ys = y_s + (warp - kEpiWarp0) * (32 * YB);
        DocCursor cursor;
        int nv = W, nv_mt = -1;  // valid taps of this thread's token in tile nv_mt
        bool full_taps = true;
        RingPos rs;
        int cur_mt = -1;
        uint32_t zc = 0;
        bool ok = true;
        for (int v = u_begin, i = 0; v < u_end && ok; ++v, ++i) {
            const int mt = v / p.n_nb, nb = v - mt * p.n_nb;
            const int b = i & 1;
            const uint32_t tph = (i >> 1) & 1;
            if (mt != cur_mt) {
                // the z items are not read here: hand each slot back once its item has arrived (an arrival for a
                // later item must not reach a slot's barrier before the phase of the item before it completed)
                for (int zi = 0; zi < p.n_zitems && ok; ++zi, rs.step(p.nslots)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&hdr->full[rs.s], rs.ph, p.wait_ns));
                    if (ok && lane == 0) mbar_arrive(&hdr->empty[rs.s]);
                }
                if (!ok) break;
                ok = __all_sync(0xffffffffu, mbar_wait(&hdr->z_full, zc & 1, p.wait_ns));
                ++zc;
                if (!ok) break;
                tc_fence_after();
                // z (fp32, this unit's accumulator) -> the z tile as bf16 hi (columns g*8..) and lo (rp + g*8..),
                // 8 columns per step; every filter MMA of the previous tile completed before the accumulators
                // this warp already waited for
                for (int g = h; g < p.rp / 8; g += NCW) {
                    uint32_t zr[8];
                    tmem_ld_x8(tmem + lane_off + b * 256 + g * 8, zr);
                    float b1v[8];  // the first projection's bias of these 8 columns (none past R)
#pragma unroll
                    for (int e = 0; e < 8; ++e) b1v[e] = (p.b1 != nullptr && g * 8 + e < p.R) ? __ldg(p.b1 + g * 8 + e) : 0.f;
                    tmem_ld_wait();
                    uint32_t whi[4], wlo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float z0 = __uint_as_float(zr[2 * e]) + b1v[2 * e];
                        const float z1 = __uint_as_float(zr[2 * e + 1]) + b1v[2 * e + 1];
                        __nv_bfloat162 hv = __float22bfloat162_rn(make_float2(z0, z1));
                        __nv_bfloat162 lv = __float22bfloat162_rn(
                            make_float2(z0 - __low2float(hv), z1 - __high2float(hv)));
                        whi[e] = *reinterpret_cast<uint32_t *>(&hv);
                        wlo[e] = *reinterpret_cast<uint32_t *>(&lv);
                    }
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const int kc = part * p.rp + g * 8;
                        const uint32_t *w = part ? wlo : whi;
                        *reinterpret_cast<uint4 *>(zt + (kc >> 6) * 16384 + row * 128 +
                                                   ((((kc & 63) >> 3) ^ (row & 7)) << 4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->z_ready);
                cur_mt = mt;
            }
            if (mt != nv_mt) {  // this thread's token, hence its valid taps, changes only with the tile
                const int t = mt * kM + row;
                nv = t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W;
                full_taps = __all_sync(0xffffffffu, nv == W);
                nv_mt = mt;
            }
            ok = mbar_wait(&hdr->tmem_full[b], tph, p.wait_ns) && mbar_wait(&hdr->full[rs.s], rs.ph, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint8_t *xs = ring + rs.s * p.slot_bytes + p.x_in_slot;
            const uint32_t trow = tmem + lane_off + b * 256;
            uint4 o[GPW];
#pragma unroll
            for (int gi = 0; gi < GPW; ++gi) {
                const int g = h * GPW + gi;  // 8-channel group
                o[gi] = lr_group_y<W, RB>(trow + g * 8 * W, xs, row, g, full_taps, nv);
            }
            // accumulator and x tile read: hand them back; stage and store this warp's y sub-tile (the staging
            // tile is free once the store issued a unit ago has read it)
            tc_fence_before();
            if (lane == 0) tma_store_wait_read<0>();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&hdr->tmem_empty[b]);
                mbar_arrive(&hdr->empty[rs.s]);
            }
#pragma unroll
            for (int gi = 0; gi < GPW; ++gi) *reinterpret_cast<uint4 *>(ys + lane * YB + gi * 16) = o[gi];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tm_y, ys, nb * CB + h * (CB / NCW), mt * kM + q * 32);
                tma_store_commit();
            }
            rs.step(p.nslots);
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
    }
    // ---- teardown: no copy or MMA of this CTA may still be in flight
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (int s = 0; s < p.nslots; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / p.nslots) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
        umma_commit(&hdr->drain);
        (void)mbar_wait(&hdr->drain, 0, kDrainLimitNs);
    }
    if (warp >= kEpiWarp0 && lane == 0) tma_store_wait_all<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

template <int W, int CB>
static dsc_status launch_zfwd(const LowrankZArgs &a, const DeviceInfo &dev)
{
    using namespace lrz;
    constexpr int NB = CB * W, RB = CB * 2, XR = kM + W - 1, NBLK = (NB + 63) / 64;
    constexpr int NCW = CB / 8 < 4 ? CB / 8 : 4;
    Params p{};
    p.b1 = a.b1;
    p.bias = a.bias;
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.Dm = a.Dm;
    p.R = a.R;
    p.N = a.D * a.W;
    p.rp = (a.R + 15) / 16 * 16;
    p.n_nb = (a.D + CB - 1) / CB;
    p.n_mt = (p.BT + kM - 1) / kM;
    const long long units = static_cast<long long>(p.n_nb) * p.n_mt;
    if (units > 0x7fffffffLL) return DSC_ERR_UNSUPPORTED;
    p.n_units = static_cast<int>(units);
    p.n_zitems = (a.Dm + 127) / 128;  // two 64-wide K chunks per item (a chunk past Dm arrives as zeros)
    p.ublk = static_cast<unsigned>(p.rp + 16) * 128;
    // a slot holds either a unit item [U rows of NBLK blocks][x tile] or a z item [h chunks][W1 chunks]
    p.x_in_slot = align_up(NBLK * p.ublk, 1024);
    const unsigned unit_slot = p.x_in_slot + align_up(XR * RB, 1024);
    p.w1_in_slot = 2 * 16384;
    const unsigned z_slot = p.w1_in_slot + 2 * p.rp * 128;
    p.slot_bytes = unit_slot > z_slot ? unit_slot : z_slot;
    p.u_bytes = NBLK * p.rp * 128;
    p.x_bytes = XR * RB;
    p.z_item_bytes = 2 * 16384 + 2 * p.rp * 128;
    // shared memory: [header 1 KB][align slack 1 KB][z tile][ones tile][y staging][ring]
    p.zt_off = 0;
    p.one_off = ((2 * p.rp + 63) / 64) * 16384;
    unsigned off = p.one_off + kM * 32;
    p.y_off = align_up(off, 1024);
    off = p.y_off + kEpiWarps * 32 * (RB / NCW);
    p.ring_off = align_up(off, 1024);
    const unsigned fixed = 2048 + p.ring_off;
    if (static_cast<unsigned>(dev.max_smem_optin) < fixed + 2 * p.slot_bytes) return DSC_ERR_UNSUPPORTED;
    const int ns = static_cast<int>((dev.max_smem_optin - fixed) / p.slot_bytes);
    p.nslots = ns > kMaxSlots ? kMaxSlots : ns;
    const unsigned smem = fixed + p.nslots * p.slot_bytes;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    CUtensorMap tm_h, tm_w1, tm_u, tm_x, tm_y;
    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    if (!encode_tmap_2d(&tm_h, a.h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.Dm, BT, static_cast<unsigned long long>(a.Dm) * 2,
                        64, kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_w1, a.W1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.Dm, a.R,
                        static_cast<unsigned long long>(a.Dm) * 2, 64, p.rp, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_u, a.U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.N, a.R, static_cast<unsigned long long>(p.N) * 2,
                        64, p.rp, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB, XR, swizzle_for(RB)) ||
        !encode_tmap_2d(&tm_y, a.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB / NCW, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_CUDA;
    auto kern = lowrank_zfwd_tc<W, CB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int grid = dev.sm_count < p.n_units ? dev.sm_count : p.n_units;
    return launch_overlapped(kern, grid, kThreads, smem, a.stream, tm_h, tm_w1, tm_u, tm_x, tm_y, p);
}

dsc_status lowrank_zproj_fwd(const LowrankZArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R > 128) return DSC_ERR_UNSUPPORTED;
    // the widest channel block (64, 32 or 16 channels: fewer units, longer DRAM row pieces) whose U rows leave
    // room for two ring slots beside the z tile; 64 only while the block's filter columns fit one accumulator
    auto launch_w = [&](auto wtag) -> dsc_status {
        constexpr int Wc = decltype(wtag)::value;
        dsc_status s = DSC_ERR_UNSUPPORTED;
        if constexpr (Wc <= 4) s = launch_zfwd<Wc, 64>(a, dev);
        if (s == DSC_ERR_UNSUPPORTED) s = launch_zfwd<Wc, 32>(a, dev);
        if (s == DSC_ERR_UNSUPPORTED) s = launch_zfwd<Wc, 16>(a, dev);
        return s;
    };
    switch (a.W) {
    case 1: return launch_w(std::integral_constant<int, 1>{});
    case 2: return launch_w(std::integral_constant<int, 2>{});
    case 3: return launch_w(std::integral_constant<int, 3>{});
    case 4: return launch_w(std::integral_constant<int, 4>{});
    case 5: return launch_w(std::integral_constant<int, 5>{});
    case 6: return launch_w(std::integral_constant<int, 6>{});
    case 7: return launch_w(std::integral_constant<int, 7>{});
    case 8: return launch_w(std::integral_constant<int, 8>{});
    default: return DSC_ERR_INVALID_ARG;
    }
}

}  // namespace dsc
