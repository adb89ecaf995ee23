// dsc_lowrank_fwd.cu -- forward pass of the low-rank dynamic short convolution
// with the filter generator fused ("Parameterization": D -> R -> W*D with a
// bias; "Efficient training": the second projection is fused into the kernel,
// reads z and U, and the generated filter never reaches HBM):
//
//   Wt[t, d*W+k] = sum_r z[t,r] U[r, d*W+k] + bias[d*W+k]        (tensor cores)
//   y[t,d]       = x[t,d] + sum_k Wt[t, d*W+k] * x~[t-k, d]       (epilogue)
//
// Work unit: 128 tokens x one block of CB channels (NB = CB*W filter columns).
// A persistent CTA takes a contiguous run of units ordered block-major, so the
// U block (TMA, 128-byte swizzle, read as an MN-major operand) stays resident
// in shared memory while the CTA streams over token tiles.
//   warp 0      TMA producer: z tile (K-major, swizzled) and the x tile with
//               its (W-1)-token causal halo; the tile's per-token valid-tap
//               counts, written beside the x tile while the loads fly
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=NB, K=16 per
//               instruction) into one of two TMEM accumulators
//   warps 2..17 epilogue: tcgen05.ld of the accumulator row of one token,
//               + bias, times the x window from shared memory, + residual,
//               bf16 into a swizzled staging tile that one thread TMA-stores
// The filter columns keep their natural order (column c*W + k for channel c,
// tap k): the W taps of one channel are adjacent accumulator columns, so tap
// pairs feed packed fp32x2 math straight from TMEM registers.
#include "dsc_internal.h"
#include "dsc_lowrank_common.cuh"  // swizzled tile offsets (swzt), swizzle_for; tcgen05 wrappers
#include "dsc_lowrank_epi.cuh"    // y of a token's 8-channel group from its filter row and x window

namespace dsc {

namespace lrf {

constexpr int kM = 128;            // tokens per tile (MMA M, TMEM lanes)
constexpr int kEpiWarps = 16;      // four per TMEM lane quadrant
constexpr int kEpiWarp0 = 2;       // warps 0, 1: producer, MMA issuer
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kMaxStages = 6;
constexpr int kTmemCols = 512;     // two accumulators of up to 256 columns

struct Params {
    const __nv_bfloat16 *U;
    const float *bias;
    const int32_t *cu;
    int n_docs;
    int BT, T, D, R, N;            // N = D * W filter columns
    int n_nb, n_mt, n_units;
    int ksteps, kchunks;           // MMA K steps of 16; 64-wide K chunks of z
    unsigned u_bytes, u_blk_bytes; // U of a block in shared memory; one 64-column block of it
    unsigned u_off, bt_off, one_off, y_off, st_off, stage_bytes, z_bytes, x_bytes, x_off_in_stage, nv_off_in_stage;
    int nstages;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t u_full, u_free;
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace lrf

template <int W, int CB>
__global__ void __launch_bounds__(lrf::kThreads, 1)
    lowrank_fwd_tc(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_u,
                   const lrf::Params p)
{
    using namespace lrf;
    constexpr int NB = CB * W;         // filter columns per block (MMA N)
    constexpr int RB = CB * 2;         // bytes per x / y tile row
    constexpr int GROUPS = CB / 8;     // 8-channel groups per block
    constexpr int NCW = GROUPS < 4 ? GROUPS : 4;  // epilogue warps with work per lane quadrant
    constexpr int GPW = GROUPS / NCW;  // groups per working epilogue warp
    constexpr int YB = RB / NCW;       // bytes of a warp's y staging row (its CB / NCW channels)
    static_assert(NB % 16 == 0 && NB <= 256 && GROUPS % NCW == 0, "MMA N, channel groups");
    constexpr uint32_t IDESC = idesc_bf16_f32(kM, NB, false, true);        // A z K-major, B U MN-major
    constexpr uint32_t IDESC_BIAS = idesc_bf16_f32(kM, NB, false, false);  // A ones, B bias tile, both K-major

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *u_s = base + p.u_off;       // [NB/64 blocks][Rp rows][128 B]: U of the block, 128-B swizzled
    uint8_t *bt_s = base + p.bt_off;     // bias as an MMA B tile: [NB rows][16 K], no swizzle
    uint8_t *one_s = base + p.one_off;   // all-ones MMA A tile [128 rows][16 K]
    uint8_t *y_s = base + p.y_off;       // per working epilogue warp: 2 x [32 rows][YB] staging for its own stores
    uint8_t *stages = base + p.st_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1 + 4 * NCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->tmem_full[b], 1);
            mbar_init(&hdr->tmem_empty[b], 4 * NCW);
        }
        mbar_init(&hdr->u_full, 1);
        mbar_init(&hdr->u_free, 1);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kM * 16 / 2; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    // bias B tile, core matrices of 8 rows x 16 B: column n's first K pair (at ((n/8)*2)*128 + (n%8)*16) holds
    // the bias as an exact bf16 hi + lo pair, the rest of its K = 16 is zero.  Only the pair changes per block.
    for (int i = threadIdx.x; i < NB * 2; i += blockDim.x)
        reinterpret_cast<uint4 *>(bt_s)[i] = make_uint4(0u, 0u, 0u, 0u);
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

    int issued_last[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
    int mma_last = -1;      // last tile whose MMAs were committed (MMA thread)
    int seg = 0;            // filter-generator loads so far (MMA warp)
    bool u_pending = false; // MMA warp: a U load is in flight and was not seen to complete

    if (warp == 0) {
        // ---------------- producer: streams z and x tiles from the first cycle, across block changes
        DocCursor cursor;  // lane l: tokens l, l+32, l+64, l+96 of each tile, increasing within a block
        int i = 0;
        int s = 0;                                  // stage and its phase: stepped, not divided, per tile
        uint32_t ph = 0;
        int nb = u_begin / p.n_mt, mt = u_begin - nb * p.n_mt;
        for (int v = u_begin; v < u_end;
             ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0), mt = (mt + 1 == p.n_mt) ? 0 : mt + 1,
                 nb += (mt == 0)) {
            bool ok = mbar_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) {
                if (lane == 0) {
                    record_status(p.status, kStatusTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            const int t0 = mt * kM;
            uint8_t *st = stages + s * p.stage_bytes;
            // valid taps of the tile's tokens (the slot is free: the epilogue read the previous ones first)
            if (mt == 0 || v == u_begin) cursor.reset();
            int8_t *nvs = reinterpret_cast<int8_t *>(st + p.nv_off_in_stage);
#pragma unroll
            for (int r = 0; r < kM; r += 32) {
                const int t = t0 + r + lane;
                nvs[r + lane] = static_cast<int8_t>(t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&hdr->full[s], p.z_bytes + p.x_bytes);
                for (int a = 0; a < p.kchunks; ++a) tma_load_2d(st + a * 16384, &tm_z, &hdr->full[s], a * 64, t0);
                tma_load_2d(st + p.x_off_in_stage, &tm_x, &hdr->full[s], nb * CB, t0 - (W - 1));
                issued_last[s] = i;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: acc = z . U_blk (K = R), then += 1 . bias.  This warp also loads each
        // block's filter generator, once the previous block's MMAs have completed, so that the producer never
        // stops streaming and no other warp waits at a block change.
        int i = 0;
        int s = 0;
        uint32_t ph = 0;
        int nb = u_begin / p.n_mt, mt = u_begin - nb * p.n_mt;
        int cur_nb = -1;
        for (int v = u_begin; v < u_end;
             ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0), mt = (mt + 1 == p.n_mt) ? 0 : mt + 1,
                 nb += (mt == 0)) {
            if (nb != cur_nb) {
                // U[:, nb*NB .. +NB) by TMA (rows past R arrive as zeros); the bias as an extra K step (exact
                // bf16 hi + lo pair) that the all-ones A tile adds in
                float bv[(NB + 31) / 32];
#pragma unroll
                for (int j = 0; j < (NB + 31) / 32; ++j) {
                    const int n = lane + 32 * j, gn = nb * NB + n;
                    bv[j] = (n < NB && gn < p.N) ? p.bias[gn] : 0.f;
                }
                bool ok = true;
                if (cur_nb >= 0) {  // the previous block's MMAs still read U and the bias tile
                    if (lane == 0) umma_commit(&hdr->u_free);
                    __syncwarp();
                    ok = mbar_wait(&hdr->u_free, (seg - 1) & 1, p.wait_ns);
                }
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (ok) {
#pragma unroll
                    for (int j = 0; j < (NB + 31) / 32; ++j) {
                        const int n = lane + 32 * j;
                        if (n < NB) {
                            const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv[j])));
                            const uint32_t lo = static_cast<uint32_t>(
                                __bfloat16_as_ushort(__float2bfloat16_rn(bv[j] - __uint_as_float(hi << 16))));
                            *reinterpret_cast<uint32_t *>(bt_s + ((n >> 3) * 2) * 128 + (n & 7) * 16) = hi | (lo << 16);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&hdr->u_full, p.u_bytes);
                        for (int blk = 0; blk < (NB + 63) / 64; ++blk)
                            tma_load_2d(u_s + blk * p.u_blk_bytes, &tm_u, &hdr->u_full, nb * NB + blk * 64, 0);
                    }
                    u_pending = true;
                    ok = __all_sync(0xffffffffu, mbar_wait(&hdr->u_full, seg & 1, p.wait_ns));
                    if (ok) u_pending = false;
                }
                ++seg;
                cur_nb = nb;
                if (!ok) {
                    if (lane == 0) {
                        record_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                    }
                    break;
                }
            }
            const int b = i & 1;
            const uint32_t tph = (i >> 1) & 1;
            bool ok = mbar_wait(&hdr->full[s], ph, p.wait_ns) && mbar_wait(&hdr->tmem_empty[b], tph ^ 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) {
                if (lane == 0) {
                    record_status(p.status, kStatusTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t zs = smem_u32(stages + s * p.stage_bytes);
                const uint32_t us = smem_u32(u_s);
                const uint32_t d = tmem + b * 256;
                for (int ks = 0; ks < p.ksteps; ++ks) {
                    // A: z, K-major, 64-column chunks; B: U, MN-major, 16 rows of R per K step, 64-column
                    // blocks p.u_blk_bytes apart
                    const int a = ks >> 2, kk = ks & 3;
                    const uint64_t ad = sdesc_kmajor_sw128(zs + a * 16384 + kk * 32);
                    const uint64_t bd = sdesc(us + ks * 2048, p.u_blk_bytes, 1024, 2);
                    umma_bf16(d, ad, bd, IDESC, ks > 0 ? 1u : 0u);
                }
                umma_bf16(d, sdesc(smem_u32(one_s), 128, 256, 0), sdesc(smem_u32(bt_s), 128, 256, 0), IDESC_BIAS,
                          1u);
                umma_commit(&hdr->empty[s]);
                umma_commit(&hdr->tmem_full[b]);
                mma_last = i;
            }
            __syncwarp();
        }
    } else if (((warp - kEpiWarp0) >> 2) < NCW) {
        // ---------------- epilogue: y = x + sum_k acc_k * x~_k (the bias is inside acc).  Each working
        // warp owns 32 tokens x CB/NCW channels of the tile and stores them itself (TMA, private double
        // buffer), so no warp ever waits for another one.
        const int q = warp & 3;                          // TMEM lane quadrant
        const int h = (warp - kEpiWarp0) >> 2;           // which share of the channel groups
        const int row = q * 32 + lane;                   // token within the tile
        uint8_t *ywarp = y_s + (warp - kEpiWarp0) * (2 * 32 * YB);
        int i = 0;
        int s = 0;
        uint32_t ph = 0;
        int nb = u_begin / p.n_mt, mt = u_begin - nb * p.n_mt;
        for (int v = u_begin; v < u_end;
             ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0), mt = (mt + 1 == p.n_mt) ? 0 : mt + 1,
                 nb += (mt == 0)) {
            const int b = i & 1;
            const uint32_t tph = (i >> 1) & 1;
            bool ok = mbar_wait(&hdr->tmem_full[b], tph, p.wait_ns) && mbar_wait(&hdr->full[s], ph, p.wait_ns);
            // the other roles' failures reach this warp through the barriers it waits on
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    record_status(p.status, kStatusTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint8_t *st = stages + s * p.stage_bytes;
            const uint8_t *xs = st + p.x_off_in_stage;
            const int nv = reinterpret_cast<const int8_t *>(st + p.nv_off_in_stage)[row];  // valid taps of this token
            const bool full_taps = __all_sync(0xffffffffu, nv == W);  // no token of this warp near a document start
            uint8_t *ys = ywarp + b * (32 * YB);
            bool ys_free = false;  // this warp's store from two tiles ago has left buffer b
            const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * 256;
#pragma unroll
            for (int gi = 0; gi < GPW; ++gi) {
                const int g = h * GPW + gi;  // 8-channel group
                const uint4 o = lr_group_y<W, RB>(trow + g * 8 * W, xs, row, g, full_taps, nv);
                if (!ys_free) {
                    if (lane == 0) tma_store_wait_read<1>();
                    __syncwarp();
                    ys_free = true;
                }
                *reinterpret_cast<uint4 *>(ys + lane * YB + gi * 16) = o;
            }
            // accumulator and x tile read: hand them back; store this warp's y sub-tile
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&hdr->tmem_empty[b]);
                mbar_arrive(&hdr->empty[s]);
                const int t0 = mt * kM;
                tma_store_2d(&tm_y, ys, nb * CB + h * (CB / NCW), t0 + q * 32);
                tma_store_commit();
            }
        }
    }
    // ---- teardown: no copy or MMA of this CTA may still be in flight
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (int s = 0; s < p.nstages; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / p.nstages) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_last >= 0)
        (void)mbar_wait(&hdr->tmem_full[mma_last & 1], (mma_last >> 1) & 1, kDrainLimitNs);
    if (warp == 1 && lane == 0 && u_pending) (void)mbar_wait(&hdr->u_full, (seg - 1) & 1, kDrainLimitNs);
    if (warp >= kEpiWarp0 && lane == 0) tma_store_wait_all<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

template <int W, int CB>
static dsc_status launch_lowrank_fwd(const LowrankArgs &a, const DeviceInfo &dev)
{
    using namespace lrf;
    constexpr int NB = CB * W, RB = CB * 2, XR = kM + W - 1;
    constexpr int NCW = CB / 8 < 4 ? CB / 8 : 4;
    Params p{};
    p.U = static_cast<const __nv_bfloat16 *>(a.U);
    p.bias = a.bias;
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.R = a.R;
    p.N = a.D * a.W;
    p.n_nb = (a.D + CB - 1) / CB;
    p.n_mt = (p.BT + kM - 1) / kM;
    const long long units = static_cast<long long>(p.n_nb) * p.n_mt;
    if (units > 0x7fffffffLL) return DSC_ERR_UNSUPPORTED;
    p.n_units = static_cast<int>(units);
    p.ksteps = (a.R + 15) / 16;
    p.kchunks = (a.R + 63) / 64;
    // shared memory: [header 1 KB][align slack 1 KB][U][bias tile][ones tile][y staging x2][stages]
    unsigned off = 0;
    p.u_off = off;
    p.u_blk_bytes = p.ksteps * 16 * 128;  // rows R rounded up to 16 (TMA fills the rest with zeros)
    p.u_bytes = ((NB + 63) / 64) * p.u_blk_bytes;
    off += p.u_bytes;
    p.bt_off = align_up(off, 1024);
    off = p.bt_off + NB * 32;
    p.one_off = align_up(off, 1024);
    off = p.one_off + kM * 32;
    p.y_off = align_up(off, 1024);
    off = p.y_off + kEpiWarps * 2 * 32 * (RB / NCW);
    p.st_off = align_up(off, 1024);
    p.z_bytes = p.kchunks * 16384;
    p.x_off_in_stage = p.z_bytes;
    p.x_bytes = XR * RB;
    p.nv_off_in_stage = align_up(p.x_off_in_stage + p.x_bytes, 128);
    p.stage_bytes = align_up(p.nv_off_in_stage + kM, 1024);
    const unsigned fixed = 2048 + p.st_off;
    // ranks above 128 leave room for one stage at their channel block (loads then wait for the tile before)
    if (static_cast<unsigned>(dev.max_smem_optin) < fixed + (a.R > 128 ? 1 : 2) * p.stage_bytes)
        return DSC_ERR_UNSUPPORTED;
    int ns = static_cast<int>((dev.max_smem_optin - fixed) / p.stage_bytes);
    p.nstages = ns > kMaxStages ? kMaxStages : ns;
    const unsigned smem = fixed + p.nstages * p.stage_bytes;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    CUtensorMap tm_z, tm_x, tm_y, tm_u;
    const CUtensorMapSwizzle sw = swizzle_for(RB);  // 128, 64 or 32 bytes: the x tile's row width
    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    if (!encode_tmap_2d(&tm_z, a.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.R, BT, static_cast<unsigned long long>(a.R) * 2,
                        64, kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB, XR, sw) ||
        !encode_tmap_2d(&tm_y, a.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB / NCW, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&tm_u, a.U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.N, a.R, static_cast<unsigned long long>(p.N) * 2,
                        64, p.ksteps * 16, CU_TENSOR_MAP_SWIZZLE_128B))
        return DSC_ERR_CUDA;
    auto kern = lowrank_fwd_tc<W, CB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    int grid = dev.sm_count < p.n_units ? dev.sm_count : p.n_units;
    return launch_overlapped(kern, grid, kThreads, smem, a.stream, tm_z, tm_x, tm_y, tm_u, p);
}

dsc_status lowrank_fwd(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R > 256) return DSC_ERR_UNSUPPORTED;
    if (a.R > 128) {
        // the block's U holds R rows: narrower channel blocks keep it resident beside a stage
        switch (a.W) {
        case 1: return launch_lowrank_fwd<1, 32>(a, dev);
        case 2: return launch_lowrank_fwd<2, 32>(a, dev);
        case 3: return launch_lowrank_fwd<3, 32>(a, dev);
        case 4: return launch_lowrank_fwd<4, 32>(a, dev);
        case 5: return launch_lowrank_fwd<5, 32>(a, dev);
        case 6: return launch_lowrank_fwd<6, 32>(a, dev);
        case 7: return launch_lowrank_fwd<7, 16>(a, dev);
        case 8: return launch_lowrank_fwd<8, 16>(a, dev);
        default: return DSC_ERR_INVALID_ARG;
        }
    }
    switch (a.W) {
    case 1: return launch_lowrank_fwd<1, 64>(a, dev);
    case 2: return launch_lowrank_fwd<2, 64>(a, dev);
    case 3: return launch_lowrank_fwd<3, 64>(a, dev);
    case 4: return launch_lowrank_fwd<4, 64>(a, dev);
    case 5: return launch_lowrank_fwd<5, 32>(a, dev);
    case 6: return launch_lowrank_fwd<6, 32>(a, dev);
    case 7: return launch_lowrank_fwd<7, 32>(a, dev);
    case 8: return launch_lowrank_fwd<8, 32>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

}  // namespace dsc
