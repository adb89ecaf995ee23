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
// U block (transposed into a K-major, 128-byte-swizzled tile) stays resident
// in shared memory while the CTA streams over token tiles.
//   warp 0      TMA producer: z tile (K-major, swizzled) and the x tile with
//               its (W-1)-token causal halo; per-token valid-tap counts
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=NB, K=16 per
//               instruction) into one of two TMEM accumulators
//   warps 2..17 epilogue: tcgen05.ld of the accumulator row of one token,
//               + bias, times the x window from shared memory, + residual,
//               bf16 into a swizzled staging tile that one thread TMA-stores
// Inside each group of 8 channels the filter columns are kept tap-major
// (MMA column g*8W + k*8 + c for channel g*8+c, tap k): the 8 channels of one
// tap are adjacent accumulator columns, so channel pairs feed packed fp32x2
// math straight from TMEM registers.
#include "dsc_internal.h"
#include "dsc_tcgen05.cuh"

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
    int ksteps, kchunks;           // MMA K steps of 16; 64-wide K chunks
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
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace lrf

// Byte offset of 16-byte chunk `c` of row `row` in a swizzled tile whose rows are RB bytes (128 or 64).
template <int RB>
__device__ __forceinline__ uint32_t swz(int row, int c)
{
    if constexpr (RB == 128) return row * 128 + ((c ^ (row & 7)) << 4);
    else return row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
}

template <int W, int CB>
__global__ void __launch_bounds__(lrf::kThreads, 1)
    lowrank_fwd_tc(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_y, const lrf::Params p)
{
    using namespace lrf;
    constexpr int NB = CB * W;         // filter columns per block (MMA N)
    constexpr int RB = CB * 2;         // bytes per x / y tile row
    constexpr int GROUPS = CB / 8;     // 8-channel groups per block
    constexpr int GPW = GROUPS / 4;    // groups per epilogue warp (four warps per lane quadrant)
    static_assert(NB % 16 == 0 && NB <= 256, "MMA N");
    constexpr uint32_t IDESC = idesc_bf16_f32(kM, NB);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *u_s = base + p.u_off;       // [kchunks][NB rows][128 B], 128-B swizzled, K-major
    uint8_t *bt_s = base + p.bt_off;     // bias as an MMA B tile: [NB rows][16 K], no swizzle
    uint8_t *one_s = base + p.one_off;   // all-ones MMA A tile [128 rows][16 K]
    uint8_t *y_s = base + p.y_off;       // per epilogue warp: 2 x [32 rows][RB/4] staging for its own stores
    uint8_t *stages = base + p.st_off;

    // block column n = (g*8 + c)*W + k  ->  MMA column g*8W + k*8 + c (tap-major inside a group)
    auto tap_major = [](int n) {
        const int g = n / (8 * W), rem = n - g * (8 * W);
        return g * (8 * W) + (rem % W) * 8 + rem / W;
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1 + kEpiWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->tmem_full[b], 1);
            mbar_init(&hdr->tmem_empty[b], kEpiWarps);
        }
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kM * 16 / 2; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    if (warp == 1) {
        tmem_alloc(&hdr->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = hdr->tmem_base;
    volatile int *abort_flag = &hdr->abort_flag;

    const int u_begin = static_cast<int>(static_cast<long long>(blockIdx.x) * p.n_units / gridDim.x);
    const int u_end = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.n_units / gridDim.x);

    int it = 0;             // tiles through the stage ring (all roles count the same)
    int issued_last[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
    int mma_last = -1;      // last tile whose MMAs were committed (MMA thread)

    for (int u = u_begin; u < u_end;) {
        const int nb = u / p.n_mt;
        const int seg_end = min(u_end, (nb + 1) * p.n_mt);

        // ---- the block's filter generator: U[:, nb*NB .. +NB) transposed to K-major, and the bias
        //      as an extra K step (exact bf16 hi + lo pair) that the all-ones A tile adds in
        {
            const int nK = p.kchunks * 64;
            const int items = nK * (NB / 8);
            for (int idx = threadIdx.x; idx < items; idx += blockDim.x) {
                const int n8 = idx / nK, r = idx - n8 * nK;
                const int n = n8 * 8, gn = nb * NB + n;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < p.R && gn < p.N) v = *reinterpret_cast<const uint4 *>(p.U + static_cast<size_t>(r) * p.N + gn);
                const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
                const int a = r >> 6, c = (r & 63) >> 3, o = (r & 7) * 2;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int row = tap_major(n + j);  // MMA column of block column n+j
                    *reinterpret_cast<uint16_t *>(u_s + a * (NB * 128) + row * 128 + ((c ^ (row & 7)) << 4) + o) = e[j];
                }
            }
            for (int n = threadIdx.x; n < NB; n += blockDim.x) {
                const int gn = nb * NB + n;
                const float bv = gn < p.N ? p.bias[gn] : 0.f;
                const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv)));
                const uint32_t lo =
                    static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv - __uint_as_float(hi << 16))));
                const int row = tap_major(n);
                // core matrices of 8 rows x 16 B: K-half 0 at ((row/8)*2)*128, K-half 1 next to it
                uint8_t *cm = bt_s + ((row >> 3) * 2) * 128 + (row & 7) * 16;
                *reinterpret_cast<uint4 *>(cm) = make_uint4(hi | (lo << 16), 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(cm + 128) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();

        if (warp == 0) {
            // ---------------- producer
            int i = it;
            int s = it % p.nstages;                     // stage and its phase: stepped, not divided, per tile
            uint32_t ph = (it / p.nstages) & 1;
            for (int v = u; v < seg_end; ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0)) {
                bool ok = mbar_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (!ok) {
                    if (lane == 0) {
                        record_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                    }
                    break;
                }
                const int mt = v - nb * p.n_mt;
                const int t0 = mt * kM;
                uint8_t *st = stages + s * p.stage_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&hdr->full[s], p.z_bytes + p.x_bytes);
                    for (int a = 0; a < p.kchunks; ++a) tma_load_2d(st + a * 16384, &tm_z, &hdr->full[s], a * 64, t0);
                    tma_load_2d(st + p.x_off_in_stage, &tm_x, &hdr->full[s], nb * CB, t0 - (W - 1));
                    issued_last[s] = i;
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer: acc = z . U_blk (K = R), then += 1 . bias
            int i = it;
            int s = it % p.nstages;
            uint32_t ph = (it / p.nstages) & 1;
            for (int v = u; v < seg_end; ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0)) {
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
                        const int a = ks >> 2, kk = ks & 3;
                        const uint64_t ad = sdesc_kmajor_sw128(zs + a * 16384 + kk * 32);
                        const uint64_t bd = sdesc_kmajor_sw128(us + a * (NB * 128) + kk * 32);
                        umma_bf16(d, ad, bd, IDESC, ks > 0 ? 1u : 0u);
                    }
                    umma_bf16(d, sdesc(smem_u32(one_s), 128, 256, 0), sdesc(smem_u32(bt_s), 128, 256, 0), IDESC, 1u);
                    umma_commit(&hdr->empty[s]);
                    umma_commit(&hdr->tmem_full[b]);
                    mma_last = i;
                }
                __syncwarp();
            }
        } else {
            // ---------------- epilogue: y = x + sum_k acc_k * x~_k (the bias is inside acc).  Each warp
            // owns 32 tokens x CB/4 channels of the tile and stores them itself (TMA, private double
            // buffer), so no warp ever waits for another one.
            const int q = warp & 3;                          // TMEM lane quadrant
            const int h = (warp - kEpiWarp0) >> 2;           // which quarter of the channel groups
            const int row = q * 32 + lane;                   // token within the tile
            uint8_t *ywarp = y_s + (warp - kEpiWarp0) * (2 * 32 * (RB / 4));
            DocCursor cursor;  // this thread's token increases from tile to tile within a run
            int i = it;
            int s = it % p.nstages;
            uint32_t ph = (it / p.nstages) & 1;
            for (int v = u; v < seg_end; ++v, ++i, s = (s + 1 == p.nstages) ? 0 : s + 1, ph ^= (s == 0)) {
                const int b = i & 1;
                const uint32_t tph = (i >> 1) & 1;
                // valid taps of this token, worked out while the tile's accumulator is still being computed
                const int t = (v - nb * p.n_mt) * kM + row;
                const int nv = t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W;  // valid taps of this token
                const bool full_taps = __all_sync(0xffffffffu, nv == W);  // no token of this warp near a document start
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
                uint8_t *ys = ywarp + b * (32 * (RB / 4));
                bool ys_free = false;  // this warp's store from two tiles ago has left buffer b
                const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * 256;
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = h * GPW + gi;  // 8-channel group
                    uint32_t acc[8 * W];         // acc[k*8 + c]: tap k of channel g*8 + c
                    tmem_ld_cols<8 * W>(trow + g * 8 * W, acc);
                    float2 out[4];
                    {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(xs + swz<RB>(row + W - 1, g));
                        out[0] = bf16x2_to_f2(raw.x);  // residual: x of the token itself
                        out[1] = bf16x2_to_f2(raw.y);
                        out[2] = bf16x2_to_f2(raw.z);
                        out[3] = bf16x2_to_f2(raw.w);
                    }
                    const float2 x0[4] = {out[0], out[1], out[2], out[3]};
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < W; ++k) {
                        float2 xk[4];
                        if (k == 0) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) xk[e] = x0[e];
                        } else {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(xs + swz<RB>(row + (W - 1) - k, g));
                            xk[0] = bf16x2_to_f2(raw.x);
                            xk[1] = bf16x2_to_f2(raw.y);
                            xk[2] = bf16x2_to_f2(raw.z);
                            xk[3] = bf16x2_to_f2(raw.w);
                            if (!full_taps && k >= nv) {  // x~ is zero before the document start
#pragma unroll
                                for (int e = 0; e < 4; ++e) xk[e] = make_float2(0.f, 0.f);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            out[e] = fma2(make_float2(__uint_as_float(acc[k * 8 + 2 * e]),
                                                      __uint_as_float(acc[k * 8 + 2 * e + 1])),
                                          xk[e], out[e]);
                    }
                    uint4 o;
                    __nv_bfloat162 h0 = __float22bfloat162_rn(out[0]), h1 = __float22bfloat162_rn(out[1]);
                    __nv_bfloat162 h2 = __float22bfloat162_rn(out[2]), h3 = __float22bfloat162_rn(out[3]);
                    o.x = *reinterpret_cast<uint32_t *>(&h0);
                    o.y = *reinterpret_cast<uint32_t *>(&h1);
                    o.z = *reinterpret_cast<uint32_t *>(&h2);
                    o.w = *reinterpret_cast<uint32_t *>(&h3);
                    if (!ys_free) {
                        if (lane == 0) tma_store_wait_read<1>();
                        __syncwarp();
                        ys_free = true;
                    }
                    *reinterpret_cast<uint4 *>(ys + lane * (RB / 4) + gi * 16) = o;
                }
                // accumulator and x tile read: hand them back; store this warp's y sub-tile
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&hdr->tmem_empty[b]);
                    mbar_arrive(&hdr->empty[s]);
                    const int t0 = (v - nb * p.n_mt) * kM;
                    tma_store_2d(&tm_y, ys, nb * CB + h * (CB / 4), t0 + q * 32);
                    tma_store_commit();
                }
            }
        }
        it += seg_end - u;
        u = seg_end;
        __syncthreads();
        if (*abort_flag) break;
    }

    // ---- teardown: no copy or MMA of this CTA may still be in flight
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (int s = 0; s < p.nstages; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / p.nstages) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_last >= 0)
        (void)mbar_wait(&hdr->tmem_full[mma_last & 1], (mma_last >> 1) & 1, kDrainLimitNs);
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
    off += p.kchunks * NB * 128;
    p.bt_off = align_up(off, 1024);
    off = p.bt_off + NB * 32;
    p.one_off = align_up(off, 1024);
    off = p.one_off + kM * 32;
    p.y_off = align_up(off, 1024);
    off = p.y_off + kEpiWarps * 2 * 32 * (RB / 4);
    p.st_off = align_up(off, 1024);
    p.z_bytes = p.kchunks * 16384;
    p.x_off_in_stage = p.z_bytes;
    p.x_bytes = XR * RB;
    p.nv_off_in_stage = align_up(p.x_off_in_stage + p.x_bytes, 128);
    p.stage_bytes = align_up(p.nv_off_in_stage + kM, 1024);
    const unsigned fixed = 2048 + p.st_off;
    if (static_cast<unsigned>(dev.max_smem_optin) < fixed + 2 * p.stage_bytes) return DSC_ERR_UNSUPPORTED;
    int ns = static_cast<int>((dev.max_smem_optin - fixed) / p.stage_bytes);
    p.nstages = ns > kMaxStages ? kMaxStages : ns;
    const unsigned smem = fixed + p.nstages * p.stage_bytes;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    CUtensorMap tm_z, tm_x, tm_y;
    const CUtensorMapSwizzle sw = RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    if (!encode_tmap_2d(&tm_z, a.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.R, BT, static_cast<unsigned long long>(a.R) * 2,
                        64, kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB, XR, sw) ||
        !encode_tmap_2d(&tm_y, a.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, static_cast<unsigned long long>(a.D) * 2,
                        CB / 4, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_CUDA;
    auto kern = lowrank_fwd_tc<W, CB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    int grid = dev.sm_count < p.n_units ? dev.sm_count : p.n_units;
    kern<<<grid, kThreads, smem, a.stream>>>(tm_z, tm_x, tm_y, p);
    return launched();
}

dsc_status lowrank_fwd(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
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
