// dsc_lowrank_bwd.cu -- backward pass of the low-rank fused dynamic short
// convolution (the derivative of eq. 2 + eq. 3 with w = zU + b, notes on
// "Dynamic Short Convolutions Improve Transformers", "Parameterization"):
//
//   Wt[t, n]  = sum_r z[t,r] U[r,n] + b[n]              recomputed on chip, n = d*W + k
//   dx[s,d]   = dy[s,d] + sum_k [s in doc(s+k)] Wt[s+k, d*W+k] dy[s+k,d]
//   G[t, n]   = dy[t,d] * x~[t-k,d]                     gradient of the generated filter
//   dz[t,r]   = sum_n G[t,n] U[r,n]     dU[r,n] = sum_t z[t,r] G[t,n]     db[n] = sum_t G[t,n]
//
// Two kernels, split by the axis each gradient sums over:
//   lowrank_bwd_dxdz (this file)   dx and dz: a CTA owns a tile of tokens and walks
//                                  every channel, so dz (a sum over all D*W filter
//                                  columns) accumulates in TMEM and is written once
//   lowrank_bwd_dudb (dsc_lowrank_bwd_du.cu)   dU and db: a CTA owns a block of filter
//                                  columns and walks the tokens
// Neither needs a workspace or a reduction across CTAs for dz; dU and db take a
// few fp32 additions per element (one per CTA whose token run covers a block).
//
// lowrank_bwd_dxdz.  Tile: 128 TMEM lanes in four quadrants of 32; quadrant q
// holds tokens t0 + q*QS + i (i < 32), QS = 33 - W, so every token a quadrant
// owns (i < QS) finds the W-1 later tokens its dx needs inside its own warp:
// the tap-k terms move by warp shuffles, with no exchange between warps.  Per
// step of SCB channels (SNB = SCB*W filter columns):
//   MMA   Wt_step = z . U_step + 1 . b_step                (A z K-major; B U MN-major)   -> TMEM
//   epi   dx (shuffles), and G = dy * x~ as an exact bf16 hi + lo pair (packed
//         bf16 multiply and fused multiply-add), written to shared memory
//   MMA   dz += G_hi . U_step^T + G_lo . U_step^T           (A G K-major; B U K-major)    -> TMEM
// Warps: a TMA producer, one warp issuing the filter MMAs, one issuing the dz
// MMAs, and 16 epilogue warps.  The filter accumulator is double-buffered, so
// the filter of step k+1 is computed while the epilogue works on step k, and
// the dz MMAs of a step run while the epilogue works on the next one.  Each
// epilogue warp stores its own dx sub-tile by TMA.
#include "dsc_internal.h"
#include "dsc_lowrank_common.cuh"

namespace dsc {

namespace lrx {

constexpr int kM = 128;
constexpr int kEpiWarps = 16;
constexpr int kEpiWarp0 = 3;  // warps 0, 1, 2: producer, filter MMAs, dz MMAs
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kMaxStages = 6;
constexpr int kTmemCols = 512;
constexpr int kColDz = 256;  // dz accumulator (<= 256 columns); two filter accumulators below it

struct Params {
    const float *bias;
    const int32_t *cu;
    int n_docs;
    __nv_bfloat16 *dz;
    __nv_bfloat16 *dx;
    const uint4 *bias_rows;  // per filter column its bias as an exact bf16 hi + lo pair, 16 bytes a column
    int BT, T, D, R, R16, N;
    int n_tiles, n_steps, kchunks, ksteps;
    unsigned z_bytes, one_off, bz_off, g_off, st_off, stage_bytes, bt_in, x_in, dy_in, u_blk_bytes, stage_tx;
    int nstages, nzbuf;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t z_full[2], z_empty[2];
    uint64_t f_full[2], f_empty[2];
    uint64_t g_full, g_empty;
    uint64_t dz_full, dz_empty;
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace lrx

template <int W, int SCB>
__global__ void __launch_bounds__(lrx::kThreads, 1)
    lowrank_bwd_dxdz(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_u,
                     const lrx::Params p)
{
    using namespace lrx;
    constexpr int SNB = SCB * W;                 // filter columns per step
    constexpr int SNBP = (SNB + 15) / 16 * 16;   // MMA N of the recompute, K of dz
    constexpr int RB = SCB * 2;                  // bytes per x / dy row
    constexpr int GPS = SCB / 8;                 // 8-channel groups per step
    constexpr int NCW = GPS < 4 ? GPS : 4;       // column warps with work (per lane quadrant)
    constexpr int GPW = GPS / NCW;               // groups per working warp
    constexpr int QS = 33 - W;                   // tokens owned per lane quadrant
    constexpr int MS = 4 * QS;                   // tokens owned per tile
    constexpr int UB = (SNBP + 63) / 64;         // 64-column blocks of U per step
    static_assert(SNBP <= 128 && GPS % NCW == 0, "step shape");
    constexpr uint32_t ID_RC = idesc_bf16_f32(kM, SNBP, false, true);    // A z K-major, B U MN-major
    constexpr uint32_t ID_BIAS = idesc_bf16_f32(kM, SNBP, false, false);  // A ones, B bias tile

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *z_s = base;                  // [nzbuf][kchunks][128 rows][128 B]
    uint8_t *one_s = base + p.one_off;    // all-ones A tile [128 rows][16 K]
    uint8_t *g_s = base + p.g_off;        // G [hi, lo][UB blocks][128 rows][128 B], 128-byte swizzled, K-major
    uint8_t *stages = base + p.st_off;    // [U blocks][bias rows][x][dy] per stage
    uint8_t *bz_s = base + p.bz_off;      // the zero K half of every bias tile [SNBP rows][16 B], above the stages

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1 + 4 * NCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->z_full[b], 1);
            mbar_init(&hdr->z_empty[b], 1);
            mbar_init(&hdr->f_full[b], 1);
            mbar_init(&hdr->f_empty[b], 4 * NCW);
            mbar_init(&hdr->drain[b], 1);
        }
        mbar_init(&hdr->g_full, 4 * NCW);
        mbar_init(&hdr->g_empty, 1);
        mbar_init(&hdr->dz_full, 1);
        mbar_init(&hdr->dz_empty, kEpiWarps);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kM * 16 / 2; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    // the bias MMA's B tile: K half 0 (the bias rows) arrives with each stage, K half 1 is this shared zero block
    for (int i = threadIdx.x; i < SNBP; i += blockDim.x) reinterpret_cast<uint4 *>(bz_s)[i] = make_uint4(0u, 0u, 0u, 0u);
    // G: the columns past the step's filter columns (MMA K padding) stay zero
    for (int i = threadIdx.x; i < 2 * UB * 1024; i += blockDim.x) reinterpret_cast<uint4 *>(g_s)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(&hdr->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // everything before this line may overlap the previous kernel; every global access comes after it.  The
    // dependent kernel (dU, db) may launch once this one runs: its own inputs are ready by now.
    grid_dependency_wait();
    grid_dependents_launch();
    const uint32_t tmem = hdr->tmem_base;
    volatile int *abort_flag = &hdr->abort_flag;
    const int n_local = p.n_tiles > static_cast<int>(blockIdx.x)
                            ? (p.n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                            : 0;
    const int k_total = n_local * p.n_steps;

    int issued_last[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
    int z_issued = -1;
    bool mma_any = false;

    if (warp == 0) {
        // ---------------- producer: z tile per token tile (four 32-row boxes, one per lane quadrant); per
        // step the U columns, the bias pairs, x (with the causal halo) and dy
        int k = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int ti = 0; ti < n_local && ok; ++ti) {
            const int t0 = (static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x)) * MS;
            const int zb = ti % p.nzbuf;
            if (ti >= p.nzbuf) ok = warp_wait(&hdr->z_empty[zb], ((ti / p.nzbuf) - 1) & 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (lane == 0) {
                uint8_t *zt = z_s + zb * p.z_bytes;
                mbar_arrive_expect_tx(&hdr->z_full[zb], p.z_bytes);
                for (int a = 0; a < p.kchunks; ++a)
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d(zt + a * 16384 + q * 4096, &tm_z, &hdr->z_full[zb], a * 64, t0 + q * QS);
                z_issued = ti;
            }
            for (int j = 0; j < p.n_steps; ++j, ++k) {
                if (k >= p.nstages) ok = warp_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                uint8_t *st = stages + s * p.stage_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&hdr->full[s], p.stage_tx);
#pragma unroll
                    for (int b = 0; b < UB; ++b)
                        tma_load_2d(st + b * p.u_blk_bytes, &tm_u, &hdr->full[s], j * SNB + b * 64, 0);
                    tma_load_2d(st + p.x_in, &tm_x, &hdr->full[s], j * SCB, t0 - (W - 1));
                    tma_load_2d(st + p.dy_in, &tm_dy, &hdr->full[s], j * SCB, t0);
                    bulk_load(st + p.bt_in, p.bias_rows + j * SNB, SNBP * 16, &hdr->full[s]);
                    issued_last[s] = k;
                }
                if (++s == p.nstages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- filter MMAs: step k into accumulator k & 1, once the epilogue has loaded step k-2's
        // filter from it.  Shared-memory descriptors are built once; a stage or K step adds (byte offset >> 4) to
        // the start-address field (bits 0-13), which never carries: shared addresses stay below 256 KB.
        const uint32_t st0 = smem_u32(stages);
        const uint64_t d_one = sdesc(smem_u32(one_s), 128, 256, 0);
        const uint64_t d_z0 = sdesc_kmajor_sw128(smem_u32(z_s));             // z, K-major (A)
        const uint64_t d_u0 = sdesc(st0, p.u_blk_bytes, 1024, 2);             // U step, MN-major (B)
        // bias tile (B of the last K step): rows of 16 B (8-row core matrices 128 B apart); its second K half is
        // the shared zero block, LBO bytes away (the LBO shrinks by a stage's size for every stage further up)
        const uint32_t bt0 = st0 + p.bt_in;
        const uint64_t d_bt0 = sdesc(bt0, smem_u32(bz_s) - bt0, 128, 0);
        const uint32_t stg16 = p.stage_bytes >> 4, z16 = p.z_bytes >> 4;
        const int ksteps = p.ksteps;
        int ti = 0, j = 0, s = 0, zb = 0;
        uint32_t ph = 0, zph = 0;
        bool ok = true;
        for (int k = 0; k < k_total; ++k) {
            const int fb = k & 1;
            bool w = warp_wait(&hdr->full[s], ph, p.wait_ns);
            if (j == 0) w = warp_wait(&hdr->z_full[zb], zph, p.wait_ns) && w;
            if (k >= 2) w = warp_wait(&hdr->f_empty[fb], ((k >> 1) & 1) ^ 1, p.wait_ns) && w;
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t so = static_cast<uint32_t>(s) * stg16;
                const uint64_t az = d_z0 + static_cast<uint32_t>(zb) * z16, bu = d_u0 + so;
                const uint32_t d = tmem + fb * 128;
                umma_bf16_nc(d, az, bu, ID_RC, 0u);
                for (int ks = 1; ks < ksteps; ++ks)  // K = R in steps of 16: 32 B into z's 128-B rows, 16 rows of U
                    umma_bf16_nc(d, az + (ks >> 2) * 1024 + (ks & 3) * 2, bu + 128 * ks, ID_RC, 1u);
                umma_bf16_nc(d, d_one, d_bt0 + so - (static_cast<uint64_t>(so) << 16), ID_BIAS, 1u);
                umma_commit(&hdr->f_full[fb]);
                if (j == p.n_steps - 1) umma_commit(&hdr->z_empty[zb]);
            }
            __syncwarp();
            mma_any = true;
            if (++j == p.n_steps) {
                j = 0;
                ++ti;
                if (++zb == p.nzbuf) {
                    zb = 0;
                    zph ^= 1;
                }
            }
            if (++s == p.nstages) {
                s = 0;
                ph ^= 1;
            }
        }
        if (lane == 0 && mma_any) umma_commit(&hdr->drain[0]);
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    } else if (warp == 2) {
        // ---------------- dz MMAs: step k once its G is in shared memory
        const uint32_t st0 = smem_u32(stages);
        const uint32_t ID_DZ = idesc_bf16_f32(kM, p.R16, false, false);
        const uint64_t d_uk0 = sdesc(st0, 16, 1024, 2);                       // U step, K-major (B)
        const uint64_t d_g = sdesc_kmajor_sw128(smem_u32(g_s));              // G hi, then lo (A)
        const uint32_t ublk16 = p.u_blk_bytes >> 4, stg16 = p.stage_bytes >> 4;
        int ti = 0, j = 0, s = 0;
        bool ok = true;
        for (int k = 0; k < k_total; ++k) {
            bool w = warp_wait(&hdr->g_full, k & 1, p.wait_ns);
            if (j == 0 && ti >= 1) w = warp_wait(&hdr->dz_empty, (ti - 1) & 1, p.wait_ns) && w;
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t b0 = d_uk0 + static_cast<uint32_t>(s) * stg16, b1 = b0 + ublk16;
                const uint32_t dzt = tmem + kColDz;
#pragma unroll
                for (int part = 0; part < 2; ++part)  // G = hi + lo
#pragma unroll
                    for (int kk = 0; kk < SNBP / 16; ++kk)  // K over the step's columns: 32 B into 128-B rows
                        umma_bf16_nc(dzt, d_g + (part * UB + (kk >> 2)) * 1024 + (kk & 3) * 2,
                                     ((kk >> 2) ? b1 : b0) + (kk & 3) * 2, ID_DZ,
                                     (part == 0 && kk == 0) ? (j > 0 ? 1u : 0u) : 1u);
                umma_commit(&hdr->g_empty);
                umma_commit(&hdr->empty[s]);
                if (j == p.n_steps - 1) umma_commit(&hdr->dz_full);
            }
            __syncwarp();
            mma_any = true;
            if (++j == p.n_steps) {
                j = 0;
                ++ti;
            }
            if (++s == p.nstages) s = 0;
        }
        if (lane == 0 && mma_any) umma_commit(&hdr->drain[1]);
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    } else {
        // ---------------- epilogue: 16 warps; lane quadrant q, column warp cw
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3, cw = ew >> 2;
        const bool active = cw < NCW;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        DocCursor cursor;
        bool ok = true;
        int k = 0, s = 0;
        uint32_t ph = 0;
        for (int ti = 0; ti < n_local && ok; ++ti) {
            const int t0 = (static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x)) * MS;
            const int yrow = q * QS + lane;  // this thread's row in the dy tile (x tile: + W - 1)
            const int row_tm = q * 32 + lane;  // its TMEM lane: the row of the filter and of G
            const int t = t0 + yrow;
            const bool owned = lane < QS && t < p.BT;
            const int nv = t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W;
            const bool full_taps = __all_sync(0xffffffffu, nv == W);  // no token of this warp near a document start
            // this thread's rows of the dy and x tiles: the same offsets in every stage of the tile
            uint32_t off_dy[GPW], off_x[GPW][W];
#pragma unroll
            for (int gi = 0; gi < GPW; ++gi) {
                off_dy[gi] = p.dy_in + swzt<RB>(yrow, cw * GPW + gi);
#pragma unroll
                for (int kk = 0; kk < W; ++kk) off_x[gi][kk] = p.x_in + swzt<RB>(yrow + (W - 1) - kk, cw * GPW + gi);
            }
            for (int j = 0; j < p.n_steps && ok; ++j, ++k) {
                const int cs = s;
                const uint32_t cph = ph;
                if (++s == p.nstages) {
                    s = 0;
                    ph ^= 1;
                }
                if (!active) continue;
                const int fb = k & 1;
                bool w = warp_wait(&hdr->f_full[fb], (k >> 1) & 1, p.wait_ns) && warp_wait(&hdr->full[cs], cph, p.wait_ns);
                if (!w) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *st = stages + cs * p.stage_bytes;
                uint32_t acc[GPW][8 * W];  // acc[gi][c*W + k]: tap k of channel c of group gi (bias included)
                uint4 dyv[GPW];
                uint4 xv[GPW][W];          // x~ rows t-k of the group's 8 channels
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = cw * GPW + gi;
                    tmem_ld_cols<8 * W>(lane_base + fb * 128 + g * 8 * W, acc[gi]);
                    dyv[gi] = lds128(st + off_dy[gi]);
#pragma unroll
                    for (int kk = 0; kk < W; ++kk) xv[gi][kk] = lds128(st + off_x[gi][kk]);
                }
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->f_empty[fb]);  // the filter of step k+2 may be computed here
                if (!full_taps) {
                    // near a document start (warp-uniform branch): x~ before the start is zero, and so is the
                    // tap-k term this token passes back to token t-k in another document
#pragma unroll
                    for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
                        for (int kk = 1; kk < W; ++kk)
                            if (kk >= nv) {
                                xv[gi][kk] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                                for (int c = 0; c < 8; ++c) acc[gi][c * W + kk] = 0u;
                            }
                }
                uint32_t ghi[GPW][4 * W], glo[GPW][4 * W];
                uint4 dxo[GPW];
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    // G: column pair (f, f+1) of the group's 8W columns f = c*W + k, as exact bf16 hi + lo
#pragma unroll
                    for (int pr = 0; pr < 4 * W; ++pr) {
                        const int f = 2 * pr;
                        const int c0 = f / W, k0 = f % W, c1 = (f + 1) / W, k1 = (f + 1) % W;
                        const uint32_t sel = half_sel(c0 & 1, c1 & 1);
                        const uint32_t d2 = __byte_perm(word_of(dyv[gi], c0 >> 1), word_of(dyv[gi], c1 >> 1), sel);
                        const uint32_t x2 = __byte_perm(word_of(xv[gi][k0], c0 >> 1), word_of(xv[gi][k1], c1 >> 1), sel);
                        exact_product_split(d2, x2, ghi[gi][pr], glo[gi][pr]);
                    }
                    // dx: residual + own tap-0 term, then the tap-k terms of the tokens k ahead (lanes + k)
                    float gy[8], dxv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t wv = word_of(dyv[gi], e);
                        gy[2 * e] = __uint_as_float(wv << 16);
                        gy[2 * e + 1] = __uint_as_float(wv & 0xffff0000u);
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) dxv[c] = fmaf(__uint_as_float(acc[gi][c * W]), gy[c], gy[c]);
#pragma unroll
                    for (int kk = 1; kk < W; ++kk)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            dxv[c] += __shfl_down_sync(0xffffffffu, __uint_as_float(acc[gi][c * W + kk]) * gy[c], kk);
                    dxo[gi] = make_uint4(pack_bf16x2(dxv[0], dxv[1]), pack_bf16x2(dxv[2], dxv[3]),
                                         pack_bf16x2(dxv[4], dxv[5]), pack_bf16x2(dxv[6], dxv[7]));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->empty[cs]);  // x and dy of the stage are read
                // G into shared memory, once the dz MMAs of the previous step have read it
                if (k >= 1 && !warp_wait(&hdr->g_empty, (k - 1) & 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = cw * GPW + gi;
#pragma unroll
                    for (int m = 0; m < W; ++m) {  // 16-byte chunk m (8 columns) of the group's 8W columns
                        const int n = g * 8 * W + m * 8;
                        const uint32_t off = (n >> 6) * 16384 + swzt<128>(row_tm, (n & 63) >> 3);
                        *reinterpret_cast<uint4 *>(g_s + off) =
                            make_uint4(ghi[gi][4 * m], ghi[gi][4 * m + 1], ghi[gi][4 * m + 2], ghi[gi][4 * m + 3]);
                        *reinterpret_cast<uint4 *>(g_s + UB * 16384 + off) =
                            make_uint4(glo[gi][4 * m], glo[gi][4 * m + 1], glo[gi][4 * m + 2], glo[gi][4 * m + 3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->g_full);
                // dx: 16 bytes (8 channels) per owned token and group, straight from registers
                if (owned) {
#pragma unroll
                    for (int gi = 0; gi < GPW; ++gi) {
                        const int ch = j * SCB + (cw * GPW + gi) * 8;
                        if (ch < p.D) *reinterpret_cast<uint4 *>(p.dx + static_cast<size_t>(t) * p.D + ch) = dxo[gi];
                    }
                }
            }
            if (!ok) break;
            // the tile's dz: every warp reads R16/4 of its columns
            bool w = warp_wait(&hdr->dz_full, ti & 1, p.wait_ns);
            w = __all_sync(0xffffffffu, w);
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int r4 = p.R16 >> 2;
            for (int c = 0; c < r4; c += 4) {
                uint32_t a4[4];
                tmem_ld_x4(lane_base + kColDz + cw * r4 + c, a4);
                tmem_ld_wait();
                const int col = cw * r4 + c;
                if (owned && col < p.R) {
                    const uint2 o = make_uint2(pack_bf16x2(__uint_as_float(a4[0]), __uint_as_float(a4[1])),
                                               pack_bf16x2(__uint_as_float(a4[2]), __uint_as_float(a4[3])));
                    *reinterpret_cast<uint2 *>(p.dz + static_cast<size_t>(t) * p.R + col) = o;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdr->dz_empty);
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    }

    // ---- teardown: nothing of this CTA may still be in flight
    if (warp == 0 && lane == 0) {  // every copy issued has landed (at once, unless the CTA gave up early)
        for (int s = 0; s < p.nstages; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait_ev(&hdr->full[s], (issued_last[s] / p.nstages) & 1, kDrainLimitNs);
        if (z_issued >= 0)
            (void)mbar_wait_ev(&hdr->z_full[z_issued % p.nzbuf], (z_issued / p.nzbuf) & 1, kDrainLimitNs);
    }
    if ((warp == 1 || warp == 2) && lane == 0 && mma_any) (void)mbar_wait_ev(&hdr->drain[warp - 1], 0, kDrainLimitNs);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

// Per filter column n its bias as an exact bf16 hi + lo pair in the first 4 bytes of a 16-byte row (the
// dx / dz kernel copies a step's rows into the B tile of the MMA that adds the bias); rows past N are zero.
// Also zeroes dU and db, which the dU / db kernel accumulates into.
__global__ void lowrank_bwd_prep(const float *bias, int N, uint4 *rows, int n_rows, float4 *dU, long long na4, float *db)
{
    grid_dependency_wait();  // the stream's previous kernel may still use dU, db or the workspace
    grid_dependents_launch();
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long i0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    for (long long i = i0; i < n_rows; i += stride) {
        const float bv = i < N ? bias[i] : 0.f;
        const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv)));
        const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv - __uint_as_float(hi << 16))));
        rows[i] = make_uint4(hi | (lo << 16), 0u, 0u, 0u);
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = i0; i < na4; i += stride) dU[i] = z4;
    for (long long i = i0; i < N; i += stride) db[i] = 0.f;
}

// Rows of the bias workspace: every filter column, plus room for the last step's padded tile.
static long long bias_rows(int D, int W) { return static_cast<long long>(D) * W + 256; }

size_t lowrank_bwd_workspace(int B, int T, int D, int W, int R)
{
    (void)B;
    (void)T;
    (void)R;
    const size_t bytes = static_cast<size_t>(bias_rows(D, W)) * 16;
    return (bytes + 255) / 256 * 256;
}

template <int W, int SCB>
static dsc_status launch_dxdz(const LowrankArgs &a, const DeviceInfo &dev)
{
    using namespace lrx;
    constexpr int SNB = SCB * W, SNBP = (SNB + 15) / 16 * 16, RB = SCB * 2, QS = 33 - W, MS = 4 * QS;
    constexpr int UB = (SNBP + 63) / 64, GPS = SCB / 8, NCW = GPS < 4 ? GPS : 4, GPW = GPS / NCW;
    constexpr int XR = 3 * QS + 32 + W - 1, YR = 3 * QS + 32;
    Params p{};
    p.bias = a.bias;
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.dz = static_cast<__nv_bfloat16 *>(a.dz);
    p.dx = static_cast<__nv_bfloat16 *>(a.dx);
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.R = a.R;
    p.R16 = (a.R + 15) / 16 * 16;
    p.N = a.D * a.W;
    p.bias_rows = static_cast<const uint4 *>(a.workspace);
    p.n_tiles = (p.BT + MS - 1) / MS;
    p.n_steps = (a.D + SCB - 1) / SCB;
    p.kchunks = (a.R + 63) / 64;
    p.ksteps = p.R16 / 16;
    p.z_bytes = p.kchunks * 16384;
    p.u_blk_bytes = p.R16 * 128;
    if (kColDz + p.R16 > kTmemCols) return DSC_ERR_UNSUPPORTED;
    // stage: [U blocks][bias tile][x][dy]
    unsigned off = UB * p.u_blk_bytes;
    p.bt_in = align_up(off, 1024);
    off = p.bt_in + SNBP * 16;
    p.x_in = align_up(off, 1024);
    off = p.x_in + XR * RB;
    p.dy_in = align_up(off, 1024);
    off = p.dy_in + YR * RB;
    p.stage_bytes = align_up(off, 1024);
    p.stage_tx = UB * p.u_blk_bytes + XR * RB + YR * RB + SNBP * 16;
    const unsigned g_bytes = 2 * UB * 16384;  // G hi and lo, one 16 KB block per 64 columns each
    const unsigned limit = static_cast<unsigned>(dev.max_smem_optin) - 2048;  // header and alignment slack
    // two z buffers when that still leaves four stages, else one
    p.nzbuf = 2;
    for (;;) {
        p.one_off = p.nzbuf * p.z_bytes;
        p.g_off = align_up(p.one_off + 4096, 1024);
        p.st_off = align_up(p.g_off + g_bytes, 1024);
        const unsigned room = limit - SNBP * 16;  // the shared zero K half of the bias tiles sits above the stages
        const int ns = p.st_off < room ? static_cast<int>((room - p.st_off) / p.stage_bytes) : 0;
        if (ns >= 4 || p.nzbuf == 1) {
            p.nstages = ns > kMaxStages ? kMaxStages : ns;
            break;
        }
        p.nzbuf = 1;
    }
    if (p.nstages < 2) return DSC_ERR_UNSUPPORTED;
    p.bz_off = p.st_off + p.nstages * p.stage_bytes;
    const unsigned smem = 2048 + p.bz_off + SNBP * 16;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    const unsigned long long row = static_cast<unsigned long long>(a.D) * 2;
    CUtensorMap tm_z, tm_x, tm_dy, tm_u;
    if (!encode_tmap_2d(&tm_z, a.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.R, BT, static_cast<unsigned long long>(a.R) * 2,
                        64, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, SCB, XR, swizzle_for(RB)) ||
        !encode_tmap_2d(&tm_dy, a.dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, SCB, YR, swizzle_for(RB)) ||
        !encode_tmap_2d(&tm_u, a.U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.N, a.R, static_cast<unsigned long long>(p.N) * 2,
                        64, p.R16, CU_TENSOR_MAP_SWIZZLE_128B))
        return DSC_ERR_CUDA;
    auto kern = lowrank_bwd_dxdz<W, SCB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int grid = dev.sm_count < p.n_tiles ? dev.sm_count : p.n_tiles;
    return launch_overlapped(kern, grid, kThreads, smem, a.stream, tm_z, tm_x, tm_dy, tm_u, p);
}

template <int W>
static dsc_status launch_dxdz_w(const LowrankArgs &a, const DeviceInfo &dev)
{
    // at most 128 filter columns per step; fewer where the U columns of a step hold more rows (R > 64), so
    // that at least two stages fit in shared memory beside G and the z tiles
    if (a.R <= 64) return launch_dxdz<W, lr_step_channels(W, 128)>(a, dev);
    if (a.R <= 128) return launch_dxdz<W, (W == 2 ? 32 : lr_step_channels(W, 128))>(a, dev);
    return launch_dxdz<W, (W == 1 ? 32 : lr_step_channels(W, 64))>(a, dev);
}

static dsc_status lowrank_bwd_main(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R % 8 != 0 || a.R > 256) return DSC_ERR_UNSUPPORTED;
    dsc_status s;
    switch (a.W) {
    case 1: s = launch_dxdz_w<1>(a, dev); break;
    case 2: s = launch_dxdz_w<2>(a, dev); break;
    case 3: s = launch_dxdz_w<3>(a, dev); break;
    case 4: s = launch_dxdz_w<4>(a, dev); break;
    case 5: s = launch_dxdz_w<5>(a, dev); break;
    case 6: s = launch_dxdz_w<6>(a, dev); break;
    case 7: s = launch_dxdz_w<7>(a, dev); break;
    case 8: s = launch_dxdz_w<8>(a, dev); break;
    default: return DSC_ERR_INVALID_ARG;
    }
    if (s != DSC_OK) return s;
    return lowrank_bwd_dudb(a, dev);
}

// The three launches of the backward: the bias rows (and zeroed dU, db), dx and dz, dU and db.
static dsc_status lowrank_bwd_all(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R % 8 != 0 || a.R > 256) return DSC_ERR_UNSUPPORTED;
    if (a.W < 1 || a.W > 8) return DSC_ERR_INVALID_ARG;
    const long long rows = bias_rows(a.D, a.W);
    const dsc_status s = launch_overlapped(lowrank_bwd_prep, dev.sm_count * 2, 256, 0, a.stream, a.bias, a.D * a.W,
                                           static_cast<uint4 *>(a.workspace), static_cast<int>(rows),
                                           reinterpret_cast<float4 *>(a.dU), static_cast<long long>(a.R) * a.D * a.W / 4,
                                           a.db);
    if (s != DSC_OK) return s;
    return lowrank_bwd_main(a);
}

dsc_status lowrank_bwd(const LowrankArgs &a) { return lowrank_bwd_all(a); }

}  // namespace dsc

// ------------------------------------------------------------------ allocation-free entry point
//
// Some callers cannot allocate device memory for the workspace: a plugin inside
// a host framework that owns the whole device memory pool under a fixed memory
// plan, or a latency-critical loop that must never enter the allocator.  For
// them, dsc_lowrank_bwd_noalloc takes the workspace (the bias rows, 16 bytes per
// filter column) from the fixed-size array below, which lives in the library's
// static device memory (every GPU that loads the library holds it until the
// process exits).

namespace dsc {

constexpr long long kNoAllocScratchRows = 131072;  // 2 MiB: D*W + 256 <= 131072
static __device__ __align__(256) uint4 g_lrb_scratch[kNoAllocScratchRows];

// Device address of g_lrb_scratch on the current device, looked up once per
// device and context (host code may not use the symbol itself as an address).
static SymbolCache g_scratch_cache;
static void *noalloc_scratch() { return symbol_address(&g_scratch_cache, &g_lrb_scratch); }

}  // namespace dsc

extern "C" dsc_status dsc_lowrank_bwd_noalloc(const void *x, const void *z, const void *U, const float *bias,
                                              const void *dy, void *dx, void *dz, float *dU, float *db, int B, int T,
                                              int D, int W, int R, dsc_dtype dt, const int32_t *cu_seqlens,
                                              int n_docs, cudaStream_t stream)
{
    const dsc_status s =
        dsc::lowrank_bwd_validate(x, z, U, bias, dy, dx, dz, dU, db, B, T, D, W, R, dt, cu_seqlens, n_docs);
    if (s != DSC_OK) return s;
    if (static_cast<long long>(D) * W + 256 > dsc::kNoAllocScratchRows) return DSC_ERR_INVALID_ARG;  // beyond the array
    void *scratch = dsc::noalloc_scratch();
    if (!scratch) return DSC_ERR_CUDA;
    return dsc_lowrank_bwd(x, z, U, bias, dy, dx, dz, dU, db, scratch, B, T, D, W, R, dt, cu_seqlens, n_docs, stream);
}
