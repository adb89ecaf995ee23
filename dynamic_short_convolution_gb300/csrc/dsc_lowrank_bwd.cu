// dsc_lowrank_bwd.cu -- backward pass of the low-rank fused dynamic short
// convolution (the derivative of eq. 2 + eq. 3 with w = zU + b, notes on
// "Dynamic Short Convolutions Improve Transformers", "Parameterization"):
//
//   Wt[t, n]  = sum_r z[t,r] U[r,n] + b[n]              recomputed on chip, n = d*W + k
//   dx[s,d]   = dy[s,d] + sum_k [s in doc(s+k)] Wt[s+k, d*W+k] dy[s+k,d]
//   G[t, n]   = dy[t,d] * x~[t-k,d]                     gradient of the generated filter
//   dz[t,r]   = sum_n G[t,n] U[r,n]     dU[r,n] = sum_t z[t,r] G[t,n]     db[n] = sum_t G[t,n]
//
// Three launches: a small prep kernel (U and the bias with their filter columns
// reordered tap-major within each group of 8 channels, into the workspace; dU
// and db zeroed), then two kernels split by the axis each gradient sums over:
//   lowrank_bwd_dxdz (this file)   dx and dz: a CTA owns a tile of tokens and walks
//                                  every channel, so dz (a sum over all D*W filter
//                                  columns) accumulates in TMEM and is written once
//   lowrank_bwd_dudb (dsc_lowrank_bwd_du.cu)   dU and db: a CTA owns a block of filter
//                                  columns and walks the tokens
//
// lowrank_bwd_dxdz.  Tile: 128 TMEM lanes in four quadrants of 32; quadrant q
// holds tokens t0 + q*QS + i (i < 32), QS = 33 - W, so every token a quadrant
// owns (i < QS) finds the W-1 later tokens its dx needs inside its own warp:
// the tap-k terms move by warp shuffles, with no exchange between warps.  Per
// step of SCB channels (SNB = SCB*W filter columns, tap-major per 8 channels):
//   MMA   Wt_step = z . U_step + 1 . b_step                (A z K-major; B U MN-major)   -> TMEM
//   epi   dx (shuffles), and G = dy * x~ as an exact bf16 hi + lo pair: with the
//         columns tap-major, a word of G is the packed product of a dy word and an
//         x word (one multiply for -hi, one fused multiply-add for lo); G goes to
//         TMEM (tcgen05.st), not to shared memory
//   MMA   dz += hi . U_step^T + lo . U_step^T          (A G from TMEM, the stored -hi
//         read with the instruction's negate-A bit; B U K-major)                    -> TMEM
// Shared memory carries only the MMA operands z and U and the x / dy tiles: the
// filter gradient never passes through it, which keeps the kernel clear of the
// shared-memory bandwidth that bounds it otherwise.  Warps: a TMA producer, one
// warp issuing the filter MMAs, one issuing the dz MMAs, and 16 epilogue warps.
// The filter accumulator is single (the epilogue hands it back as soon as it
// holds it in registers); G is double-buffered in TMEM, so the dz MMAs of a step
// run while the epilogue works on the next one.
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
constexpr int kColG = 128;    // G buffers of 128 columns from here (hi words, lo words 64 columns up); filter below

struct Params {
    const int32_t *cu;
    int n_docs;
    __nv_bfloat16 *dz;
    __nv_bfloat16 *dx;
    const uint4 *bias_rows;  // per permuted filter column its bias as an exact bf16 hi + lo pair, 16 bytes a column
    int BT, T, D, R, R16, N;
    int n_tiles, n_steps, kchunks, ksteps;
    unsigned z_bytes, one_off, bz_off, st_off, stage_bytes, bt_in, x_in, dy_in, u_blk_bytes, stage_tx;
    int nstages, nzbuf, ngbuf, col_dz;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t z_full[2], z_empty[2];
    uint64_t f_full, f_empty;
    uint64_t g_full[2], g_empty[2];
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
    constexpr int GW = 4 * W;                    // G words (bf16 pairs) of one group: 8 channels x W taps
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
            mbar_init(&hdr->g_full[b], 4 * NCW);
            mbar_init(&hdr->g_empty[b], 1);
            mbar_init(&hdr->drain[b], 1);
        }
        mbar_init(&hdr->f_full, 1);
        mbar_init(&hdr->f_empty, 4 * NCW);
        mbar_init(&hdr->dz_full, 1);
        mbar_init(&hdr->dz_empty, kEpiWarps);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kM * 16 / 2; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    // the bias MMA's B tile: K half 0 (the bias rows) arrives with each stage, K half 1 is this shared zero block
    for (int i = threadIdx.x; i < SNBP; i += blockDim.x) reinterpret_cast<uint4 *>(bz_s)[i] = make_uint4(0u, 0u, 0u, 0u);
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
        // step the permuted U columns, the bias pairs, x (with the causal halo) and dy
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
        // ---------------- filter MMAs: step k into the filter accumulator once the epilogue holds step k-1's
        // filter in registers.  Shared-memory descriptors are built once; a stage or K step adds
        // (byte offset >> 4) to the start-address field (bits 0-13), which never carries: shared addresses stay
        // below 256 KB.
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
        int j = 0, s = 0, zb = 0;
        uint32_t ph = 0, zph = 0;
        bool ok = true;
        for (int k = 0; k < k_total; ++k) {
            bool w = warp_wait(&hdr->full[s], ph, p.wait_ns);
            if (j == 0) w = warp_wait(&hdr->z_full[zb], zph, p.wait_ns) && w;
            if (k >= 1) w = warp_wait(&hdr->f_empty, (k - 1) & 1, p.wait_ns) && w;
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t so = static_cast<uint32_t>(s) * stg16;
                const uint64_t az = d_z0 + static_cast<uint32_t>(zb) * z16, bu = d_u0 + so;
                umma_bf16_nc(tmem, az, bu, ID_RC, 0u);
                for (int ks = 1; ks < ksteps; ++ks)  // K = R in steps of 16: 32 B into z's 128-B rows, 16 rows of U
                    umma_bf16_nc(tmem, az + (ks >> 2) * 1024 + (ks & 3) * 2, bu + 128 * ks, ID_RC, 1u);
                umma_bf16_nc(tmem, d_one, d_bt0 + so - (static_cast<uint64_t>(so) << 16), ID_BIAS, 1u);
                umma_commit(&hdr->f_full);
                if (j == p.n_steps - 1) umma_commit(&hdr->z_empty[zb]);
            }
            __syncwarp();
            mma_any = true;
            if (++j == p.n_steps) {
                j = 0;
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
        // ---------------- dz MMAs: step k once its G is in tensor memory.  A = G from TMEM (hi words with the
        // instruction's negate-A bit: the epilogue stores the negated high half), B = the step's U columns,
        // K-major, from the stage.
        const uint32_t st0 = smem_u32(stages);
        const uint32_t ID_DZ = idesc_bf16_f32(kM, p.R16, false, false);
        const uint32_t ID_DZN = ID_DZ | (1u << 13);                           // negate A
        const uint64_t d_uk0 = sdesc(st0, 16, 1024, 2);                       // U step, K-major (B)
        const uint32_t ublk16 = p.u_blk_bytes >> 4, stg16 = p.stage_bytes >> 4;
        const uint32_t dzt = tmem + static_cast<uint32_t>(p.col_dz);
        int ti = 0, j = 0, s = 0, gb = 0;
        uint32_t gph = 0;
        bool ok = true;
        for (int k = 0; k < k_total; ++k) {
            bool w = warp_wait(&hdr->g_full[gb], gph, p.wait_ns);
            if (j == 0 && ti >= 1) w = warp_wait(&hdr->dz_empty, (ti - 1) & 1, p.wait_ns) && w;
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t b0 = d_uk0 + static_cast<uint32_t>(s) * stg16, b1 = b0 + ublk16;
                const uint32_t g0 = tmem + static_cast<uint32_t>(kColG + gb * 128);
#pragma unroll
                for (int part = 0; part < 2; ++part)  // G = hi + lo (hi stored negated)
#pragma unroll
                    for (int kk = 0; kk < SNBP / 16; ++kk)  // K over the step's columns: 8 TMEM columns, 32 B of U rows
                        umma_bf16_tmem_a(dzt, g0 + part * 64 + kk * 8, ((kk >> 2) ? b1 : b0) + (kk & 3) * 2,
                                         part == 0 ? ID_DZN : ID_DZ, (part == 0 && kk == 0) ? (j > 0 ? 1u : 0u) : 1u);
                umma_commit(&hdr->g_empty[gb]);
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
            if (++gb == p.ngbuf) {
                gb = 0;
                gph ^= 1;
            }
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
        if constexpr (SNBP != SNB) {
            // the K padding of G (words SNB/2 .. SNBP/2 of hi and lo) meets U columns of the next step: zero it
            // once; no step writes it
            if (cw == 0) {
                const uint32_t zr[4] = {0u, 0u, 0u, 0u};
                for (int b = 0; b < p.ngbuf; ++b) {
                    tmem_st_x4(lane_base + kColG + b * 128 + SNB / 2, zr);
                    tmem_st_x4(lane_base + kColG + b * 128 + 64 + SNB / 2, zr);
                }
            }
        }
        DocCursor cursor;
        bool ok = true;
        int k = 0, s = 0, gb = 0;
        uint32_t ph = 0, gph = 0;
        for (int ti = 0; ti < n_local && ok; ++ti) {
            const int t0 = (static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x)) * MS;
            const int yrow = q * QS + lane;  // this thread's row in the dy tile (x tile: + W - 1)
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
                const int cs = s, cgb = gb;
                const uint32_t cph = ph, cgph = gph;
                if (++s == p.nstages) {
                    s = 0;
                    ph ^= 1;
                }
                if (++gb == p.ngbuf) {
                    gb = 0;
                    gph ^= 1;
                }
                if (!active) continue;
                bool w = warp_wait(&hdr->f_full, k & 1, p.wait_ns) && warp_wait(&hdr->full[cs], cph, p.wait_ns);
                if (!w) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *st = stages + cs * p.stage_bytes;
                // filter columns of group gi in tap-major order: acc[gi][kk*8 + c] is tap kk of channel c
                uint32_t acc[GPW][8 * W];
                uint4 dyv[GPW];
                uint4 xv[GPW][W];  // x~ rows t-k of the group's 8 channels
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = cw * GPW + gi;
                    tmem_ld_cols<8 * W>(lane_base + g * 8 * W, acc[gi]);
                    dyv[gi] = lds128(st + off_dy[gi]);
#pragma unroll
                    for (int kk = 0; kk < W; ++kk) xv[gi][kk] = lds128(st + off_x[gi][kk]);
                }
                // the filter is in registers: hand the accumulator back at once, so the next step's recompute
                // overlaps this step's arithmetic
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->f_empty);
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
                                for (int c = 0; c < 8; ++c) acc[gi][kk * 8 + c] = 0u;
                            }
                }
                // G = dy * x~ per tap and channel pair, as -hi (rounded product of the negated dy) and
                // lo = dy * x~ - hi (exact); word kk*4 + e holds channels 2e, 2e+1 of tap kk
                uint32_t gh[GPW][GW], gl[GPW][GW];
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t d = word_of(dyv[gi], e), nd = d ^ 0x80008000u;
#pragma unroll
                        for (int kk = 0; kk < W; ++kk) {
                            const uint32_t xw = word_of(xv[gi][kk], e);
                            gh[gi][kk * 4 + e] = bmul2(nd, xw);
                            gl[gi][kk * 4 + e] = bfma2(d, xw, gh[gi][kk * 4 + e]);
                        }
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->empty[cs]);  // x and dy of the stage are read
                // G into its TMEM buffer, once the dz MMAs ngbuf steps back have read it
                if (k >= p.ngbuf && !warp_wait(&hdr->g_empty[cgb], cgph ^ 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t gcol = lane_base + kColG + cgb * 128;
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = cw * GPW + gi;
                    tmem_st_cols<GW>(gcol + g * GW, gh[gi]);
                    tmem_st_cols<GW>(gcol + 64 + g * GW, gl[gi]);
                }
                // dx: residual + own tap-0 term, then the tap-k terms of the tokens k ahead (lanes + k)
                uint4 dxo[GPW];
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    float2 gy[4], dx2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t wv = word_of(dyv[gi], e);
                        gy[e] = make_float2(__uint_as_float(wv << 16), __uint_as_float(wv & 0xffff0000u));
                        dx2[e] = fma2(make_float2(__uint_as_float(acc[gi][2 * e]), __uint_as_float(acc[gi][2 * e + 1])),
                                      gy[e], gy[e]);
                    }
#pragma unroll
                    for (int kk = 1; kk < W; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 pr = mul2(make_float2(__uint_as_float(acc[gi][kk * 8 + 2 * e]),
                                                               __uint_as_float(acc[gi][kk * 8 + 2 * e + 1])),
                                                   gy[e]);
                            dx2[e].x += __shfl_down_sync(0xffffffffu, pr.x, kk);
                            dx2[e].y += __shfl_down_sync(0xffffffffu, pr.y, kk);
                        }
                    dxo[gi] = make_uint4(pack_bf16x2(dx2[0].x, dx2[0].y), pack_bf16x2(dx2[1].x, dx2[1].y),
                                         pack_bf16x2(dx2[2].x, dx2[2].y), pack_bf16x2(dx2[3].x, dx2[3].y));
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->g_full[cgb]);
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
                tmem_ld_x4(lane_base + p.col_dz + cw * r4 + c, a4);
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

// The workspace: [bias rows: 16 B per permuted filter column, N + 256 rows][U permuted, bf16 [R, N]].  Within
// each group of 8 channels the filter columns are reordered tap-major: permuted column g*8W + k*8 + c holds
// original column (g*8 + c)*W + k, so that one bf16 pair of channels (c, c+1) at tap k is one 32-bit word of
// the filter gradient G (a plain product of a dy word and an x word).
static long long bias_rows(int D, int W) { return static_cast<long long>(D) * W + 256; }
static size_t ws_u_offset(int D, int W) { return (static_cast<size_t>(bias_rows(D, W)) * 16 + 1023) / 1024 * 1024; }

// Writes the permuted bias (as exact bf16 hi + lo pairs in the first 4 bytes of a 16-byte row; rows past N
// are zero) and the permuted U into the workspace, and zeroes dU and db, which the dU / db kernel
// accumulates into.
template <int W>
__global__ void lowrank_bwd_prep(const __nv_bfloat16 *U, const float *bias, int R, int D, uint4 *rows, int n_rows,
                                 uint4 *Up, float4 *dU, float *db)
{
    grid_dependency_wait();  // the stream's previous kernel may still use dU, db or the workspace
    grid_dependents_launch();
    const int N = D * W, G = D / 8;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long i0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    for (long long i = i0; i < n_rows; i += stride) {
        float bv = 0.f;
        if (i < N) {
            const int n = static_cast<int>(i), g = n / (8 * W), rem = n - g * 8 * W, kk = rem >> 3, c = rem & 7;
            bv = bias[(g * 8 + c) * W + kk];
        }
        const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv)));
        const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv - __uint_as_float(hi << 16))));
        rows[i] = make_uint4(hi | (lo << 16), 0u, 0u, 0u);
    }
    // U: one group of 8W consecutive columns of one row per thread (W 16-byte loads, W 16-byte stores)
    const long long n_groups = static_cast<long long>(R) * G;
    for (long long i = i0; i < n_groups; i += stride) {
        const long long r = i / G, g = i - r * G;
        const uint4 *src = reinterpret_cast<const uint4 *>(U) + (r * N + g * 8 * W) / 8;
        uint32_t v[4 * W];  // bf16 pairs of the original order (c*W + k)
#pragma unroll
        for (int m = 0; m < W; ++m) {
            const uint4 q = src[m];
            v[4 * m] = q.x;
            v[4 * m + 1] = q.y;
            v[4 * m + 2] = q.z;
            v[4 * m + 3] = q.w;
        }
        auto half = [&](int n) -> uint32_t { return (v[n >> 1] >> ((n & 1) * 16)) & 0xffffu; };
        uint4 *dst = Up + (r * N + g * 8 * W) / 8;
#pragma unroll
        for (int kk = 0; kk < W; ++kk) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = half((2 * e) * W + kk) | (half((2 * e + 1) * W + kk) << 16);
            dst[kk] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const long long na4 = static_cast<long long>(R) * N / 4;
    for (long long i = i0; i < na4; i += stride) dU[i] = z4;
    for (long long i = i0; i < N; i += stride) db[i] = 0.f;
}

size_t lowrank_bwd_workspace(int B, int T, int D, int W, int R)
{
    (void)B;
    (void)T;
    const size_t u = static_cast<size_t>(R) * D * W * 2;
    return ws_u_offset(D, W) + (u + 255) / 256 * 256;
}

template <int W, int SCB>
static dsc_status launch_dxdz(const LowrankArgs &a, const DeviceInfo &dev)
{
    using namespace lrx;
    constexpr int SNB = SCB * W, SNBP = (SNB + 15) / 16 * 16, RB = SCB * 2, QS = 33 - W, MS = 4 * QS;
    constexpr int UB = (SNBP + 63) / 64;
    constexpr int XR = 3 * QS + 32 + W - 1, YR = 3 * QS + 32;
    Params p{};
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
    const void *Up = static_cast<const uint8_t *>(a.workspace) + ws_u_offset(a.D, a.W);
    p.n_tiles = (p.BT + MS - 1) / MS;
    p.n_steps = (a.D + SCB - 1) / SCB;
    p.kchunks = (a.R + 63) / 64;
    p.ksteps = p.R16 / 16;
    p.z_bytes = p.kchunks * 16384;
    p.u_blk_bytes = p.R16 * 128;
    // TMEM: the filter [0, 128), G buffers of 128 columns, dz
    p.ngbuf = p.R16 <= 128 ? 2 : 1;
    p.col_dz = kColG + 128 * p.ngbuf;
    if (p.col_dz + p.R16 > kTmemCols) return DSC_ERR_UNSUPPORTED;
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
    const unsigned limit = static_cast<unsigned>(dev.max_smem_optin) - 2048;  // header and alignment slack
    // two z buffers when that still leaves four stages, else one
    p.nzbuf = 2;
    for (;;) {
        p.one_off = p.nzbuf * p.z_bytes;
        p.st_off = align_up(p.one_off + 4096, 1024);
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
        !encode_tmap_2d(&tm_u, Up, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.N, a.R, static_cast<unsigned long long>(p.N) * 2,
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
    // that at least two stages fit in shared memory beside the z tiles
    if (a.R <= 64) return launch_dxdz<W, lr_step_channels(W, 128)>(a, dev);
    if (a.R <= 128) return launch_dxdz<W, (W == 2 ? 32 : lr_step_channels(W, 128))>(a, dev);
    return launch_dxdz<W, (W == 1 ? 32 : lr_step_channels(W, 64))>(a, dev);
}

template <int W>
static dsc_status launch_prep(const LowrankArgs &a, const DeviceInfo &dev)
{
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    return launch_overlapped(lowrank_bwd_prep<W>, dev.sm_count * 2, 256, 0, a.stream,
                             static_cast<const __nv_bfloat16 *>(a.U), a.bias, a.R, a.D, reinterpret_cast<uint4 *>(ws),
                             static_cast<int>(bias_rows(a.D, a.W)), reinterpret_cast<uint4 *>(ws + ws_u_offset(a.D, a.W)),
                             reinterpret_cast<float4 *>(a.dU), a.db);
}

// The three launches of the backward: the permuted bias and U (and zeroed dU, db), dx and dz, dU and db.
static dsc_status lowrank_bwd_all(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R % 8 != 0 || a.R > 256) return DSC_ERR_UNSUPPORTED;
    dsc_status s;
    switch (a.W) {
    case 1: s = launch_prep<1>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<1>(a, dev); break;
    case 2: s = launch_prep<2>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<2>(a, dev); break;
    case 3: s = launch_prep<3>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<3>(a, dev); break;
    case 4: s = launch_prep<4>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<4>(a, dev); break;
    case 5: s = launch_prep<5>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<5>(a, dev); break;
    case 6: s = launch_prep<6>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<6>(a, dev); break;
    case 7: s = launch_prep<7>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<7>(a, dev); break;
    case 8: s = launch_prep<8>(a, dev); if (s == DSC_OK) s = launch_dxdz_w<8>(a, dev); break;
    default: return DSC_ERR_INVALID_ARG;
    }
    if (s != DSC_OK) return s;
    return lowrank_bwd_dudb(a, dev);
}

dsc_status lowrank_bwd(const LowrankArgs &a) { return lowrank_bwd_all(a); }

}  // namespace dsc

// ------------------------------------------------------------------ allocation-free entry point
//
// Some callers cannot allocate device memory for the workspace: a plugin inside
// a host framework that owns the whole device memory pool under a fixed memory
// plan, or a latency-critical loop that must never enter the allocator.  For
// them, dsc_lowrank_bwd_noalloc takes the workspace (the reordered bias rows and
// generator U, see lowrank_bwd_workspace) from the fixed-size array below, which lives in the library's
// static device memory (every GPU that loads the library holds it until the
// process exits).

namespace dsc {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB: the workspace of the call must fit
static __device__ __align__(256) uint4 g_lrb_scratch[kNoAllocScratchBytes / 16];

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
    if (dsc::lowrank_bwd_workspace(B, T, D, W, R) > dsc::kNoAllocScratchBytes) return DSC_ERR_INVALID_ARG;  // beyond the array
    void *scratch = dsc::noalloc_scratch();
    if (!scratch) return DSC_ERR_CUDA;
    return dsc_lowrank_bwd(x, z, U, bias, dy, dx, dz, dU, db, scratch, B, T, D, W, R, dt, cu_seqlens, n_docs, stream);
}
