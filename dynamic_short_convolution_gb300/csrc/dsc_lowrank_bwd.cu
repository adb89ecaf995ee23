// dsc_lowrank_bwd.cu -- backward pass of the low-rank fused dynamic short
// convolution (the derivative of eq. 2 + eq. 3 with w = zU + b, notes on
// "Dynamic Short Convolutions Improve Transformers", "Parameterization"):
//
//   Wt[t, n]  = sum_r z[t,r] U[r,n] + b[n]              recomputed on chip, n = d*W + k
//   dx[s,d]   = dy[s,d] + sum_k [s in doc(s+k)] Wt[s+k, d*W+k] dy[s+k,d]
//   G[t, n]   = dy[t,d] * x~[t-k,d]                     gradient of the generated filter
//   dz[t,r]   = sum_n G[t,n] U[r,n]     dU[r,n] = sum_t z[t,r] G[t,n]     db[n] = sum_t G[t,n]
//
// Work unit: one block of CB channels (NB = CB*W filter columns) x one tile of
// 128 tokens.  Tiles overlap by W-1 tokens (step MS = 128-(W-1)): a tile owns
// its first MS tokens, and the last W-1 rows only feed the dx of owned tokens
// (their filter rows come out of the same M=128 MMA).  A persistent CTA walks a
// block-major run of units; per block it keeps U's columns resident (TMA, 128-B
// swizzle) and accumulates dU^T and db in TMEM over all of its tiles.
// The block is processed in NSB sub-blocks of SNB <= 128 columns:
//   MMA  Wt_sub = z . U_sub                (A z K-major; B U_sub MN-major)   -> TMEM acc_W
//   epi  dx, and G = dy * x~ split exactly into bf16 hi + lo (a product of two
//        bf16 values has 16 significant bits), written K-major to smem
//   MMA  dz  += G . U_sub^T               (A G K-major;  B U_sub K-major)   -> TMEM acc_dz
//        dU^T += G^T . z                   (A G MN-major; B z MN-major)      -> TMEM acc_dU
//        db   += G^T . 1                   (B an all-ones tile)              -> TMEM acc_db
// dz partial sums of a tile over this block's columns are added with vector
// atomics into an fp32 workspace (one partial per block); a last small kernel
// rounds them to bf16.  dU and db are added atomically once per run of tiles.
// Row exchange for dx: the tap-k term of token t lands on token t-k, which is
// another TMEM lane: warp shuffles inside a warp, a small shared edge buffer
// across the four lane quadrants.
#include <mutex>

#include "dsc_internal.h"
#include "dsc_tcgen05.cuh"

namespace dsc {

namespace lrb {

constexpr int kM = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kStages = 2;
constexpr int kTmemCols = 512;
constexpr int kColW = 0;    // filter recompute accumulator, <= 128 columns
constexpr int kColDz = 128; // two dz accumulators of R <= 64 columns
constexpr int kColDu = 256; // NSB <= 2 dU^T accumulators of R columns
constexpr int kColDb = 384; // NSB db accumulators of 16 columns

template <int W, int CB>
struct Cfg {
    static constexpr int NB = CB * W;
    static constexpr int SCB = (W <= 2) ? CB : (W <= 4 ? 32 : 16);  // channels per sub-block
    static constexpr int NSB = CB / SCB;
    static constexpr int SNB = SCB * W;                             // columns per sub-block
    static constexpr int UCH = (SNB + 63) / 64;                     // 64-column chunks per U sub-tile
    static constexpr int GPS = SCB / 8;                             // 8-channel groups per sub-block
    static constexpr int GPH = GPS / 2;                             // groups per epilogue half
    static constexpr int RB = CB * 2;                               // bytes per x / dy / dx row
    static constexpr int XR = kM + W - 1;
    static constexpr int MS = kM - (W - 1);                         // owned tokens per tile
    static_assert(SNB % 16 == 0 && SNB <= 128 && NSB <= 2 && GPH >= 1, "sub-block shape");
};

struct Params {
    const float *bias;
    const int32_t *cu;
    int n_docs;
    float *dz_ws;
    float *dU;
    float *db;
    int BT, T, D, R, N;
    int n_nb, n_mt, n_units, MS;
    unsigned u_off, bt_off, one_off, g_off, dx_off, e_off, st_off, stage_bytes;
    unsigned u_bytes, z_bytes, x_in, x_bytes, dy_in, dy_bytes, nv_in;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t u_full;
    uint64_t accw_full, accw_empty;
    uint64_t g_full[2], g_empty[2];
    uint64_t dz_full[2], dz_empty[2];
    uint64_t flush;
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace lrb

// Four fp32 additions to global memory, no value returned.
__device__ __forceinline__ void red_add_v4(float *dst, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <int RB>
__device__ __forceinline__ uint32_t swz_b(int row, int c)
{
    if constexpr (RB == 128) return row * 128 + ((c ^ (row & 7)) << 4);
    else return row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
}

__device__ __forceinline__ uint32_t bf16_bits(float v)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// Bounded wait that records a timeout and sets the CTA abort flag, but lets the
// caller continue (used where a warp may not leave its group mid-step).
__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity, unsigned long long ns, int *status,
                                             volatile int *abort_flag)
{
    if (!mbar_wait(bar, parity, ns)) {
        record_status(status, kStatusTimeout);
        *abort_flag = 1;
    }
}

template <int W, int CB>
__global__ void __launch_bounds__(lrb::kThreads, 1)
    lowrank_bwd_tc(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_u,
                   const __grid_constant__ CUtensorMap tm_dx, const lrb::Params p)
{
    using namespace lrb;
    using C = Cfg<W, CB>;
    constexpr int NSB = C::NSB, SNB = C::SNB, UCH = C::UCH, GPH = C::GPH, RB = C::RB, SCB = C::SCB;
    constexpr int MS = C::MS;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *u_s = base + p.u_off;                            // [NSB][UCH][R rows][128 B]
    uint8_t *bt_s = base + p.bt_off;                          // bias as MMA B tiles (K half 0 per sub-block, shared zero K half 1)
    uint8_t *one_s = base + p.one_off;                        // 4 KB of bf16 ones (an MMA A tile of 128 x 16)
    uint8_t *g_s = base + p.g_off;                            // [2 (hi, lo)][2 chunks][128 rows][128 B]
    uint8_t *dx_s = base + p.dx_off;                          // [128 rows][RB], swizzled
    float2 *edge = reinterpret_cast<float2 *>(base + p.e_off);
    uint8_t *stages = base + p.st_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = p.R;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1 + kEpiWarps);
        }
        mbar_init(&hdr->u_full, 1);
        mbar_init(&hdr->accw_full, 1);
        mbar_init(&hdr->accw_empty, kEpiWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->g_full[b], kEpiWarps);
            mbar_init(&hdr->g_empty[b], 1);
            mbar_init(&hdr->dz_full[b], 1);
            mbar_init(&hdr->dz_empty[b], kEpiWarps);
        }
        mbar_init(&hdr->flush, 1);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < 1024; i += blockDim.x)
        reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;  // bf16 1.0 pairs
    fence_proxy_async_smem();
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

    int it = 0;   // tiles processed by this CTA so far (all roles count alike)
    int seg = 0;  // runs of tiles (U block loads)
    int issued_last[kStages] = {-1, -1};
    bool mma_any = false;

    for (int u = u_begin; u < u_end;) {
        const int nb = u / p.n_mt;
        const int seg_end = min(u_end, (nb + 1) * p.n_mt);
        const int ntiles = seg_end - u;

        // ---- U columns of this block (TMA) and its bias
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&hdr->u_full, p.u_bytes);
            for (int j = 0; j < NSB; ++j)
                for (int c = 0; c < UCH; ++c)
                    tma_load_2d(u_s + (j * UCH + c) * R * 128, &tm_u, &hdr->u_full, nb * C::NB + j * SNB + c * 64, 0);
        }
        // bias of each sub-block as an extra MMA K step: rows = filter columns, K = (hi, lo, 0, ...)
        for (int n = threadIdx.x; n < C::NB; n += blockDim.x) {
            const int gn = nb * C::NB + n;
            const float bv = gn < p.N ? p.bias[gn] : 0.f;
            const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv)));
            const uint32_t lo =
                static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv - __uint_as_float(hi << 16))));
            const int j = n / SNB, r = n - j * SNB;
            // core matrices of 8 rows x 16 B: K half 0 of sub-block j at j*SNB*16 + (r/8)*128; every K half 1
            // is the zero region that follows the NSB sub-blocks
            *reinterpret_cast<uint4 *>(bt_s + j * (SNB * 16) + (r >> 3) * 128 + (r & 7) * 16) =
                make_uint4(hi | (lo << 16), 0u, 0u, 0u);
        }
        for (int i = threadIdx.x; i < SNB * 16 / 16; i += blockDim.x)
            reinterpret_cast<uint4 *>(bt_s + NSB * SNB * 16)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncthreads();

        if (warp == 0) {
            // ---------------- producer: z, x (with the causal halo) and dy tiles
            for (int v = 0; v < ntiles; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                const uint32_t ph = (i / kStages) & 1;
                bool ok = mbar_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (!ok) {
                    if (lane == 0) {
                        record_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                    }
                    break;
                }
                const int mt = u + v - nb * p.n_mt;
                const int t0 = mt * MS;
                uint8_t *st = stages + s * p.stage_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&hdr->full[s], p.z_bytes + p.x_bytes + p.dy_bytes);
                    tma_load_2d(st, &tm_z, &hdr->full[s], 0, t0);
                    tma_load_2d(st + p.x_in, &tm_x, &hdr->full[s], nb * CB, t0 - (W - 1));
                    tma_load_2d(st + p.dy_in, &tm_dy, &hdr->full[s], nb * CB, t0);
                    issued_last[s] = i;
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer
            constexpr uint32_t ID_RC = idesc_bf16_f32(kM, SNB, false, true);
            constexpr uint32_t ID_BIAS = idesc_bf16_f32(kM, SNB, false, false);
            const uint32_t ID_DZ = idesc_bf16_f32(kM, R, false, false);
            const uint32_t ID_DU = idesc_bf16_f32(kM, R, true, true);
            constexpr uint32_t ID_DB = idesc_bf16_f32(kM, 16, true, false);
            const uint32_t us = smem_u32(u_s), gs = smem_u32(g_s), ones = smem_u32(one_s);
            bool ok = mbar_wait(&hdr->u_full, seg & 1, p.wait_ns);
            int prev_i = -1, prev_j = 0, prev_s = 0;
            auto issue_dzdu = [&](int i, int j, int s) {
                const bool first_tile = (i == it);
                const uint32_t zs = smem_u32(stages + s * p.stage_bytes);
                const int step = i * NSB + j;
                for (int part = 0; part < 2; ++part) {
                    ok = mbar_wait(&hdr->g_full[part], step & 1, p.wait_ns) && ok;
                    if (j == 0 && part == 0) ok = mbar_wait(&hdr->dz_empty[i & 1], ((i >> 1) & 1) ^ 1, p.wait_ns) && ok;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t gb = gs + part * 32768;
                        for (int ks = 0; ks < SNB / 16; ++ks) {  // dz += G . U_sub^T over this sub-block's columns
                            const int a = ks >> 2, kq = ks & 3;
                            umma_bf16(tmem + kColDz + (i & 1) * R, sdesc(gb + a * 16384 + kq * 32, 16, 1024, 2),
                                      sdesc(us + (j * UCH + a) * R * 128 + kq * 32, 16, 1024, 2), ID_DZ,
                                      (j == 0 && part == 0 && ks == 0) ? 0u : 1u);
                        }
                        for (int ks = 0; ks < kM / 16; ++ks) {  // dU^T += G^T . z and db += G^T . 1 over the tokens
                            const uint64_t ad = sdesc(gb + ks * 2048, 16384, 1024, 2);
                            const uint32_t acc = (first_tile && part == 0 && ks == 0) ? 0u : 1u;
                            umma_bf16(tmem + kColDu + j * R, ad, sdesc(zs + ks * 2048, 16384, 1024, 2), ID_DU, acc);
                            umma_bf16(tmem + kColDb + j * 16, ad, sdesc(ones, 128, 256, 0), ID_DB, acc);
                        }
                        umma_commit(&hdr->g_empty[part]);
                    }
                    __syncwarp();
                }
                if (j == NSB - 1 && lane == 0) {
                    umma_commit(&hdr->dz_full[i & 1]);
                    umma_commit(&hdr->empty[s]);
                }
                __syncwarp();
            };
            for (int v = 0; v < ntiles && ok; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                for (int j = 0; j < NSB; ++j) {
                    const int step = i * NSB + j;
                    if (j == 0) ok = mbar_wait(&hdr->full[s], (i / kStages) & 1, p.wait_ns) && ok;
                    ok = mbar_wait(&hdr->accw_empty, (step & 1) ^ 1, p.wait_ns) && ok;
                    ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t zs = smem_u32(stages + s * p.stage_bytes);
                        for (int ks = 0; ks < R / 16; ++ks)  // Wt_sub = z . U_sub (K = R)
                            umma_bf16(tmem + kColW, sdesc(zs + ks * 32, 16, 1024, 2),
                                      sdesc(us + j * UCH * R * 128 + ks * 2048, R * 128, 1024, 2), ID_RC,
                                      ks > 0 ? 1u : 0u);
                        umma_bf16(tmem + kColW, sdesc(ones, 128, 256, 0),  // + 1 . bias (exact hi + lo)
                                  sdesc(smem_u32(bt_s) + j * (SNB * 16), (NSB - j) * (SNB * 16), 128, 0), ID_BIAS, 1u);
                        umma_commit(&hdr->accw_full);
                    }
                    __syncwarp();
                    mma_any = true;
                    if (prev_i >= 0) issue_dzdu(prev_i, prev_j, prev_s);
                    prev_i = i;
                    prev_j = j;
                    prev_s = s;
                }
            }
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (ok && prev_i >= 0) issue_dzdu(prev_i, prev_j, prev_s);
            if (lane == 0) umma_commit(&hdr->flush);
            if (!ok && lane == 0) {
                record_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            __syncwarp();
        } else {
            // ---------------- epilogue
            const int q = warp & 3, h = (warp - 2) >> 2;
            const int row = q * 32 + lane;
            const bool store_thread = (threadIdx.x == 64);
            int gcount = 0;  // groups processed (edge-buffer parity), equal across a half
            bool epi_abort = false;
            DocCursor cursor;  // this thread's token increases from tile to tile within a run
            for (int v = 0; v < ntiles && !epi_abort; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                const int mt = u + v - nb * p.n_mt;
                const int t0 = mt * MS;
                const uint8_t *st = stages + s * p.stage_bytes;
                const uint8_t *xs = st + p.x_in;
                const uint8_t *gys = st + p.dy_in;
                for (int j = 0; j < NSB && !epi_abort; ++j) {
                    const int step = i * NSB + j;
                    bool ok = mbar_wait(&hdr->accw_full, step & 1, p.wait_ns);
                    if (j == 0) {
                        ok = mbar_wait(&hdr->full[s], (i / kStages) & 1, p.wait_ns) && ok;
                        if (store_thread) tma_store_wait_read<0>();  // dx staging free again
                    }
                    ok = ok && (*abort_flag == 0);
                    if (named_bar_any(1, 32 * kEpiWarps, !ok)) {  // every epilogue warp leaves together
                        if (lane == 0) {
                            record_status(p.status, kStatusTimeout);
                            *abort_flag = 1;
                        }
                        epi_abort = true;
                        break;
                    }
                    tc_fence_after();
                    const int nv = (t0 + row < p.BT) ? cursor.taps(t0 + row, p.T, W, p.cu, p.n_docs) : W;
                    const bool full_taps = __all_sync(0xffffffffu, nv == W);  // no token of this warp near a document start
                    const bool owned = row < MS;
                    uint32_t ghi[GPH][4 * W], glo[GPH][4 * W];
#pragma unroll
                    for (int gi = 0; gi < GPH; ++gi) {
                        const int gl = h * GPH + gi;          // group within the sub-block
                        const int ch0 = j * SCB + gl * 8;     // first channel within the block
                        uint32_t acc[8 * W];                  // filter (bias included), column c*W + k
                        tmem_ld_cols<8 * W>(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColW + gl * 8 * W, acc);
                        const uint4 gr = *reinterpret_cast<const uint4 *>(gys + swz_b<RB>(row, ch0 >> 3));
                        uint4 xr[W];
#pragma unroll
                        for (int k = 0; k < W; ++k)
                            xr[k] = *reinterpret_cast<const uint4 *>(xs + swz_b<RB>(row + (W - 1) - k, ch0 >> 3));
                        float gy[8], go[8];
                        {
                            const uint32_t wv[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                gy[2 * e] = __uint_as_float(wv[e] << 16);
                                gy[2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 8; ++c) go[c] = owned ? gy[c] : 0.f;  // G of a non-owned row is 0
                        tmem_ld_wait();
                        // dx: residual + own tap-0 term; the tap-k terms (k >= 1) of this token go to token row-k
                        float dxv[8];
                        float pk[W > 1 ? W - 1 : 1][8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            dxv[c] = fmaf(__uint_as_float(acc[c * W]), gy[c], gy[c]);
#pragma unroll
                            for (int k = 1; k < W; ++k) pk[k - 1][c] = __uint_as_float(acc[c * W + k]) * gy[c];
                        }
                        if (!full_taps) {
#pragma unroll
                            for (int k = 1; k < W; ++k)
#pragma unroll
                                for (int c = 0; c < 8; ++c) pk[k - 1][c] = k < nv ? pk[k - 1][c] : 0.f;
                        }
                        // G = dy * x~ in column order c*W + k, split exactly: hi = top 16 bits of the fp32 product,
                        // lo = the rest (it has at most 8 significant bits, so its top 16 bits hold it exactly)
#pragma unroll
                        for (int f = 0; f < 8 * W; f += 2) {
                            const int c0 = f / W, k0 = f % W, c1 = (f + 1) / W, k1 = (f + 1) % W;
                            const uint32_t xw0 = (&xr[k0].x)[c0 >> 1], xw1 = (&xr[k1].x)[c1 >> 1];
                            float x0 = __uint_as_float((c0 & 1) ? (xw0 & 0xffff0000u) : (xw0 << 16));
                            float x1 = __uint_as_float((c1 & 1) ? (xw1 & 0xffff0000u) : (xw1 << 16));
                            if (!full_taps) {
                                x0 = k0 < nv ? x0 : 0.f;
                                x1 = k1 < nv ? x1 : 0.f;
                            }
                            const float g0 = go[c0] * x0, g1 = go[c1] * x1;
                            const uint32_t b0 = __float_as_uint(g0), b1 = __float_as_uint(g1);
                            const float l0 = g0 - __uint_as_float(b0 & 0xffff0000u);
                            const float l1 = g1 - __uint_as_float(b1 & 0xffff0000u);
                            ghi[gi][f / 2] = __byte_perm(b0, b1, 0x7632);
                            glo[gi][f / 2] = __byte_perm(__float_as_uint(l0), __float_as_uint(l1), 0x7632);
                        }
                        if constexpr (W > 1) {
                            // rows row+k of this warp by shuffle; the first W-1 rows of the next quadrant by edge buffer
                            const int par = gcount & 1;
                            float2 *eh = edge + ((h * 4) * 2) * (W - 1) * (W - 1) * 4;  // [q][par][j][k-1][4]
                            if (lane < W - 1) {
#pragma unroll
                                for (int k = 1; k < W; ++k) {
                                    float2 *dst = eh + (((q * 2 + par) * (W - 1) + lane) * (W - 1) + (k - 1)) * 4;
#pragma unroll
                                    for (int e = 0; e < 4; ++e) dst[e] = make_float2(pk[k - 1][2 * e], pk[k - 1][2 * e + 1]);
                                }
                            }
                            float recv[W - 1][8];
#pragma unroll
                            for (int k = 1; k < W; ++k)
#pragma unroll
                                for (int c = 0; c < 8; ++c) recv[k - 1][c] = __shfl_down_sync(0xffffffffu, pk[k - 1][c], k);
                            named_bar(2 + h, 32 * kEpiWarps / 2);
                            if (q < 3) {
#pragma unroll
                                for (int k = 1; k < W; ++k) {
                                    if (lane + k >= 32) {
                                        const float2 *src =
                                            eh + ((((q + 1) * 2 + par) * (W - 1) + (lane + k - 32)) * (W - 1) + (k - 1)) * 4;
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            const float2 v2 = src[e];
                                            recv[k - 1][2 * e] = v2.x;
                                            recv[k - 1][2 * e + 1] = v2.y;
                                        }
                                    }
                                }
                            }
#pragma unroll
                            for (int k = 1; k < W; ++k)
#pragma unroll
                                for (int c = 0; c < 8; ++c) dxv[c] += recv[k - 1][c];
                        }
                        ++gcount;
                        if (owned) {
                            uint4 o;
                            o.x = pack_bf16x2(dxv[0], dxv[1]);
                            o.y = pack_bf16x2(dxv[2], dxv[3]);
                            o.z = pack_bf16x2(dxv[4], dxv[5]);
                            o.w = pack_bf16x2(dxv[6], dxv[7]);
                            *reinterpret_cast<uint4 *>(dx_s + swz_b<RB>(row, ch0 >> 3)) = o;
                        }
                    }
                    // the filter accumulator is consumed: the next sub-block may be recomputed
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&hdr->accw_empty);
                    // G hi, then G lo, into the two operand buffers (each freed by the MMAs of the previous step)
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        wait_or_flag(&hdr->g_empty[part], (step & 1) ^ 1, p.wait_ns, p.status, abort_flag);
                        uint8_t *gb = g_s + part * 32768;
#pragma unroll
                        for (int gi = 0; gi < GPH; ++gi) {
                            const int gl = h * GPH + gi;
#pragma unroll
                            for (int m = 0; m < W; ++m) {  // 16-byte chunk m of the group's 8W columns
                                const int col = gl * 8 * W + m * 8;
                                const uint32_t *src = part == 0 ? &ghi[gi][m * 4] : &glo[gi][m * 4];
                                *reinterpret_cast<uint4 *>(gb + (col >> 6) * 16384 + row * 128 +
                                                           ((((col & 63) >> 3) ^ (row & 7)) << 4)) =
                                    make_uint4(src[0], src[1], src[2], src[3]);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&hdr->g_full[part]);
                    }
                }
                if (epi_abort) break;
                // this tile's x / dy are no longer needed; its dx tile is complete
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->empty[s]);
                fence_proxy_async_smem();
                named_bar(1, 32 * kEpiWarps);
                if (store_thread) {
                    tma_store_2d(&tm_dx, dx_s, nb * CB, t0);
                    tma_store_commit();
                }
                // dz partial sums of the previous tile (its MMAs have had a whole tile to finish)
                if (v > 0) {
                    const int ip = i - 1;
                    wait_or_flag(&hdr->dz_full[ip & 1], (ip >> 1) & 1, p.wait_ns, p.status, abort_flag);
                    tc_fence_after();
                    const int tp = (mt - 1) * MS + row;
                    for (int c0 = h * (R / 2); c0 < (h + 1) * (R / 2); c0 += 8) {
                        uint32_t a8[8];
                        tmem_ld_x8(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColDz + (ip & 1) * R + c0, a8);
                        tmem_ld_wait();
                        if (row < MS && tp < p.BT) {
                            float *dst = p.dz_ws + static_cast<size_t>(tp) * R + c0;
                            red_add_v4(dst, __uint_as_float(a8[0]), __uint_as_float(a8[1]), __uint_as_float(a8[2]),
                                       __uint_as_float(a8[3]));
                            red_add_v4(dst + 4, __uint_as_float(a8[4]), __uint_as_float(a8[5]), __uint_as_float(a8[6]),
                                       __uint_as_float(a8[7]));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&hdr->dz_empty[ip & 1]);
                }
            }
            if (!epi_abort) {
                // end of the run: the last tile's dz, then this block's dU and db partial sums
                wait_or_flag(&hdr->flush, seg & 1, p.wait_ns, p.status, abort_flag);
                tc_fence_after();
                const int ip = it + ntiles - 1;
                const int tp = (seg_end - 1 - nb * p.n_mt) * MS + row;
                for (int c0 = h * (R / 2); c0 < (h + 1) * (R / 2); c0 += 8) {
                    uint32_t a8[8];
                    tmem_ld_x8(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColDz + (ip & 1) * R + c0, a8);
                    tmem_ld_wait();
                    if (row < MS && tp < p.BT && !*abort_flag) {
                        float *dst = p.dz_ws + static_cast<size_t>(tp) * R + c0;
                        red_add_v4(dst, __uint_as_float(a8[0]), __uint_as_float(a8[1]), __uint_as_float(a8[2]),
                                   __uint_as_float(a8[3]));
                        red_add_v4(dst + 4, __uint_as_float(a8[4]), __uint_as_float(a8[5]), __uint_as_float(a8[6]),
                                   __uint_as_float(a8[7]));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->dz_empty[ip & 1]);
#pragma unroll
                for (int j = 0; j < NSB; ++j) {
                    const int n_local = row;  // dU^T / db lane = filter column within the sub-block
                    const int gn = nb * C::NB + j * SNB + n_local;
                    const bool valid = n_local < SNB && gn < p.N && !*abort_flag;
                    for (int c0 = h * (R / 2); c0 < (h + 1) * (R / 2); c0 += 8) {
                        uint32_t a8[8];
                        tmem_ld_x8(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColDu + j * R + c0, a8);
                        tmem_ld_wait();
                        if (valid) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                atomicAdd(p.dU + static_cast<size_t>(c0 + e) * p.N + gn, __uint_as_float(a8[e]));
                        }
                    }
                    if (h == 0) {
                        uint32_t a8[8];
                        tmem_ld_x8(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColDb + j * 16, a8);
                        tmem_ld_wait();
                        if (valid) atomicAdd(p.db + gn, __uint_as_float(a8[0]));
                    }
                }
                tc_fence_before();
            }
        }
        it += ntiles;
        u = seg_end;
        ++seg;
        __syncthreads();
        if (*abort_flag) break;
    }

    // ---- teardown: nothing of this CTA may still be in flight
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (int s = 0; s < kStages; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / kStages) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_any && *abort_flag) (void)mbar_wait(&hdr->flush, (seg - 1) & 1, kDrainLimitNs);
    if (threadIdx.x == 64) tma_store_wait_all<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Zero the fp32 accumulation targets (the dz workspace, dU, db).
__global__ void lowrank_bwd_zero(float4 *a, long long na4, float4 *b, long long nb4, float *c, int nc)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long i0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = i0; i < na4; i += stride) a[i] = z;
    for (long long i = i0; i < nb4; i += stride) b[i] = z;
    for (long long i = i0; i < nc; i += stride) c[i] = 0.f;
}

// dz = bf16(dz workspace), 8 elements per thread.
__global__ void lowrank_bwd_cast(const float4 *src, uint4 *dst, long long n8)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
        const float4 a = src[2 * i], b = src[2 * i + 1];
        dst[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
}

// ------------------------------------------------------------------ host side

size_t lowrank_bwd_workspace(int B, int T, int D, int W, int R)
{
    (void)D;
    (void)W;
    const size_t bytes = static_cast<size_t>(B) * T * R * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

template <int W, int CB>
static dsc_status launch_lowrank_bwd(const LowrankArgs &a, const DeviceInfo &dev)
{
    using namespace lrb;
    using C = Cfg<W, CB>;
    Params p{};
    p.bias = a.bias;
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.dz_ws = static_cast<float *>(a.workspace);
    p.dU = a.dU;
    p.db = a.db;
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.R = a.R;
    p.N = a.D * a.W;
    p.MS = C::MS;
    p.n_nb = (a.D + CB - 1) / CB;
    p.n_mt = (p.BT + C::MS - 1) / C::MS;
    const long long units = static_cast<long long>(p.n_nb) * p.n_mt;
    if (units > 0x7fffffffLL) return DSC_ERR_UNSUPPORTED;
    p.n_units = static_cast<int>(units);
    const int R = a.R;
    unsigned off = 0;
    p.u_off = off;
    p.u_bytes = C::NSB * C::UCH * R * 128;
    off += p.u_bytes;
    p.bt_off = align_up(off, 1024);
    off = p.bt_off + (C::NSB + 1) * C::SNB * 16;
    p.one_off = align_up(off, 1024);
    off = p.one_off + 4096;
    p.g_off = align_up(off, 1024);
    off = p.g_off + 2 * 32768;
    p.dx_off = align_up(off, 1024);
    off = p.dx_off + kM * C::RB;
    p.e_off = align_up(off, 128);
    off = p.e_off + 2 * 4 * 2 * (W - 1) * (W - 1) * 32;
    p.st_off = align_up(off, 1024);
    p.z_bytes = 16384;
    p.x_in = p.z_bytes;
    p.x_bytes = C::XR * C::RB;
    p.dy_in = align_up(p.x_in + p.x_bytes, 1024);
    p.dy_bytes = kM * C::RB;
    p.nv_in = 0;
    p.stage_bytes = align_up(p.dy_in + p.dy_bytes, 1024);
    const unsigned smem = 2048 + p.st_off + kStages * p.stage_bytes;
    if (smem > static_cast<unsigned>(dev.max_smem_optin)) return DSC_ERR_UNSUPPORTED;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    const CUtensorMapSwizzle sw = C::RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    const unsigned long long row = static_cast<unsigned long long>(a.D) * 2;
    CUtensorMap tm_z, tm_x, tm_dy, tm_u, tm_dx;
    if (!encode_tmap_2d(&tm_z, a.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, R, BT, static_cast<unsigned long long>(R) * 2, 64,
                        kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, CB, C::XR, sw) ||
        !encode_tmap_2d(&tm_dy, a.dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, CB, kM, sw) ||
        !encode_tmap_2d(&tm_u, a.U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.N, R, static_cast<unsigned long long>(p.N) * 2,
                        64, R, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_dx, a.dx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, CB, C::MS, sw))
        return DSC_ERR_CUDA;

    const long long nz = static_cast<long long>(p.BT) * R;
    lowrank_bwd_zero<<<dev.sm_count * 4, 256, 0, a.stream>>>(reinterpret_cast<float4 *>(p.dz_ws), nz / 4,
                                                            reinterpret_cast<float4 *>(a.dU),
                                                            static_cast<long long>(R) * p.N / 4, a.db, p.N);
    dsc_status s = launched();
    if (s != DSC_OK) return s;
    auto kern = lowrank_bwd_tc<W, CB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int grid = dev.sm_count < p.n_units ? dev.sm_count : p.n_units;
    kern<<<grid, kThreads, smem, a.stream>>>(tm_z, tm_x, tm_dy, tm_u, tm_dx, p);
    s = launched();
    if (s != DSC_OK) return s;
    lowrank_bwd_cast<<<dev.sm_count * 4, 256, 0, a.stream>>>(reinterpret_cast<const float4 *>(p.dz_ws),
                                                             static_cast<uint4 *>(a.dz), nz / 8);
    return launched();
}

dsc_status lowrank_bwd(const LowrankArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    if (a.R % 16 != 0 || a.R > 64) return DSC_ERR_UNSUPPORTED;
    switch (a.W) {
    case 1: return launch_lowrank_bwd<1, 64>(a, dev);
    case 2: return launch_lowrank_bwd<2, 64>(a, dev);
    case 3: return launch_lowrank_bwd<3, 64>(a, dev);
    case 4: return launch_lowrank_bwd<4, 64>(a, dev);
    case 5: return launch_lowrank_bwd<5, 32>(a, dev);
    case 6: return launch_lowrank_bwd<6, 32>(a, dev);
    case 7: return launch_lowrank_bwd<7, 32>(a, dev);
    case 8: return launch_lowrank_bwd<8, 32>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

// ------------------------------------------------------------------ allocation-free entry point
//
// Some callers cannot allocate device memory for the workspace: a plugin inside
// a host framework that owns the whole device memory pool under a fixed memory
// plan, or a latency-critical loop that must never enter the allocator.  For
// them, dsc_lowrank_bwd_noalloc takes its fp32 dz partial sums from the
// fixed-size array below, which lives in the library's static device memory
// (every GPU that loads the library holds it until the process exits).

constexpr size_t kNoAllocScratchFloats = size_t(1) << 21;  // 8 MiB: B*T*R <= 2,097,152
static __device__ __align__(256) float g_lrb_scratch[kNoAllocScratchFloats];

// Device address of g_lrb_scratch on the current device, looked up once per
// device (host code may not use the symbol itself as an address).
static float *noalloc_scratch()
{
    static std::mutex mu;
    static float *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_lrb_scratch) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<float *>(ptr);
    }
    return addr[dev];
}

}  // namespace dsc

extern "C" dsc_status dsc_lowrank_bwd_noalloc(const void *x, const void *z, const void *U, const float *bias,
                                              const void *dy, void *dx, void *dz, float *dU, float *db, int B, int T,
                                              int D, int W, int R, dsc_dtype dt, const int32_t *cu_seqlens,
                                              int n_docs, cudaStream_t stream)
{
    if (B < 1 || T < 1 || R < 1) return DSC_ERR_INVALID_ARG;
    if (static_cast<size_t>(B) * T * R > dsc::kNoAllocScratchFloats) return DSC_ERR_INVALID_ARG;  // beyond the array
    float *scratch = dsc::noalloc_scratch();
    if (!scratch) return DSC_ERR_CUDA;
    return dsc_lowrank_bwd(x, z, U, bias, dy, dx, dz, dU, db, scratch, B, T, D, W, R, dt, cu_seqlens, n_docs, stream);
}
