// dsc_lowrank_bwd_du.cu -- the parameter gradients of the low-rank fused
// dynamic short convolution (notes on "Dynamic Short Convolutions Improve
// Transformers", "Parameterization", low-rank form w = zU + b):
//
//   G[t, n]  = dy[t,d] * x~[t-k,d]          n = d*W + k, formed on chip
//   dU[r, n] = sum_t z[t,r] G[t,n]          db[n] = sum_t G[t,n]
//
// Work unit: one block of SCB channels (SNB = SCB*W filter columns) x one tile
// of 128 tokens.  A persistent CTA walks a block-major run of units and keeps
// the block's dU and db in TMEM over all of its tiles:
//   epi  G = dy * x~ as an exact bf16 pair: -hi (the rounded product of the
//        negated dy) and lo = dy * x~ - hi (one packed multiply and one fused
//        multiply-add per two entries), with the W taps of each group of 8
//        channels in tap-major order, so that an entry pair is the product of a
//        dy word and an x word; written 128-byte swizzled, tokens as rows
//   MMA  [acc_hi | acc_lo] += [z^T; 1] . [-G_hi | G_lo]  (A MN-major: the z
//        tile, then an all-ones block whose rows give db; B MN-major; hi and lo
//        side by side along N, so one MMA of N = 2*SNB reads A once for both)
// At the end of a run the epilogue forms lo - (-hi) per accumulator column, puts
// the columns back in the d*W + k order and reduces them into dU and db (fp32
// additions: a block's tokens are split between at most a few CTAs).  CTAs work
// in pairs on the two blocks of a block pair over the same token tiles, so the
// two halves of every 128-byte row of x and dy are read together.  dU and db are
// zeroed by the prep kernel two launches back; every addition comes after the
// wait for the kernel before this one (which itself waited for the prep).  For
// R > 64 the z tile fills all 128 rows of A and db has an MMA of its own
// (A = ones); for R > 128 dU takes two MMAs of 128 rows.
#include "dsc_internal.h"
#include "dsc_lowrank_common.cuh"

namespace dsc {

namespace lrg {

constexpr int kM = 128;  // tokens per tile (MMA K per unit)
constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kMaxStages = 6;
constexpr int kTmemCols = 512;

struct Params {
    const int32_t *cu;
    int n_docs;
    float *dU;
    float *db;
    int BT, T, D, R, N;
    int n_mt, n_units, n_units_odd, kchunks, rclass;
    unsigned gbuf_bytes, z_off, z_bytes, xy_off, xy_bytes, dy_in, one_off;
    int nz, nxy, col_du1, col_db;
    int *status;
    unsigned long long wait_ns;
};

// Two rings: the z tiles (read by the MMAs, released by their commit) and the x / dy tiles (read by the
// epilogue, released as soon as it holds them in registers), so x and dy stream further ahead.
struct Header {
    uint64_t z_full[kMaxStages], z_empty[kMaxStages];
    uint64_t xy_full[kMaxStages], xy_empty[kMaxStages];
    uint64_t g_full[2], g_empty[2];
    uint64_t flush, acc_empty, drain;
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace lrg

// Four fp32 additions to global memory, no value returned.
__device__ __forceinline__ void red_add_f4(float *dst, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <int W, int SCB>
__global__ void __launch_bounds__(lrg::kThreads, 1)
    lowrank_bwd_dudb(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_dy, const lrg::Params p)
{
    using namespace lrg;
    constexpr int SNB = SCB * W;
    constexpr int SNBP = (SNB + 15) / 16 * 16;
    constexpr int NM = 2 * SNBP;            // MMA N: hi columns, then lo columns
    constexpr int RB = SCB * 2;
    constexpr int GPS = SCB / 8, NCW = GPS < 4 ? GPS : 4, GPW = GPS / NCW;
    static_assert(NM <= 256 && GPS % NCW == 0, "step shape");
    constexpr uint32_t ID_DU = idesc_bf16_f32(kM, NM, true, true);  // A MN-major ([z^T; 1]), B MN-major (G)

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *g_s = base;                  // [2][NM/64 blocks][128 token rows][128 B]
    uint8_t *z_s = base + p.z_off;        // [nz][z chunks]
    uint8_t *xy_s = base + p.xy_off;      // [nxy][x, dy]
    uint8_t *one_s = base + p.one_off;    // 4 KB of bf16 ones, above every z tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nz; ++s) {
            mbar_init(&hdr->z_full[s], 1);
            mbar_init(&hdr->z_empty[s], 1);
        }
        for (int s = 0; s < p.nxy; ++s) {
            mbar_init(&hdr->xy_full[s], 1);
            mbar_init(&hdr->xy_empty[s], 4 * NCW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->g_full[b], 4 * NCW);
            mbar_init(&hdr->g_empty[b], 1);
        }
        mbar_init(&hdr->flush, 1);
        mbar_init(&hdr->acc_empty, kEpiWarps);
        mbar_init(&hdr->drain, 1);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) reinterpret_cast<uint32_t *>(one_s)[i] = 0x3F803F80u;
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(&hdr->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the kernel before this one (lowrank_bwd_dxdz) let it launch after its own wait for the inputs, so the
    // inputs may be read at once; dU and db (zeroed by the prep kernel before that one) are touched only after
    // grid_dependency_wait
    const uint32_t tmem = hdr->tmem_base;
    volatile int *abort_flag = &hdr->abort_flag;
    // CTAs work in pairs: the two CTAs of a pair walk the same run of (block pair, token tile) units, the even
    // one on the pair's first channel block, the odd one on its second, so the two 64-byte halves of the x and
    // dy rows they read are fetched at about the same time.  Unit u of a CTA is block 2*(u / n_mt) + half.
    const int half = static_cast<int>(blockIdx.x & 1u);
    const long long pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int n_valid = half ? p.n_units_odd : p.n_units;  // an odd block count leaves the last pair one block
    int u_end = static_cast<int>((pair + 1) * p.n_units / n_pairs);
    u_end = u_end < n_valid ? u_end : n_valid;
    int u_begin = static_cast<int>(pair * p.n_units / n_pairs);
    u_begin = u_begin < u_end ? u_begin : u_end;

    int z_last[kMaxStages], xy_last[kMaxStages];  // last unit loaded into each slot (producer)
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) z_last[s] = xy_last[s] = -1;
    bool mma_any = false;

    if (warp == 0) {
        // ---------------- producer: per unit its x (with the causal halo) and dy tiles, and its z tile
        int zs = 0, xs = 0;
        uint32_t zph = 0, xph = 0;
        bool ok = true;
        for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
            const int bp = u / p.n_mt, nb = 2 * bp + half, t0 = (u - bp * p.n_mt) * kM;
            if (i >= p.nxy) ok = warp_wait(&hdr->xy_empty[xs], xph ^ 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) break;
            if (lane == 0) {
                uint8_t *st = xy_s + xs * p.xy_bytes;
                mbar_arrive_expect_tx(&hdr->xy_full[xs], (kM + W - 1 + kM) * RB);
                tma_load_2d(st, &tm_x, &hdr->xy_full[xs], nb * SCB, t0 - (W - 1));
                tma_load_2d(st + p.dy_in, &tm_dy, &hdr->xy_full[xs], nb * SCB, t0);
                xy_last[xs] = i;
            }
            if (i >= p.nz) ok = warp_wait(&hdr->z_empty[zs], zph ^ 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) break;
            if (lane == 0) {
                uint8_t *zt = z_s + zs * p.z_bytes;
                mbar_arrive_expect_tx(&hdr->z_full[zs], p.z_bytes);
                for (int a = 0; a < p.kchunks; ++a) tma_load_2d(zt + a * 16384, &tm_z, &hdr->z_full[zs], a * 64, t0);
                z_last[zs] = i;
            }
            if (++xs == p.nxy) {
                xs = 0;
                xph ^= 1;
            }
            if (++zs == p.nz) {
                zs = 0;
                zph ^= 1;
            }
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        const uint32_t z0 = smem_u32(z_s), g0 = smem_u32(g_s), ones = smem_u32(one_s);
        const uint64_t d_ones2 = sdesc(ones, 2048, 1024, 2);  // [1; 1]: two 64-row all-ones blocks
        int s = 0, run = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int u = u_begin, i = 0; u < u_end; ++u, ++i) {
            const int mt = u % p.n_mt;
            const bool first = (u == u_begin) || mt == 0, last = (u + 1 == u_end) || (mt + 1 == p.n_mt);
            const int gb = i & 1;
            bool w = warp_wait(&hdr->z_full[s], ph, p.wait_ns);
            w = warp_wait(&hdr->g_full[gb], (i >> 1) & 1, p.wait_ns) && w;
            if (first && run >= 1) w = warp_wait(&hdr->acc_empty, (run - 1) & 1, p.wait_ns) && w;
            w = __all_sync(0xffffffffu, w) && (*abort_flag == 0);
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                // descriptors built once per unit; a K step of 16 tokens adds 2048 B (128 units) to the start address
                const uint32_t zs = z0 + s * p.z_bytes;
                const uint64_t bd = sdesc(g0 + gb * p.gbuf_bytes, 16384, 1024, 2);  // G, MN-major, 64-column blocks
                const uint32_t acc0 = first ? 0u : 1u;
                if (p.rclass == 0) {
                    // [z^T; 1]: the ones block lies LBO bytes above the z rows; each K step moves the start up and
                    // the LBO down by the same amount, so the ones block stays put
                    const uint64_t ad = sdesc(zs, ones - zs, 1024, 2);
#pragma unroll
                    for (int ks = 0; ks < kM / 16; ++ks)
                        umma_bf16_nc(tmem, ad + 128u * ks - (static_cast<uint64_t>(128u * ks) << 16), bd + 128u * ks,
                                     ID_DU, ks == 0 ? acc0 : 1u);
                } else {
                    const uint64_t ad = sdesc(zs, 16384, 1024, 2);
#pragma unroll
                    for (int ks = 0; ks < kM / 16; ++ks) {
                        const uint32_t acc = ks == 0 ? acc0 : 1u;
                        umma_bf16_nc(tmem, ad + 128u * ks, bd + 128u * ks, ID_DU, acc);
                        if (p.rclass == 2) umma_bf16_nc(tmem + p.col_du1, ad + 2048u + 128u * ks, bd + 128u * ks, ID_DU, acc);
                        umma_bf16_nc(tmem + p.col_db, d_ones2, bd + 128u * ks, ID_DU, acc);
                    }
                }
                umma_commit(&hdr->g_empty[gb]);
                umma_commit(&hdr->z_empty[s]);
                if (last) umma_commit(&hdr->flush);
            }
            __syncwarp();
            mma_any = true;
            if (last) ++run;
            if (++s == p.nz) {
                s = 0;
                ph ^= 1;
            }
        }
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    } else {
        // ---------------- epilogue: G of 32 tokens x this warp's channel groups; the run's dU / db flush
        const int ew = warp - 2;
        const int q = warp & 3, cw = ew >> 2;
        const bool active = cw < NCW;
        const int row = q * 32 + lane;  // token within the tile (and, at a flush, the TMEM lane = row of dU)
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        DocCursor cursor;
        int s = 0, run = 0;
        uint32_t ph = 0;
        bool ok = true, waited = false;
        // this thread's rows of the x and dy tiles: the same offsets in every slot
        uint32_t off_dy[GPW], off_x[GPW][W];
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
            off_dy[gi] = p.dy_in + swzt<RB>(row, cw * GPW + gi);
#pragma unroll
            for (int kk = 0; kk < W; ++kk) off_x[gi][kk] = swzt<RB>(row + (W - 1) - kk, cw * GPW + gi);
        }
        for (int u = u_begin, i = 0; u < u_end && ok; ++u, ++i) {
            const int bp = u / p.n_mt, nb = 2 * bp + half, mt = u - bp * p.n_mt;
            const bool first = (u == u_begin) || mt == 0, last = (u + 1 == u_end) || (mt + 1 == p.n_mt);
            const int cs = s;
            const uint32_t cph = ph;
            if (++s == p.nxy) {
                s = 0;
                ph ^= 1;
            }
            if (active) {
                if (first) cursor.reset();
                const int t = mt * kM + row;
                const int nv = t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W;
                const bool full_taps = __all_sync(0xffffffffu, nv == W);
                bool w = warp_wait(&hdr->xy_full[cs], cph, p.wait_ns);
                w = __all_sync(0xffffffffu, w) && (*abort_flag == 0);
                if (!w) {
                    ok = false;
                    break;
                }
                const uint8_t *st = xy_s + cs * p.xy_bytes;
                uint4 dyv[GPW];
                uint4 xv[GPW][W];
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    dyv[gi] = lds128(st + off_dy[gi]);
#pragma unroll
                    for (int kk = 0; kk < W; ++kk) xv[gi][kk] = lds128(st + off_x[gi][kk]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->xy_empty[cs]);  // x and dy are in registers
                if (!full_taps) {
#pragma unroll
                    for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
                        for (int kk = 1; kk < W; ++kk)
                            if (kk >= nv) xv[gi][kk] = make_uint4(0u, 0u, 0u, 0u);
                }
                // G per tap and channel pair, tap-major within the group (word kk*4 + e: channels 2e, 2e+1 of
                // tap kk): -hi = the rounded product of the negated dy, lo = dy * x~ - hi (exact)
                uint32_t ghi[GPW][4 * W], glo[GPW][4 * W];
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t d = word_of(dyv[gi], e), nd = d ^ 0x80008000u;
#pragma unroll
                        for (int kk = 0; kk < W; ++kk) {
                            const uint32_t xw = word_of(xv[gi][kk], e);
                            ghi[gi][kk * 4 + e] = bmul2(nd, xw);
                            glo[gi][kk * 4 + e] = bfma2(d, xw, ghi[gi][kk * 4 + e]);
                        }
                    }
                const int gb = i & 1;
                w = i < 2 || warp_wait(&hdr->g_empty[gb], ((i >> 1) & 1) ^ 1, p.wait_ns);
                w = __all_sync(0xffffffffu, w);
                if (!w) {
                    ok = false;
                    break;
                }
                uint8_t *gs = g_s + gb * p.gbuf_bytes;
#pragma unroll
                for (int gi = 0; gi < GPW; ++gi) {
                    const int g = cw * GPW + gi;
#pragma unroll
                    for (int m = 0; m < W; ++m) {  // 16-byte chunk m of the group's 8W columns
                        const int n = g * 8 * W + m * 8;
                        const int nl = n + SNBP;
                        *reinterpret_cast<uint4 *>(gs + (n >> 6) * 16384 + swzt<128>(row, (n & 63) >> 3)) =
                            make_uint4(ghi[gi][4 * m], ghi[gi][4 * m + 1], ghi[gi][4 * m + 2], ghi[gi][4 * m + 3]);
                        *reinterpret_cast<uint4 *>(gs + (nl >> 6) * 16384 + swzt<128>(row, (nl & 63) >> 3)) =
                            make_uint4(glo[gi][4 * m], glo[gi][4 * m + 1], glo[gi][4 * m + 2], glo[gi][4 * m + 3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->g_full[gb]);
            }
            if (last) {
                // the run's dU and db: hi + lo of each accumulator column, added into the zeroed outputs
                if (!waited) {
                    grid_dependency_wait();
                    waited = true;
                }
                bool w = warp_wait(&hdr->flush, run & 1, p.wait_ns);
                w = __all_sync(0xffffffffu, w) && (*abort_flag == 0);
                if (!w) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // accumulator column g*8W + kk*8 + c (tap-major) is filter column (g*8 + c)*W + kk of the block;
                // the high half was accumulated negated
                for (int g = cw; g < GPS; g += 4) {
                    const int n0 = nb * SNB + g * 8 * W;  // first filter column of the group
                    auto flush_rows = [&](uint32_t col_acc, float *dst_row, bool on) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {  // channels 4hh .. 4hh+3 of the group
                            uint32_t h[4 * W], l[4 * W];  // [kk*4 + e]: tap kk of channel 4hh + e
#pragma unroll
                            for (int kk = 0; kk < W; ++kk) {
                                tmem_ld_x4(lane_base + col_acc + g * 8 * W + kk * 8 + 4 * hh, h + kk * 4);
                                tmem_ld_x4(lane_base + col_acc + SNBP + g * 8 * W + kk * 8 + 4 * hh, l + kk * 4);
                            }
                            tmem_ld_wait();
                            if (on && n0 < p.N) {
#pragma unroll
                                for (int j4 = 0; j4 < W; ++j4) {  // global columns n0 + 4hh*W + 4*j4 .. +3
                                    float o[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int m = 4 * j4 + e, ch = m / W, kk = m % W;
                                        o[e] = __uint_as_float(l[kk * 4 + ch]) - __uint_as_float(h[kk * 4 + ch]);
                                    }
                                    red_add_f4(dst_row + n0 + 4 * hh * W + 4 * j4, o[0], o[1], o[2], o[3]);
                                }
                            }
                        }
                    };
                    if (p.rclass == 2) flush_rows(p.col_du1, p.dU + static_cast<size_t>(128 + row) * p.N, 128 + row < p.R);
                    if (p.rclass == 0) {
                        flush_rows(0u, row < 64 ? p.dU + static_cast<size_t>(row) * p.N : p.db,
                                   row < p.R || row == 64);
                    } else {
                        flush_rows(0u, p.dU + static_cast<size_t>(row) * p.N, row < p.R);
                        flush_rows(p.col_db, p.db, row == 0);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->acc_empty);
                ++run;
            }
        }
        if (!waited) grid_dependency_wait();  // this grid completes only after the one it depends on
        if (!ok && lane == 0) lr_abort(p.status, abort_flag);
        __syncwarp();
    }
    // the next kernel in the stream may begin its prologue
    grid_dependents_launch();

    // ---- teardown: nothing of this CTA may still be in flight
    if (warp == 0 && lane == 0) {  // every copy issued has landed (at once, unless the CTA gave up early)
        for (int s = 0; s < p.nz; ++s)
            if (z_last[s] >= 0) (void)mbar_wait_ev(&hdr->z_full[s], (z_last[s] / p.nz) & 1, kDrainLimitNs);
        for (int s = 0; s < p.nxy; ++s)
            if (xy_last[s] >= 0) (void)mbar_wait_ev(&hdr->xy_full[s], (xy_last[s] / p.nxy) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_any) {
        umma_commit(&hdr->drain);
        (void)mbar_wait_ev(&hdr->drain, 0, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

template <int W, int SCB>
static dsc_status launch_dudb(const LowrankArgs &a, const DeviceInfo &dev)
{
    using namespace lrg;
    constexpr int SNB = SCB * W, SNBP = (SNB + 15) / 16 * 16, NM = 2 * SNBP, RB = SCB * 2, XR = kM + W - 1;
    Params p{};
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.dU = a.dU;
    p.db = a.db;
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.R = a.R;
    p.N = a.D * a.W;
    p.n_mt = (p.BT + kM - 1) / kM;
    const int n_nb = (a.D + SCB - 1) / SCB;
    const long long units = static_cast<long long>((n_nb + 1) / 2) * p.n_mt;  // (block pair, token tile) units
    if (units > 0x7fffffffLL) return DSC_ERR_UNSUPPORTED;
    p.n_units = static_cast<int>(units);
    p.n_units_odd = (n_nb / 2) * p.n_mt;
    p.rclass = a.R <= 64 ? 0 : a.R <= 128 ? 1 : 2;
    p.kchunks = p.rclass == 0 ? 1 : p.rclass == 1 ? 2 : 4;  // z chunks of 64 columns (TMA zero-fills past R)
    p.col_du1 = NM;
    p.col_db = p.rclass == 2 ? 2 * NM : NM;
    if ((p.rclass == 0 ? NM : p.rclass == 1 ? 2 * NM : 3 * NM) > kTmemCols) return DSC_ERR_UNSUPPORTED;
    p.gbuf_bytes = ((NM + 63) / 64) * 16384;
    p.z_bytes = p.kchunks * 16384;
    p.dy_in = align_up(XR * RB, 1024);
    p.xy_bytes = align_up(p.dy_in + kM * RB, 1024);
    const unsigned budget = static_cast<unsigned>(dev.max_smem_optin) - 2048 - 4096 - 2 * p.gbuf_bytes;  // header, ones, G
    p.nz = (3 * p.z_bytes + 2 * p.xy_bytes <= budget) ? 3 : 2;
    if (p.nz * p.z_bytes + 2 * p.xy_bytes > budget) return DSC_ERR_UNSUPPORTED;
    p.nxy = static_cast<int>((budget - p.nz * p.z_bytes) / p.xy_bytes);
    if (p.nxy > kMaxStages) p.nxy = kMaxStages;
    p.z_off = 2 * p.gbuf_bytes;
    p.xy_off = p.z_off + p.nz * p.z_bytes;
    p.one_off = p.xy_off + p.nxy * p.xy_bytes;
    const unsigned smem = 2048 + p.one_off + 4096;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    const unsigned long long BT = static_cast<unsigned long long>(p.BT);
    const unsigned long long row = static_cast<unsigned long long>(a.D) * 2;
    CUtensorMap tm_z, tm_x, tm_dy;
    if (!encode_tmap_2d(&tm_z, a.z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.R, BT, static_cast<unsigned long long>(a.R) * 2,
                        64, kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, SCB, XR, swizzle_for(RB)) ||
        !encode_tmap_2d(&tm_dy, a.dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, BT, row, SCB, kM, swizzle_for(RB)))
        return DSC_ERR_CUDA;
    auto kern = lowrank_bwd_dudb<W, SCB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int pairs = dev.sm_count / 2 < p.n_units ? dev.sm_count / 2 : p.n_units;
    return launch_overlapped(kern, 2 * pairs, kThreads, smem, a.stream, tm_z, tm_x, tm_dy, p);
}

template <int W>
static dsc_status launch_dudb_w(const LowrankArgs &a, const DeviceInfo &dev)
{
    // hi and lo side by side: at most 128 filter columns per unit, fewer where the z tile grows with R, so
    // that two G buffers and at least two stages fit in shared memory
    if (a.R <= 64) return launch_dudb<W, (W == 2 ? 32 : lr_step_channels(W, 128))>(a, dev);
    if (a.R <= 128) return launch_dudb<W, lr_step_channels(W, 64)>(a, dev);
    return launch_dudb<W, (W == 1 ? 32 : W == 2 ? 16 : lr_step_channels(W, 64))>(a, dev);
}

dsc_status lowrank_bwd_dudb(const LowrankArgs &a, const DeviceInfo &dev)
{
    switch (a.W) {
    case 1: return launch_dudb_w<1>(a, dev);
    case 2: return launch_dudb_w<2>(a, dev);
    case 3: return launch_dudb_w<3>(a, dev);
    case 4: return launch_dudb_w<4>(a, dev);
    case 5: return launch_dudb_w<5>(a, dev);
    case 6: return launch_dudb_w<6>(a, dev);
    case 7: return launch_dudb_w<7>(a, dev);
    case 8: return launch_dudb_w<8>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

}  // namespace dsc
