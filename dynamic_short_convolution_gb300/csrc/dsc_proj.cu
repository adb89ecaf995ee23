// dsc_proj.cu -- the projection that produces the dynamic short convolution's
// input and its filter, with the convolution applied in the GEMM's epilogue
// (notes on "Dynamic Short Convolutions Improve Transformers", "Placement":
// the filter generator's projection sits beside the Q/K/V projection; the
// all-linear discussion: fusing the convolution into the matmul epilogue saves
// the round trip of its input and filter through memory):
//
//   acc[t, c]       = sum_j h[t, j] Wx[n0 + c, j]          c < CBX        x of the tile's channels
//   acc[t, CBX + i] = sum_j h[t, j] Wg[g0 W + i, j]        i < GB         their heads' filters (+ bg)
//   y[t, c] = x[t, c] + sum_{k<W} w[t, c/H, k] x~[t-k, c]                 eq. 2 + eq. 3
// x[t] (the residual and tap 0) is used as accumulated, in fp32; the earlier
// tokens' x[t-k] of taps k >= 1 is rounded to bf16 first, as it would be had
// the projection stored it (which halves the warp exchange that delivers it).
//
// Only y is written: x and w live in the TMEM accumulator and never reach HBM.
//
// Tile: 128 token rows x NP accumulator columns (CBX channels of x followed by
// the GB = (CBX/H) W columns of their filters).  Rows 0 .. W-2 of a tile are
// the W-1 tokens before it, recomputed so that every owned token (rows W-1 ..
// 127) finds its whole history in the tile; tiles advance by 128 - (W-1)
// tokens.  K (the projection's input width Dm) runs in steps of 64 through a
// TMA ring (128-byte swizzle, K-major A and B; B = Wx rows then Wg rows).
// Warps: a TMA producer, the MMA issuer (which owns TMEM), and 8 epilogue
// warps, two per TMEM lane quadrant, each taking every other 8-channel group.
// Two accumulators in TMEM (2 x 256 columns): the MMAs of the next tile run
// while the epilogue works on this one.  The epilogue reads the tap-k input
// x[t-k] from lane - k by a warp rotation; for it, the last W-1 lanes of a
// quadrant offer the previous quadrant's last rows (exchanged through shared
// memory once per tile, behind one named barrier that also carries the warps'
// common abort decision), which is what the first lanes need.
#include "dsc_internal.h"
#include "dsc_lowrank_common.cuh"  // warp_wait (bounded, suspending), tcgen05 wrappers

namespace dsc {

namespace prj {

constexpr int kM = 128;           // token rows per tile (MMA M, TMEM lanes)
constexpr int kK = 64;            // K per stage: one 128-byte swizzled row of bf16
constexpr int kEpiWarps = 8;      // two per TMEM lane quadrant
constexpr int kEpiWarp0 = 2;      // warps 0, 1: producer, MMA issuer
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kMaxStages = 6;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;     // one accumulator

struct Params {
    const float *bg;   // generator bias [(D/H) W] or nullptr
    const int32_t *cu;
    int n_docs;
    __nv_bfloat16 *y;
    int BT, T, D, H;
    int CBX, GB, NP;   // x channels, generator columns and MMA N of a tile
    int n_mt, n_nt, n_tiles, ksteps;
    unsigned a_bytes, stage_bytes, st_off, bnd_off, bnd_half;
    int nstages;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2], tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

}  // namespace prj

// 32 TMEM lanes x N consecutive columns (any N from 1 to 64) into registers.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t *r)
{
    static_assert(N >= 1 && N <= 64, "1..64 columns");
    int o = 0;
    if constexpr (N >= 32) { tmem_ld_x32(taddr, r); o = 32; }
    if constexpr (N >= 64) { tmem_ld_x32(taddr + 32, r + 32); o = 64; }
    if constexpr ((N % 32) >= 16) { tmem_ld_x16(taddr + o, r + o); o += 16; }
    if constexpr ((N % 16) >= 8) { tmem_ld_x8(taddr + o, r + o); o += 8; }
    if constexpr ((N % 8) >= 4) { tmem_ld_x4(taddr + o, r + o); o += 4; }
    if constexpr ((N % 4) >= 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                     : "=r"(r[o]), "=r"(r[o + 1])
                     : "r"(taddr + o));
        o += 2;
    }
    if constexpr ((N % 2) == 1) asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[o]) : "r"(taddr + o));
}

// W: taps; HG: heads per 8-channel group (8 / H for H = 1, 2, 4; 1 when 8 divides H)
template <int W, int HG>
__global__ void __launch_bounds__(prj::kThreads, 1)
    proj_fwd_tc(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_wx,
                const __grid_constant__ CUtensorMap tm_wg, const prj::Params p)
{
    using namespace prj;
    constexpr int MO = kM - (W - 1);  // owned tokens per tile
    constexpr int WC = HG * W;        // filter columns of one 8-channel group
    constexpr int HB = W > 1 ? W - 1 : 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *stages = base + p.st_off;            // [A: 128 rows x 128 B][B: NP rows x 128 B] per stage
    uint32_t *bnd = reinterpret_cast<uint32_t *>(base + p.bnd_off);  // [2][4 quadrants][CBX/8 groups][W-1][4 bf16 pairs]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hdr->tfull[b], 1);
            mbar_init(&hdr->tempty[b], kEpiWarps);
        }
        mbar_init(&hdr->drain, 1);
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&hdr->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // this launch may overlap the end of the stream's previous kernel: every global access comes after the wait
    grid_dependents_launch();
    grid_dependency_wait();
    const uint32_t tmem = hdr->tmem_base;
    volatile int *abort_flag = &hdr->abort_flag;
    const int n_local = p.n_tiles > static_cast<int>(blockIdx.x)
                            ? (p.n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                            : 0;

    int issued_last[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) issued_last[s] = -1;
    bool mma_any = false;

    if (warp == 0) {
        // ---------------- producer: per tile and K step the h rows (with the W-1 rows before the tile), the
        // Wx rows of the tile's channels and the Wg rows of their heads
        int k = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true;
        const unsigned tx = p.a_bytes + static_cast<unsigned>(p.CBX + p.GB) * 128u;
        for (int li = 0; li < n_local && ok; ++li) {
            const int tile = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
            const int mt = tile / p.n_nt, nt = tile - mt * p.n_nt;
            const int r0 = mt * MO - (W - 1);           // first token row of the tile (may be negative: zeros)
            const int n0 = nt * p.CBX, g0 = (n0 / p.H) * W;
            for (int ks = 0; ks < p.ksteps; ++ks, ++k) {
                if (k >= p.nstages) ok = warp_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (!ok) break;
                if (lane == 0) {
                    uint8_t *st = stages + s * p.stage_bytes;
                    mbar_arrive_expect_tx(&hdr->full[s], tx);
                    tma_load_2d(st, &tm_h, &hdr->full[s], ks * kK, r0);
                    tma_load_2d(st + p.a_bytes, &tm_wx, &hdr->full[s], ks * kK, n0);
                    tma_load_2d(st + p.a_bytes + p.CBX * 128, &tm_wg, &hdr->full[s], ks * kK, g0);
                    issued_last[s] = k;
                }
                if (++s == p.nstages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok && lane == 0) {
            record_status(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer: acc[b] = A . B^T over K, 4 MMAs of K = 16 per stage
        const uint32_t IDESC = idesc_bf16_f32(kM, p.NP, false, false);  // A, B K-major
        const uint32_t st0 = smem_u32(stages);
        const uint64_t d_a0 = sdesc_kmajor_sw128(st0), d_b0 = sdesc_kmajor_sw128(st0 + p.a_bytes);
        const uint32_t stg16 = p.stage_bytes >> 4;
        int k = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int li = 0; li < n_local && ok; ++li) {
            const int b = li & 1;
            if (li >= 2) ok = warp_wait(&hdr->tempty[b], ((li >> 1) & 1) ^ 1, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + b * kAccCols;
            for (int ks = 0; ks < p.ksteps; ++ks, ++k) {
                ok = warp_wait(&hdr->full[s], ph, p.wait_ns) && (*abort_flag == 0);
                if (!ok) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t da = d_a0 + static_cast<uint32_t>(s) * stg16, db = d_b0 + static_cast<uint32_t>(s) * stg16;
#pragma unroll
                    for (int kk = 0; kk < kK / 16; ++kk)  // 32 bytes into the 128-byte rows per K step of 16
                        umma_bf16_nc(d, da + kk * 2, db + kk * 2, IDESC, (ks > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&hdr->empty[s]);
                    if (ks == p.ksteps - 1) umma_commit(&hdr->tfull[b]);
                }
                __syncwarp();
                mma_any = true;
                if (++s == p.nstages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok && lane == 0) {
            record_status(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warp (lane quadrant q, column warp cw): rows 32q .. 32q+31 of the tile,
        // every (kEpiWarps / 4)-th 8-channel group of its G = CBX / 8, from group cw
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3, cw = ew >> 2;
        const int row = q * 32 + lane;
        const bool halo_row = row < W - 1;                // the tokens before the tile: inputs only
        const bool tail = lane >= 32 - (W - 1);           // this lane's row is among the quadrant's last W-1
        const int tj = lane - (32 - (W - 1));             // its index among them (tail lanes)
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const int G = p.CBX / 8;
        DocCursor cursor;
        bool ok = true;
        for (int li = 0; li < n_local; ++li) {
            const int tile = static_cast<int>(blockIdx.x) + li * static_cast<int>(gridDim.x);
            const int mt = tile / p.n_nt, nt = tile - mt * p.n_nt;
            const int b = li & 1;
            const int n0 = nt * p.CBX;
            const int t = mt * MO - (W - 1) + row;        // this thread's token
            const int nv = (t >= 0 && t < p.BT) ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W;
            const bool full_taps = __all_sync(0xffffffffu, nv == W);
            ok = ok && warp_wait(&hdr->tfull[b], (li >> 1) & 1, p.wait_ns);
            tc_fence_after();
            const uint32_t acc = lane_base + b * kAccCols;
            // pass 1: the last W-1 rows of this quadrant (x of every group of this warp), for the quadrant below
            if (ok && W > 1) {
                for (int g = cw; g < G; g += kEpiWarps / 4) {
                    uint32_t xv[8];
                    tmem_ld_x8(acc + g * 8, xv);
                    tmem_ld_wait();
                    if (tail)
                        *reinterpret_cast<uint4 *>(bnd + (((b * 4 + q) * G + g) * HB + tj) * 4) = make_uint4(
                            pack_bf16x2(__uint_as_float(xv[0]), __uint_as_float(xv[1])),
                            pack_bf16x2(__uint_as_float(xv[2]), __uint_as_float(xv[3])),
                            pack_bf16x2(__uint_as_float(xv[4]), __uint_as_float(xv[5])),
                            pack_bf16x2(__uint_as_float(xv[6]), __uint_as_float(xv[7])));
                }
            }
            // every epilogue warp reaches this barrier once per tile, and they decide together whether to stop
            if (named_bar_any(1, kEpiWarps * 32, !ok)) {
                ok = false;
                break;
            }
            // pass 2: eq. 2 + 3 for this warp's groups
            for (int g = cw; g < G; g += kEpiWarps / 4) {
                const int lc0 = g * 8;                    // first channel of the group within the tile
                const int c0 = n0 + lc0;
                uint32_t xv[8], wv[WC];
                tmem_ld_x8(acc + lc0, xv);
                tmem_ld_n<WC>(acc + p.CBX + (lc0 / p.H) * W, wv);
                // tail lanes: the previous quadrant's row of the same tail index (rows before the tile for
                // quadrant 0, whose lanes below W-1 are not stored)
                uint4 e4 = make_uint4(0u, 0u, 0u, 0u);  // bf16 pairs of channels (0,1) .. (6,7)
                if (tail && q > 0 && W > 1) e4 = *reinterpret_cast<const uint4 *>(bnd + (((b * 4 + q - 1) * G + g) * HB + tj) * 4);
                float wk[WC];
                const int gcol = (c0 / p.H) * W;          // generator row of the group's first head, first tap
                const bool in_range = c0 < p.D;
#pragma unroll
                for (int i = 0; i < WC; ++i) wk[i] = (p.bg != nullptr && in_range) ? __ldg(p.bg + gcol + i) : 0.f;
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < WC; ++i) wk[i] += __uint_as_float(wv[i]);
                float xf[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) xf[c] = __uint_as_float(xv[c]);
                // tap k of channel c: wk[hx(c) * W + k], hx(c) the channel's head within the group
                auto wpair = [&](int c, int kk) {
                    const int h0 = HG > 1 ? c / (8 / HG) : 0, h1 = HG > 1 ? (c + 1) / (8 / HG) : 0;
                    return make_float2(wk[h0 * W + kk], wk[h1 * W + kk]);
                };
                float2 y2[4];
                uint32_t xp[4];  // this row's x as bf16 pairs: what the earlier taps of the rows below read
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float2 x2 = make_float2(xf[2 * e2], xf[2 * e2 + 1]);
                    y2[e2] = fma2(wpair(2 * e2, 0), x2, x2);  // residual + tap 0, unrounded
                    xp[e2] = pack_bf16x2(x2.x, x2.y);
                }
                const uint32_t ep[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                for (int kk = 1; kk < W; ++kk) {
                    // x[t-k] (bf16, as a stored projection output would be): a rotation by kk lanes; lanes >= 32-kk
                    // offer the previous quadrant's tail rows
                    const bool on = full_taps || kk < nv;  // x~ is zero before the token's document start
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        uint32_t v = __shfl_sync(0xffffffffu, lane >= 32 - kk ? ep[e2] : xp[e2], (lane - kk) & 31);
                        v = on ? v : 0u;
                        y2[e2] = fma2(wpair(2 * e2, kk),
                                      make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u)), y2[e2]);
                    }
                }
                if (!halo_row && t < p.BT && in_range) {
                    const uint4 o = make_uint4(pack_bf16x2(y2[0].x, y2[0].y), pack_bf16x2(y2[1].x, y2[1].y),
                                               pack_bf16x2(y2[2].x, y2[2].y), pack_bf16x2(y2[3].x, y2[3].y));
                    *reinterpret_cast<uint4 *>(p.y + static_cast<size_t>(t) * p.D + c0) = o;
                }
            }
            // every TMEM load of this accumulator has completed: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdr->tempty[b]);
        }
        if (!ok && lane == 0) {
            record_status(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
    }

    // ---- teardown: nothing of this CTA may still be in flight
    if (warp == 0 && lane == 0) {  // every copy issued has landed (at once, unless the CTA gave up early)
        for (int s = 0; s < p.nstages; ++s)
            if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / p.nstages) & 1, kDrainLimitNs);
    }
    if (warp == 1 && lane == 0 && mma_any) {  // every MMA this thread issued has completed
        umma_commit(&hdr->drain);
        (void)mbar_wait(&hdr->drain, 0, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

// x channels per tile: a multiple of 16 (two halves of whole 8-channel groups) and of H (whole heads), with
// the tile's filter columns beside them in at most 256 accumulator columns.  0 when none fits.
static int proj_channels(int D, int W, int H)
{
    int g = 16, h = H;
    while (h != 0) {
        const int r = g % h;
        g = h;
        h = r;
    }
    const int L = 16 / g * H;  // lcm(16, H)
    int cbx = 0;
    for (int c = L; c * (H + W) <= 256 * H; c += L) cbx = c;  // c + c W / H <= 256
    if (cbx == 0) return 0;
    const int need = (D + L - 1) / L * L;
    return need < cbx ? need : cbx;
}

template <int W, int HG>
static dsc_status launch_proj(const ProjArgs &a, const DeviceInfo &dev)
{
    using namespace prj;
    constexpr int MO = kM - (W - 1);
    Params p{};
    p.bg = a.bg;
    p.cu = a.cu;
    p.n_docs = a.n_docs;
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.BT = a.B * a.T;
    p.T = a.T;
    p.D = a.D;
    p.H = a.H;
    p.CBX = proj_channels(a.D, W, a.H);
    if (p.CBX == 0) return DSC_ERR_UNSUPPORTED;
    p.GB = p.CBX / a.H * W;
    p.NP = (p.CBX + p.GB + 15) / 16 * 16;
    if (p.NP > kAccCols) return DSC_ERR_UNSUPPORTED;
    p.n_mt = (p.BT + MO - 1) / MO;
    p.n_nt = (a.D + p.CBX - 1) / p.CBX;
    const long long tiles = static_cast<long long>(p.n_mt) * p.n_nt;
    if (tiles > 0x7fffffffLL) return DSC_ERR_UNSUPPORTED;
    p.n_tiles = static_cast<int>(tiles);
    p.ksteps = (a.Dm + kK - 1) / kK;
    p.a_bytes = kM * 128;
    p.stage_bytes = align_up(p.a_bytes + p.NP * 128, 1024);
    const int hb = W > 1 ? W - 1 : 1;
    p.bnd_half = static_cast<unsigned>(4 * (p.CBX / 8) * hb * 16);  // one buffer: 4 quadrants x groups x rows, 16 B
    p.bnd_off = 0;
    p.st_off = align_up(2 * p.bnd_half, 1024);
    const unsigned room = static_cast<unsigned>(dev.max_smem_optin) - 2048 - p.st_off;
    const int ns = static_cast<int>(room / p.stage_bytes);
    if (ns < 2) return DSC_ERR_UNSUPPORTED;
    p.nstages = ns > kMaxStages ? kMaxStages : ns;
    const unsigned smem = 2048 + p.st_off + p.nstages * p.stage_bytes;
    p.status = device_status_word();
    p.wait_ns = wait_limit_ns();

    const unsigned long long BT = static_cast<unsigned long long>(p.BT), Dm = static_cast<unsigned long long>(a.Dm);
    const unsigned long long NG = static_cast<unsigned long long>(a.D / a.H) * W;
    CUtensorMap tm_h, tm_wx, tm_wg;
    if (!encode_tmap_2d(&tm_h, a.h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dm, BT, Dm * 2, kK, kM,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_wx, a.Wx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dm, static_cast<unsigned long long>(a.D), Dm * 2,
                        kK, static_cast<unsigned>(p.CBX), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_wg, a.Wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dm, NG, Dm * 2, kK,
                        static_cast<unsigned>(p.GB), CU_TENSOR_MAP_SWIZZLE_128B))
        return DSC_ERR_CUDA;
    auto kern = proj_fwd_tc<W, HG>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int grid = dev.sm_count < p.n_tiles ? dev.sm_count : p.n_tiles;
    return launch_overlapped(kern, grid, kThreads, smem, a.stream, tm_h, tm_wx, tm_wg, p);
}

template <int W>
static dsc_status launch_proj_w(const ProjArgs &a, const DeviceInfo &dev)
{
    switch (a.H) {
    case 1: return launch_proj<W, 8>(a, dev);
    case 2: return launch_proj<W, 4>(a, dev);
    case 4: return launch_proj<W, 2>(a, dev);
    default: return a.H % 8 == 0 ? launch_proj<W, 1>(a, dev) : DSC_ERR_UNSUPPORTED;
    }
}

dsc_status proj_fwd(const ProjArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    switch (a.W) {
    case 1: return launch_proj_w<1>(a, dev);
    case 2: return launch_proj_w<2>(a, dev);
    case 3: return launch_proj_w<3>(a, dev);
    case 4: return launch_proj_w<4>(a, dev);
    case 5: return launch_proj_w<5>(a, dev);
    case 6: return launch_proj_w<6>(a, dev);
    case 7: return launch_proj_w<7>(a, dev);
    case 8: return launch_proj_w<8>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

}  // namespace dsc
