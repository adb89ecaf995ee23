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
// swizzle) and accumulates dU and db in TMEM over all of its tiles.
// Each tile is processed in NSB steps of SNB <= 128 filter columns, so that every
// MMA but dz has N >= 96 (a tcgen05 MMA of N <= 64 costs about as much as N = 128):
//   MMA  Wt_sub  = z . U_sub + 1 . b_sub       (A z K-major; B U_sub MN-major)  -> TMEM
//   epi  dx, and G = dy * x~ split exactly into bf16 hi + lo (a product of two
//        bf16 values has 16 significant bits), written K-major to shared memory
//   MMA  dz     += G . U_sub^T                 (A G K-major; B U_sub K-major)   -> TMEM, per tile
//        [dU; db] += [z^T; 1] . G               (A MN-major: z then an all-ones block; B G MN-major)
//                                               -> TMEM rows 0..R-1 = dU, rows 64..127 = db
// The filter accumulator is handed back as soon as the epilogue has loaded it, so
// the next step's recompute overlaps the epilogue's arithmetic.  dx is written
// over dy in the stage (each dy element is read only by the thread that overwrites
// it) and stored by the producer warp once the tile is done.
// dz partial sums of a tile over this block's columns are added with vector
// reductions into an fp32 workspace (one partial per block); a last small
// kernel rounds them to bf16.  dU and db are added once per run of tiles.
// Row exchange for dx: the tap-k term of token t lands on token t-k, which is
// another TMEM lane: warp shuffles inside a warp, a small shared edge buffer
// across the four lane quadrants.
#include "dsc_internal.h"
#include "dsc_tcgen05.cuh"

namespace dsc {

namespace lrb {

constexpr int kM = 128;
constexpr int kEpiWarps = 16;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kStages = 2;
constexpr int kTmemCols = 512;
constexpr int kColW = 0;        // filter accumulator, SNB <= 128 columns
constexpr int kColDz = 128;     // two dz accumulators of R <= 64 columns
constexpr int kColDu = 256;     // [dU; db] accumulator, NSB * SNB <= 256 columns
constexpr int kGBlock = 16384;  // one 64-column block of G: 128 rows x 128 B
constexpr int kGPart = 2 * kGBlock;

// Channels per step: the largest multiple of 8 that divides CB with SCB*W <= 128
// and SCB*W a multiple of 16 (the MMA N granularity).
__host__ __device__ constexpr int step_channels(int W, int CB)
{
    for (int s = (128 / W) / 8 * 8; s >= 8; s -= 8)
        if (s <= CB && CB % s == 0 && (s * W) % 16 == 0) return s;
    return 0;
}

template <int W, int CB>
struct Cfg {
    static constexpr int NB = CB * W;
    static constexpr int SCB = step_channels(W, CB);
    static constexpr int NSB = CB / SCB;
    static constexpr int SNB = SCB * W;                  // filter columns per step (MMA N)
    static constexpr int GB = (SNB + 63) / 64;           // 64-column blocks of G and of a U step
    static constexpr int GPS = SCB / 8;                  // 8-channel groups per step
    static constexpr int NCA = GPS < 4 ? GPS : 4;        // column warps with work
    static constexpr int GPW = GPS / NCA;                // groups per working warp
    static constexpr int RB = CB * 2;                    // bytes per x / dy / dx row
    static constexpr int XR = kM + W - 1;
    static constexpr int MS = kM - (W - 1);              // owned tokens per tile
    static constexpr int QDU = NSB * SNB / 4;            // dU columns flushed per column warp
    static_assert(SCB >= 8 && SNB <= 128 && SNB % 16 == 0 && NSB * SNB <= 256 && GPS % NCA == 0, "step shape");
    static_assert(QDU % 8 == 0, "flush chunks");
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
    unsigned u_off, bt_off, one_off, g_off, e_off, st_off, stage_bytes;
    unsigned u_bytes, z_bytes, x_in, x_bytes, dy_in, dy_bytes;
    int *status;
    unsigned long long wait_ns;
};

struct Header {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t dx_full[kStages];
    uint64_t u_full;
    uint64_t accw_full, accw_empty;
    uint64_t g_full, g_empty;
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
    constexpr int NSB = C::NSB, SNB = C::SNB, GB = C::GB, GPW = C::GPW, RB = C::RB, SCB = C::SCB, MS = C::MS;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Header *hdr = reinterpret_cast<Header *>(smem_raw);
    uint8_t *base = smem_raw + 1024;
    base += (1024u - (smem_u32(base) & 1023u)) & 1023u;
    uint8_t *u_s = base + p.u_off;       // [NSB][GB][R rows][128 B]: U columns of each step, 128-B swizzle
    uint8_t *bt_s = base + p.bt_off;     // bias as MMA B tiles (K half 0 per step, one shared zero K half 1)
    uint8_t *one_s = base + p.one_off;   // 4 KB of bf16 ones, above every stage
    uint8_t *g_s = base + p.g_off;       // [hi, lo][GB][128 rows][128 B]: G, swizzled
    float2 *edge = reinterpret_cast<float2 *>(base + p.e_off);
    uint8_t *stages = base + p.st_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = p.R;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], 1);
            mbar_init(&hdr->dx_full[s], kEpiWarps);
        }
        mbar_init(&hdr->u_full, 1);
        mbar_init(&hdr->accw_full, 1);
        mbar_init(&hdr->accw_empty, kEpiWarps);
        mbar_init(&hdr->g_full, kEpiWarps);
        mbar_init(&hdr->g_empty, 1);
        for (int b = 0; b < 2; ++b) {
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

        // ---- U columns of this block (TMA, 64-column boxes per step) and its bias
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&hdr->u_full, p.u_bytes);
            for (int j = 0; j < NSB; ++j)
                for (int b = 0; b < GB; ++b)
                    tma_load_2d(u_s + (j * GB + b) * R * 128, &tm_u, &hdr->u_full, nb * C::NB + j * SNB + b * 64, 0);
        }
        // bias of each step as an extra MMA K step: rows = filter columns, K = (hi, lo, 0, ...)
        for (int n = threadIdx.x; n < NSB * SNB; n += blockDim.x) {
            const int j = n / SNB, r = n - j * SNB;
            const int gn = nb * C::NB + n;
            const float bv = gn < p.N ? p.bias[gn] : 0.f;
            const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv)));
            const uint32_t lo =
                static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(bv - __uint_as_float(hi << 16))));
            // core matrices of 8 rows x 16 B: K half 0 of step j at j*SNB*16 + (r/8)*128
            *reinterpret_cast<uint4 *>(bt_s + j * (SNB * 16) + (r >> 3) * 128 + (r & 7) * 16) =
                make_uint4(hi | (lo << 16), 0u, 0u, 0u);
        }
        for (int i = threadIdx.x; i < SNB; i += blockDim.x)  // the shared zero K half
            reinterpret_cast<uint4 *>(bt_s + NSB * SNB * 16)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncthreads();

        if (warp == 0) {
            // ---------------- producer: z, x (with the causal halo) and dy tiles in; dx tiles out
            bool ok = true;
            for (int v = 0; v < ntiles; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                if (i >= kStages) {  // stage s last held tile i-2: its MMAs and its epilogue are done
                    const uint32_t par = ((i / kStages) & 1) ^ 1;
                    ok = mbar_wait(&hdr->empty[s], par, p.wait_ns);
                    ok = mbar_wait(&hdr->dx_full[s], par, p.wait_ns) && ok;
                }
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (!ok) break;
                const int mt = u + v - nb * p.n_mt;
                uint8_t *st = stages + s * p.stage_bytes;
                if (lane == 0) {
                    if (v >= kStages) {  // dx of tile i-2 (same run) sits over its dy
                        tma_store_2d(&tm_dx, st + p.dy_in, nb * CB, (mt - kStages) * MS);
                        tma_store_commit();
                        tma_store_wait_read<0>();
                    }
                    const int t0 = mt * MS;
                    mbar_arrive_expect_tx(&hdr->full[s], p.z_bytes + p.x_bytes + p.dy_bytes);
                    tma_load_2d(st, &tm_z, &hdr->full[s], 0, t0);
                    tma_load_2d(st + p.x_in, &tm_x, &hdr->full[s], nb * CB, t0 - (W - 1));
                    tma_load_2d(st + p.dy_in, &tm_dy, &hdr->full[s], nb * CB, t0);
                    issued_last[s] = i;
                }
                __syncwarp();
            }
            // the dx of the run's last (up to two) tiles
            for (int v = ntiles > kStages ? ntiles - kStages : 0; v < ntiles && ok; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                ok = mbar_wait(&hdr->dx_full[s], (i / kStages) & 1, p.wait_ns);
                ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                if (ok && lane == 0) {
                    tma_store_2d(&tm_dx, stages + s * p.stage_bytes + p.dy_in, nb * CB, (u + v - nb * p.n_mt) * MS);
                    tma_store_commit();
                }
            }
            if (lane == 0) tma_store_wait_read<0>();  // the stages may be refilled by the next run
            if (!ok && lane == 0) {
                record_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            __syncwarp();
        } else if (warp == 1) {
            // ---------------- MMA issuer: per step k, the filter of step k and the gradients of step k-1
            constexpr uint32_t ID_RC = idesc_bf16_f32(kM, SNB, false, true);
            constexpr uint32_t ID_BIAS = idesc_bf16_f32(kM, SNB, false, false);
            constexpr uint32_t ID_DU = idesc_bf16_f32(kM, SNB, true, true);
            const uint32_t ID_DZ = idesc_bf16_f32(kM, R, false, false);
            const uint32_t ones = smem_u32(one_s), st0 = smem_u32(stages);
            // descriptors are built once; a K step, block or buffer change adds (byte offset >> 4) to the
            // start-address field (bits 0-13), which never carries: shared addresses stay below 256 KB
            const uint64_t d_g = sdesc(smem_u32(g_s), kGBlock, 1024, 2);  // G, MN-major (dU B): LBO = block stride
            const uint64_t d_gk = sdesc(smem_u32(g_s), 16, 1024, 2);      // G, K-major (dz A)
            const uint64_t d_u = sdesc(smem_u32(u_s), R * 128, 1024, 2);  // U step, MN-major (rc B): LBO = block stride
            const uint64_t d_uk = sdesc(smem_u32(u_s), 16, 1024, 2);      // U step, K-major (dz B)
            const uint64_t d_z = sdesc(st0, 16, 1024, 2);                 // z tile, K-major (rc A)
            const uint64_t d_one = sdesc(ones, 128, 256, 0);              // all-ones A of the bias step
            const uint64_t d_bt = sdesc(smem_u32(bt_s), 0, 128, 0);       // bias B; LBO set per step
            const uint32_t ublk = static_cast<uint32_t>(R * 128) >> 4;     // one U block, descriptor units
            const int nkr = R / 16;
            bool ok = mbar_wait(&hdr->u_full, seg & 1, p.wait_ns);
            const int k0 = it * NSB, nsteps = ntiles * NSB;
            for (int kk = 0; kk <= nsteps && ok; ++kk) {
                const int k = k0 + kk;
                if (kk < nsteps) {
                    // filter of step k: once the epilogue holds step k-1's filter in registers
                    const int i = k / NSB, j = k - i * NSB, s = i % kStages;
                    if (j == 0) ok = mbar_wait(&hdr->full[s], (i / kStages) & 1, p.wait_ns) && ok;
                    ok = mbar_wait(&hdr->accw_empty, (k & 1) ^ 1, p.wait_ns) && ok;
                    ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t a_z = d_z + ((s * p.stage_bytes) >> 4);
                        const uint64_t b_u = d_u + static_cast<uint32_t>(j * GB) * ublk;
                        const uint32_t d = tmem + kColW;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)  // Wt_sub = z . U_sub, K = R: 32 B in z, 16 rows in U
                            if (ks < nkr) umma_bf16_nc(d, a_z + 2 * ks, b_u + 128 * ks, ID_RC, ks > 0 ? 1u : 0u);
                        // + 1 . bias (exact hi + lo): K half 0 at this step's tile, K half 1 the shared zero tile
                        umma_bf16_nc(d, d_one,
                                     d_bt + static_cast<uint32_t>(j * SNB) +
                                         (static_cast<uint64_t>((NSB - j) * SNB) << 16),
                                     ID_BIAS, 1u);
                        umma_commit(&hdr->accw_full);
                    }
                    __syncwarp();
                    mma_any = true;
                }
                if (kk > 0) {
                    // gradients of step k-1, once its G is in shared memory
                    const int kg = k - 1;
                    const int i = kg / NSB, j = kg - i * NSB, s = i % kStages;
                    ok = mbar_wait(&hdr->g_full, kg & 1, p.wait_ns) && ok;
                    if (j == 0) ok = mbar_wait(&hdr->dz_empty[i & 1], ((i >> 1) & 1) ^ 1, p.wait_ns) && ok;
                    ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
                    if (!ok) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t zs = st0 + s * p.stage_bytes;
                        // [z^T; 1], MN-major: the second 64-row block (the ones) lies LBO bytes above the z tile
                        const uint64_t a_zt = sdesc(zs, ones - zs, 1024, 2);
                        const uint64_t b_uk = d_uk + static_cast<uint32_t>(j * GB) * ublk;
                        const uint32_t t_dz = tmem + kColDz + (i & 1) * R, t_du = tmem + kColDu + j * SNB;
                        const uint32_t acc_dz = j > 0 ? 1u : 0u, acc_du = i > it ? 1u : 0u;
#pragma unroll
                        for (int part = 0; part < 2; ++part) {  // G = hi + lo
                            const uint64_t ga = d_g + part * (kGPart >> 4), gak = d_gk + part * (kGPart >> 4);
#pragma unroll
                            for (int ks = 0; ks < SNB / 16; ++ks)  // dz += G . U_sub^T: K over the step's columns
                                umma_bf16_nc(t_dz, gak + (ks / 4) * (kGBlock >> 4) + (ks % 4) * 2,
                                             b_uk + (ks / 4) * ublk + (ks % 4) * 2, ID_DZ,
                                             (part == 0 && ks == 0) ? acc_dz : 1u);
#pragma unroll
                            for (int ks = 0; ks < kM / 16; ++ks)  // [dU; db] += [z^T; 1] . G: K over 16-token rows
                                umma_bf16_nc(t_du,
                                             a_zt + static_cast<uint64_t>(128 * ks) -
                                                 (static_cast<uint64_t>(128 * ks) << 16),
                                             ga + 128 * ks, ID_DU, (part == 0 && ks == 0) ? acc_du : 1u);
                        }
                        umma_commit(&hdr->g_empty);
                        if (j == NSB - 1) {
                            umma_commit(&hdr->dz_full[i & 1]);
                            umma_commit(&hdr->empty[s]);
                        }
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) umma_commit(&hdr->flush);
            if (!ok && lane == 0) {
                record_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            __syncwarp();
        } else {
            // ---------------- epilogue: 16 warps, lane quadrant q, column warp c
            const int q = warp & 3, c = (warp - 2) >> 2;
            const int row = q * 32 + lane;
            const bool active = c < C::NCA;
            const bool owned = row < MS;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
            int gcount = 0;  // groups processed (edge-buffer parity), equal across one column warp's quadrants
            bool epi_abort = false;
            // the accumulation targets are zeroed by the kernel launched just before this one, which this
            // kernel may overlap: every reduction into them comes after this wait
            if (u == u_begin) grid_dependency_wait();
            DocCursor cursor;  // this thread's token increases from tile to tile within a run
            for (int v = 0; v < ntiles && !epi_abort; ++v) {
                const int i = it + v;
                const int s = i % kStages;
                const int mt = u + v - nb * p.n_mt;
                const int t0 = mt * MS;
                uint8_t *st = stages + s * p.stage_bytes;
                const uint8_t *xs = st + p.x_in;
                uint8_t *dys = st + p.dy_in;
                int nv = W;
                bool full_taps = true;
                for (int j = 0; j < NSB && !epi_abort; ++j) {
                    const int k = i * NSB + j;
                    bool ok = mbar_wait(&hdr->accw_full, k & 1, p.wait_ns);
                    if (j == 0) ok = mbar_wait(&hdr->full[s], (i / kStages) & 1, p.wait_ns) && ok;
                    ok = ok && (*abort_flag == 0);
                    // A warp leaves only together with the warps it meets at a named barrier: the four quadrants
                    // of a column warp decide at their exchange barrier; a warp with no such barrier decides alone.
                    // Every other wait is bounded, so the rest of the CTA follows through the abort flag.
                    bool bad = !ok;
                    if (!(active && W > 1)) {
                        if (__any_sync(0xffffffffu, bad)) {
                            if (lane == 0) {
                                record_status(p.status, kStatusTimeout);
                                *abort_flag = 1;
                            }
                            epi_abort = true;
                            break;
                        }
                        bad = false;
                    }
                    tc_fence_after();
                    if (j == 0) {
                        nv = (t0 + row < p.BT) ? cursor.taps(t0 + row, p.T, W, p.cu, p.n_docs) : W;
                        full_taps = __all_sync(0xffffffffu, nv == W);  // no token of this warp near a document start
                    }
                    // this warp's filter columns (bias included) of the step: group gl, column c*W + k
                    uint32_t acc[GPW][8 * W];
                    uint4 gpre[GPW];  // dy of this token, read from shared memory while the TMEM load is in flight
                    if (active) {
#pragma unroll
                        for (int gi = 0; gi < GPW; ++gi)
                            tmem_ld_cols<8 * W>(lane_base + kColW + (c * GPW + gi) * 8 * W, acc[gi]);
#pragma unroll
                        for (int gi = 0; gi < GPW; ++gi)
                            gpre[gi] = *reinterpret_cast<const uint4 *>(
                                dys + swz_b<RB>(row, (j * SCB + (c * GPW + gi) * 8) >> 3));
                    }
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&hdr->accw_empty);  // the next step's filter may be computed
                    if (active) {
#pragma unroll
                        for (int gi = 0; gi < GPW; ++gi) {
                            const int gl = c * GPW + gi;       // group within the step
                            const int ch0 = j * SCB + gl * 8;  // first channel within the block
                            const uint32_t dy_off = swz_b<RB>(row, ch0 >> 3);
                            float gy[8];  // dy of this token
                            float dxv[8];
                            {
                                const uint4 gr = gpre[gi];
                                const uint32_t wv[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    gy[2 * e] = __uint_as_float(wv[e] << 16);
                                    gy[2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
                                }
                            }
                            // dx: residual + own tap-0 term
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float2 d2 = __ffma2_rn(
                                    make_float2(__uint_as_float(acc[gi][e * W]), __uint_as_float(acc[gi][(e + 1) * W])),
                                    make_float2(gy[e], gy[e + 1]), make_float2(gy[e], gy[e + 1]));
                                dxv[e] = d2.x;
                                dxv[e + 1] = d2.y;
                            }
                            if constexpr (W > 1) {
                                // the tap-k term of this token goes to token row-k: rows of this warp by shuffle, one
                                // tap at a time; the first W-1 rows of the next quadrant through the edge buffer
                                // [c][q][par][lane][k-1][4]
                                const int par = gcount & 1;
                                float2 *eh = edge + c * (4 * 2 * (W - 1) * (W - 1) * 4);
#pragma unroll
                                for (int kk = 1; kk < W; ++kk) {
                                    float pk[8];
#pragma unroll
                                    for (int e = 0; e < 8; e += 2) {
                                        const float2 p2 = __fmul2_rn(make_float2(__uint_as_float(acc[gi][e * W + kk]),
                                                                                 __uint_as_float(acc[gi][(e + 1) * W + kk])),
                                                                     make_float2(gy[e], gy[e + 1]));
                                        pk[e] = p2.x;
                                        pk[e + 1] = p2.y;
                                    }
                                    if (!full_taps) {
#pragma unroll
                                        for (int e = 0; e < 8; ++e) pk[e] = kk < nv ? pk[e] : 0.f;
                                    }
                                    if (lane < W - 1) {
                                        float2 *dst = eh + (((q * 2 + par) * (W - 1) + lane) * (W - 1) + (kk - 1)) * 4;
#pragma unroll
                                        for (int e = 0; e < 4; ++e) dst[e] = make_float2(pk[2 * e], pk[2 * e + 1]);
                                    }
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        const float v = __shfl_down_sync(0xffffffffu, pk[e], kk);
                                        dxv[e] += lane + kk < 32 ? v : 0.f;
                                    }
                                }
                                if (named_bar_any(2 + c, 128, bad)) {
                                    if (lane == 0) {
                                        record_status(p.status, kStatusTimeout);
                                        *abort_flag = 1;
                                    }
                                    epi_abort = true;
                                    break;
                                }
                                if (q < 3) {  // the last quadrant's last W-1 rows are not owned
#pragma unroll
                                    for (int kk = 1; kk < W; ++kk) {
                                        if (lane + kk >= 32) {
                                            const float2 *src =
                                                eh + ((((q + 1) * 2 + par) * (W - 1) + (lane + kk - 32)) * (W - 1) +
                                                      (kk - 1)) * 4;
#pragma unroll
                                            for (int e = 0; e < 4; ++e) {
                                                const float2 ev = src[e];
                                                dxv[2 * e] += ev.x;
                                                dxv[2 * e + 1] += ev.y;
                                            }
                                        }
                                    }
                                }
                            }
                            ++gcount;
                            // x~ rows row+W-1-k of this group's 8 channels: one 16-byte load per tap (conflict-free
                            // under the 128-byte swizzle) where registers allow, 4-byte loads otherwise
                            uint4 xr[W <= 4 ? W : 1];
                            if constexpr (W <= 4) {
#pragma unroll
                                for (int kk = 0; kk < W; ++kk)
                                    xr[kk] = *reinterpret_cast<const uint4 *>(xs + swz_b<RB>(row + (W - 1) - kk, ch0 >> 3));
                            }
                            // G of this group into the step's buffer, once the previous step's MMAs have read it
                            if (gi == 0)
                                wait_or_flag(&hdr->g_empty, (k & 1) ^ 1, p.wait_ns, p.status, abort_flag);
#pragma unroll
                            for (int m = 0; m < W; ++m) {  // 16-byte chunk m of the group's 8W columns
                                // G = dy * x~, column c*W + k: hi = top 16 bits of the fp32 product (exact), lo =
                                // the rest (at most 8 significant bits, so its top 16 bits hold it exactly)
                                uint32_t hi4[4], lo4[4];
#pragma unroll
                                for (int f2 = 0; f2 < 4; ++f2) {
                                    const int f = m * 8 + 2 * f2;
                                    const int c0 = f / W, k0 = f % W, c1 = (f + 1) / W, k1 = (f + 1) % W;
                                    uint32_t xw0, xw1;
                                    if constexpr (W <= 4) {
                                        xw0 = (&xr[k0].x)[c0 >> 1];
                                        xw1 = (&xr[k1].x)[c1 >> 1];
                                    } else {
                                        xw0 = *reinterpret_cast<const uint32_t *>(
                                            xs + swz_b<RB>(row + (W - 1) - k0, ch0 >> 3) + (c0 >> 1) * 4);
                                        xw1 = *reinterpret_cast<const uint32_t *>(
                                            xs + swz_b<RB>(row + (W - 1) - k1, ch0 >> 3) + (c1 >> 1) * 4);
                                    }
                                    float x0 = __uint_as_float((c0 & 1) ? (xw0 & 0xffff0000u) : (xw0 << 16));
                                    float x1 = __uint_as_float((c1 & 1) ? (xw1 & 0xffff0000u) : (xw1 << 16));
                                    if (!full_taps) {
                                        x0 = k0 < nv ? x0 : 0.f;
                                        x1 = k1 < nv ? x1 : 0.f;
                                    }
                                    // G of a non-owned row is 0
                                    const float2 g = __fmul2_rn(make_float2(owned ? gy[c0] : 0.f, owned ? gy[c1] : 0.f),
                                                                make_float2(x0, x1));
                                    const uint32_t b0 = __float_as_uint(g.x), b1 = __float_as_uint(g.y);
                                    // lo = g - hi, exact (fused: g + (-1) * hi)
                                    const float2 l = __ffma2_rn(make_float2(__uint_as_float(b0 & 0xffff0000u),
                                                                            __uint_as_float(b1 & 0xffff0000u)),
                                                                make_float2(-1.f, -1.f), g);
                                    hi4[f2] = __byte_perm(b0, b1, 0x7632);
                                    lo4[f2] = __byte_perm(__float_as_uint(l.x), __float_as_uint(l.y), 0x7632);
                                }
                                const int col = gl * 8 * W + m * 8;
                                const uint32_t off = (col >> 6) * kGBlock + row * 128 +
                                                     ((((col & 63) >> 3) ^ (row & 7)) << 4);
                                *reinterpret_cast<uint4 *>(g_s + off) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
                                *reinterpret_cast<uint4 *>(g_s + kGPart + off) =
                                    make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
                            }
                            // dx over this token's dy (read above by this thread only)
                            if (owned) {
                                uint4 o;
                                o.x = pack_bf16x2(dxv[0], dxv[1]);
                                o.y = pack_bf16x2(dxv[2], dxv[3]);
                                o.z = pack_bf16x2(dxv[4], dxv[5]);
                                o.w = pack_bf16x2(dxv[6], dxv[7]);
                                *reinterpret_cast<uint4 *>(dys + dy_off) = o;
                            }
                        }
                    }
                    if (epi_abort) break;
                    // a warp without G to write still keeps step with the G buffer before it signals the step
                    if (!active) wait_or_flag(&hdr->g_empty, (k & 1) ^ 1, p.wait_ns, p.status, abort_flag);
                    // G of step k is written; after the tile's last step its dx is complete too
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&hdr->g_full);
                        if (j == NSB - 1) mbar_arrive(&hdr->dx_full[s]);
                    }
                }
                if (epi_abort) break;
                // dz partial sums of the previous tile (its MMAs have had a whole tile to finish)
                if (v > 0) {
                    const int ip = i - 1;
                    wait_or_flag(&hdr->dz_full[ip & 1], (ip >> 1) & 1, p.wait_ns, p.status, abort_flag);
                    tc_fence_after();
                    const int tp = (mt - 1) * MS + row;
                    uint32_t a[16];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        if (cc < R / 16) tmem_ld_x4(lane_base + kColDz + (ip & 1) * R + c * (R / 4) + cc * 4, a + 4 * cc);
                    tmem_ld_wait();
                    if (row < MS && tp < p.BT) {
                        float *dst = p.dz_ws + static_cast<size_t>(tp) * R + c * (R / 4);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            if (cc < R / 16)
                                red_add_v4(dst + 4 * cc, __uint_as_float(a[4 * cc]), __uint_as_float(a[4 * cc + 1]),
                                           __uint_as_float(a[4 * cc + 2]), __uint_as_float(a[4 * cc + 3]));
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
                uint32_t a[16];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    if (cc < R / 16) tmem_ld_x4(lane_base + kColDz + (ip & 1) * R + c * (R / 4) + cc * 4, a + 4 * cc);
                tmem_ld_wait();
                if (row < MS && tp < p.BT && !*abort_flag) {
                    float *dst = p.dz_ws + static_cast<size_t>(tp) * R + c * (R / 4);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        if (cc < R / 16)
                            red_add_v4(dst + 4 * cc, __uint_as_float(a[4 * cc]), __uint_as_float(a[4 * cc + 1]),
                                       __uint_as_float(a[4 * cc + 2]), __uint_as_float(a[4 * cc + 3]));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->dz_empty[ip & 1]);
                // [dU; db] accumulator: TMEM lane m < R is row m of dU, lane 64 is db; column j*SNB + n
                const bool du_row = row < R, db_row = row == 64;
                for (int cc = c * C::QDU; cc < (c + 1) * C::QDU; cc += 8) {
                    uint32_t a8[8];
                    tmem_ld_x8(lane_base + kColDu + cc, a8);
                    tmem_ld_wait();
                    const int gn0 = nb * C::NB + cc;  // a multiple of 8; N is too, so all 8 are valid or none
                    if ((du_row || db_row) && gn0 < p.N && !*abort_flag) {
                        float *dst = du_row ? p.dU + static_cast<size_t>(row) * p.N + gn0 : p.db + gn0;
                        red_add_v4(dst, __uint_as_float(a8[0]), __uint_as_float(a8[1]), __uint_as_float(a8[2]),
                                   __uint_as_float(a8[3]));
                        red_add_v4(dst + 4, __uint_as_float(a8[4]), __uint_as_float(a8[5]), __uint_as_float(a8[6]),
                                   __uint_as_float(a8[7]));
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

    // ---- teardown: nothing of this CTA may still be in flight; the dz cast kernel may start launching
    grid_dependents_launch();
    if (warp == 0 && lane == 0) {
        if (*abort_flag)
            for (int s = 0; s < kStages; ++s)
                if (issued_last[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued_last[s] / kStages) & 1, kDrainLimitNs);
        tma_store_wait_all<0>();
    }
    if (warp == 1 && lane == 0 && mma_any && *abort_flag) (void)mbar_wait(&hdr->flush, (seg - 1) & 1, kDrainLimitNs);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Zero the fp32 accumulation targets (the dz workspace, dU, db).
__global__ void lowrank_bwd_zero(float4 *a, long long na4, float4 *b, long long nb4, float *c, int nc)
{
    grid_dependents_launch();  // the backward kernel may start its loads and MMAs now
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
    grid_dependents_launch();  // the next kernel may begin its prologue
    grid_dependency_wait();    // every partial sum of the backward kernel is in
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
    // shared memory: [header][slack][U steps][bias tiles][G hi, lo][edges][stages x2][ones]
    unsigned off = 0;
    p.u_off = off;
    p.u_bytes = C::NSB * C::GB * R * 128;
    off += p.u_bytes;
    p.bt_off = align_up(off, 1024);
    off = p.bt_off + (C::NSB + 1) * C::SNB * 16;
    p.g_off = align_up(off, 1024);
    off = p.g_off + 2 * kGPart;
    p.e_off = align_up(off, 128);
    off = p.e_off + C::NCA * 4 * 2 * (W - 1) * (W - 1) * 32;
    p.st_off = align_up(off, 1024);
    p.z_bytes = 16384;
    p.x_in = p.z_bytes;
    p.x_bytes = C::XR * C::RB;
    p.dy_in = align_up(p.x_in + p.x_bytes, 1024);
    p.dy_bytes = kM * C::RB;
    p.stage_bytes = align_up(p.dy_in + p.dy_bytes, 1024);
    // the all-ones block sits above every z tile: the dU MMA reaches it from a z tile through a positive
    // leading-byte offset
    p.one_off = p.st_off + kStages * p.stage_bytes;
    const unsigned smem = 2048 + p.one_off + 4096;
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
    s = launch_overlapped(kern, grid, kThreads, smem, a.stream, tm_z, tm_x, tm_dy, tm_u, tm_dx, p);
    if (s != DSC_OK) return s;
    return launch_overlapped(lowrank_bwd_cast, dev.sm_count * 4, 256, 0, a.stream,
                             reinterpret_cast<const float4 *>(p.dz_ws), static_cast<uint4 *>(a.dz), nz / 8);
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
// device and context (host code may not use the symbol itself as an address).
static SymbolCache g_scratch_cache;
static float *noalloc_scratch() { return static_cast<float *>(symbol_address(&g_scratch_cache, &g_lrb_scratch)); }

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
