// dsc_static.cu -- the static short convolution and the decode step.
//
// Static form (notes on "Dynamic Short Convolutions Improve Transformers", section "Parameterization",
// eq. 1: one filter w[d][k] shared by every token), applied with the residual placement of eq. 3 and the
// same zero history before every sequence / packed-document start as the dynamic kernels:
//
//   y[t,d]  = x[t,d] + sum_k w[d,k] x~[t-k,d]
//   dx[s,d] = dy[s,d] + sum_{k : s lies in the document of s+k} w[d,k] dy[s+k,d]
//   dw[d,k] = sum over every token t of dy[t,d] x~[t-k,d]            (fp32)
//
// TMA path: a CTA keeps one block of kDC = 256 channels for its whole run and walks every cpb-th token
// tile of it, so the filter of its 8 channels per lane stays in registers and the backward sums its dw
// partials over all of its tiles before a single flush.  CTAs with consecutive indices hold consecutive
// channel blocks of the same token tiles, so together they stream whole rows of x (and dy).  One producer
// warp stages each tile with TMA (x with its W-1 row causal halo; in the backward dy with its W-1 row
// future halo) and the per-token valid-tap counts; consumer warps each walk RPW tokens with a register
// window of x rows (forward) or of x rows and dx accumulators (backward).
//
// Decode step (eq. 2 + eq. 3 for one new token per sequence): a per-sequence ring of the last W-1 inputs,
// slot (p mod (W-1)) holding the input at document position p; the token's position also says how much
// history its document has.  One thread per 16-byte chunk of channels: it reads the chunk's history,
// writes y, then overwrites the slot of the oldest history token with this token's input.
#include <type_traits>

#include "dsc_dense_common.cuh"
#include "dsc_tcgen05.cuh"  // named_bar

namespace dsc {

namespace stc {

// Tokens per tile and per consumer warp, and the depth of the stage ring (from measured sweeps on GB300).
// Forward: 16 warps (bf16) of 3 tokens, tiles of 48 tokens, up to 8 stages in flight.  Backward: 8 warps
// of 6 tokens -- the dx ring, the x window, the filter and the dw partials all live in registers -- and up
// to 4 stages (a deeper ring of smaller tiles was slower).
template <typename E, bool BWD>
struct Tile {
    static constexpr int TT = (sizeof(E) == 2 ? 48 : 24);
    static constexpr int RPW = BWD ? 6 : 3;
    static constexpr int NCW = TT / RPW;
    static constexpr int kStageCap = BWD ? 4 : 8;
};

struct Params {
    const void *w;
    void *out0;        // fwd: y; bwd: dx
    float *dw;         // bwd
    const int32_t *cu;
    int n_docs;
    int BT, T, D, W;
    int n_cb, n_tt, cpb;
    unsigned x_off, dy_off, nv_off, stage_bytes, tx_bytes;
    int nstages;
    int *status;
    unsigned long long wait_ns;
};

struct Plan {
    int x_rows = 0, g_rows = 0;
    unsigned x_off = 0, dy_off = 0, nv_off = 0, stage_bytes = 0, tx_bytes = 0;
    int nstages = 0, n_cb = 0, n_tt = 0, cpb = 0, grid = 0, threads = 0;
    unsigned smem = 0;
};

// Lay out the stages; false when the TMA path cannot take the arguments (the scalar path does).
inline bool make_plan(const StaticArgs &a, bool bwd, int TT, int NCW, int W, int stage_cap, const DeviceInfo &dev,
                      Plan *p)
{
    const int es = a.dt == DSC_BF16 ? 2 : 4;
    if (a.D % 8 != 0) return false;  // whole 8-channel lane vectors
    if (!aligned16(a.x) || !aligned16(a.w)) return false;
    if (bwd ? (!aligned16(a.dy) || !aligned16(a.dx)) : !aligned16(a.y)) return false;
    p->x_rows = TT + W - 1;
    p->g_rows = bwd ? TT + W - 1 : TT;
    const unsigned xb = static_cast<unsigned>(kDC * es * p->x_rows);
    const unsigned gb = bwd ? static_cast<unsigned>(kDC * es * p->g_rows) : 0u;
    unsigned off = 0;
    p->x_off = off;
    off = align_up(off + xb, 1024);
    p->dy_off = off;
    off = align_up(off + gb, 1024);
    p->nv_off = off;
    off = align_up(off + static_cast<unsigned>(p->g_rows), 1024);
    p->stage_bytes = off;
    p->tx_bytes = xb + gb;
    const unsigned header = 2048;
    const int fit = static_cast<int>((static_cast<unsigned>(dev.max_smem_optin) - header) / p->stage_bytes);
    if (fit < 2) return false;
    p->nstages = fit < stage_cap ? fit : stage_cap;
    // the backward's dw reduction reuses the stages: NCW partials of kDC * W values (fp32 for bf16 inputs,
    // fp64 for fp32 inputs)
    if (bwd && static_cast<unsigned>(NCW * kDC * W * 2 * es) > p->nstages * p->stage_bytes) return false;
    p->smem = header + p->nstages * p->stage_bytes;
    const long long BT = static_cast<long long>(a.B) * a.T;
    const long long n_tt = (BT + TT - 1) / TT;
    if (n_tt > 0x7fffffffLL) return false;
    p->n_tt = static_cast<int>(n_tt);
    p->n_cb = (a.D + kDC - 1) / kDC;
    // CTAs per channel block: as many as fill the SMs, never more than the block has tiles.  The fp32
    // backward gives each channel block to one CTA, which sums its dw in fp64 and stores it once (no fp32
    // additions across CTAs), so that dw is the exactly rounded fp64 sum up to the partials' own rounding.
    int cpb = dev.sm_count / p->n_cb;
    if (cpb < 1 || (bwd && es == 4)) cpb = 1;
    if (cpb > p->n_tt) cpb = p->n_tt;
    p->cpb = cpb;
    p->grid = cpb * p->n_cb;
    p->threads = 32 * (1 + NCW);
    return true;
}

inline Params make_params(const StaticArgs &a, const Plan &pl, void *out0, float *dw)
{
    Params q{};
    q.w = a.w;
    q.out0 = out0;
    q.dw = dw;
    q.cu = a.cu;
    q.n_docs = a.n_docs;
    q.BT = a.B * a.T;
    q.T = a.T;
    q.D = a.D;
    q.W = a.W;
    q.n_cb = pl.n_cb;
    q.n_tt = pl.n_tt;
    q.cpb = pl.cpb;
    q.x_off = pl.x_off;
    q.dy_off = pl.dy_off;
    q.nv_off = pl.nv_off;
    q.stage_bytes = pl.stage_bytes;
    q.tx_bytes = pl.tx_bytes;
    q.nstages = pl.nstages;
    q.status = device_status_word();
    q.wait_ns = wait_limit_ns();
    return q;
}

}  // namespace stc

// The filter of a lane's 8 channels as channel pairs: wp[i][k] = (w[c+2i][k], w[c+2i+1][k]).
template <typename E, int W>
__device__ __forceinline__ void static_filter(const E *w, int c, bool valid, float2 (&wp)[4][W])
{
    float wv[8 * W];
    if (valid) {
        load_n<E, 8 * W>(w + static_cast<size_t>(c) * W, wv);
    } else {
#pragma unroll
        for (int i = 0; i < 8 * W; ++i) wv[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < W; ++k) wp[i][k] = make_float2(wv[(2 * i) * W + k], wv[(2 * i + 1) * W + k]);
}

// Producer loop shared by both directions: tile `it` of this CTA is token tile j0 + it*cpb of block cb.
template <int TT, int W, bool BWD>
__device__ __forceinline__ void static_producer(const CUtensorMap *tm_x, const CUtensorMap *tm_dy, const stc::Params &p,
                                                RingHeader *hdr, uint8_t *stages, int cb, int j0, int lane,
                                                volatile int *abort_flag)
{
    constexpr int GR = BWD ? TT + W - 1 : TT;  // tokens with a valid-tap count per tile
    int issued[kMaxStages];
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) issued[s] = -1;
    bool aborted = false;
    DocCursor cursor;  // this lane's tokens increase from tile to tile
    int it = 0;
    for (int tt = j0; tt < p.n_tt; tt += p.cpb, ++it) {
        const int s = it % p.nstages;
        const uint32_t ph = (it / p.nstages) & 1;
        bool ok = mbar_wait(&hdr->empty[s], ph ^ 1, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
        if (!ok) {
            if (lane == 0) {
                record_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            aborted = true;
            break;
        }
        const int t0 = tt * TT;
        uint8_t *st = stages + s * p.stage_bytes;
        int8_t *nv = reinterpret_cast<int8_t *>(st + p.nv_off);
        if (BWD && it > 0) cursor.reset();  // the future halo rows run ahead of the next tile's first rows
        for (int r = lane; r < GR; r += 32) {
            const int t = t0 + r;
            nv[r] = static_cast<int8_t>(t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(&hdr->full[s], p.tx_bytes);
            tma_load_2d(st + p.x_off, tm_x, &hdr->full[s], cb * kDC, t0 - (W - 1));
            if constexpr (BWD) tma_load_2d(st + p.dy_off, tm_dy, &hdr->full[s], cb * kDC, t0);
            issued[s] = it;
        }
    }
    if (aborted && lane == 0) {
        for (int s = 0; s < p.nstages; ++s)
            if (issued[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued[s] / p.nstages) & 1, kDrainLimitNs);
    }
}

template <typename E, int W>
__global__ void __launch_bounds__(32 * (1 + stc::Tile<E, false>::NCW), 1)
    static_fwd_tma(const __grid_constant__ CUtensorMap tm_x, const stc::Params p)
{
    using Tl = stc::Tile<E, false>;
    constexpr int TT = Tl::TT, RPW = Tl::RPW, NCW = Tl::NCW;
    extern __shared__ __align__(1024) uint8_t smem[];
    RingHeader *hdr = reinterpret_cast<RingHeader *>(smem);
    uint8_t *stages = stage_base(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], NCW);
        }
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    // this launch may overlap the end of the stream's previous kernel: every access to global memory
    // comes after the wait; the next kernel may begin its own prologue as soon as this one runs
    grid_dependents_launch();
    grid_dependency_wait();
    volatile int *abort_flag = &hdr->abort_flag;
    const int cb = blockIdx.x % p.n_cb, j0 = blockIdx.x / p.n_cb;

    if (warp == 0) {
        if (lane == 0) prefetch_tmap(&tm_x);
        static_producer<TT, W, false>(&tm_x, nullptr, p, hdr, stages, cb, j0, lane, abort_flag);
    } else {
        const int r0 = (warp - 1) * RPW;
        const int c = cb * kDC + lane * 8;
        const bool cvalid = c < p.D;
        float2 wp[4][W];
        static_filter<E, W>(static_cast<const E *>(p.w), c, cvalid, wp);
        E *y = static_cast<E *>(p.out0);
        int it = 0;
        for (int tt = j0; tt < p.n_tt; tt += p.cpb, ++it) {
            const int s = it % p.nstages;
            const uint32_t ph = (it / p.nstages) & 1;
            bool ok = mbar_wait(&hdr->full[s], ph, p.wait_ns);
            ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
            if (!ok) {
                if (lane == 0) {
                    record_status(p.status, kStatusTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            const int t0 = tt * TT;
            const uint8_t *st = stages + s * p.stage_bytes;
            const E *xs = reinterpret_cast<const E *>(st + p.x_off) + lane * 8;  // row i <-> token t0-(W-1)+i
            const int8_t *nvs = reinterpret_cast<const int8_t *>(st + p.nv_off);
            // x window as a ring: the row of step r (token t0+r0+r) sits in slot ring(r, W)
            float2 xw[W][4];
#pragma unroll
            for (int r = -(W - 1); r < 0; ++r) load8x2(xs + (r0 + r + W - 1) * kDC, xw[ring(r, W)]);
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int j = r0 + r;
                load8x2(xs + (j + W - 1) * kDC, xw[ring(r, W)]);
                const int nv = nvs[j];
                float2 out[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) out[i] = xw[ring(r, W)][i];  // residual
                if (nv == W) {
#pragma unroll
                    for (int k = 0; k < W; ++k)
#pragma unroll
                        for (int i = 0; i < 4; ++i) out[i] = fma2(wp[i][k], xw[ring(r - k, W)][i], out[i]);
                } else {
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        if (k < nv) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) out[i] = fma2(wp[i][k], xw[ring(r - k, W)][i], out[i]);
                        }
                }
                const int t = t0 + j;
                if (cvalid && t < p.BT) store8x2(y + static_cast<size_t>(t) * p.D + c, out);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdr->empty[s]);
        }
    }
}

template <typename E, int W>
__global__ void __launch_bounds__(32 * (1 + stc::Tile<E, true>::NCW), 1)
    static_bwd_tma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                   const stc::Params p)
{
    using Tl = stc::Tile<E, true>;
    constexpr int TT = Tl::TT, RPW = Tl::RPW, NCW = Tl::NCW;
    extern __shared__ __align__(1024) uint8_t smem[];
    RingHeader *hdr = reinterpret_cast<RingHeader *>(smem);
    uint8_t *stages = stage_base(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&hdr->full[s], 1);
            mbar_init(&hdr->empty[s], NCW);
        }
        hdr->abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    // may overlap the previous kernel (the one that zeroes dw): global accesses come after the wait
    grid_dependents_launch();
    grid_dependency_wait();
    volatile int *abort_flag = &hdr->abort_flag;
    const int cb = blockIdx.x % p.n_cb, j0 = blockIdx.x / p.n_cb;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_dy);
        }
        static_producer<TT, W, true>(&tm_x, &tm_dy, p, hdr, stages, cb, j0, lane, abort_flag);
        return;  // the dw reduction below is the consumers' alone
    }
    const int r0 = (warp - 1) * RPW;
    const int c = cb * kDC + lane * 8;
    const bool cvalid = c < p.D;
    float2 wp[4][W];
    static_filter<E, W>(static_cast<const E *>(p.w), c, cvalid, wp);
    E *dx = static_cast<E *>(p.out0);
    // dw partials of this lane's 8 channels, summed over every token this warp sees: fp32 pairs for bf16
    // inputs (exact products), fp64 for fp32 inputs
    using Acc = typename std::conditional<std::is_same<E, float>::value, double, float>::type;
    Acc dwp[8][W];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < W; ++k) dwp[i][k] = Acc(0);
    int it = 0;
    for (int tt = j0; tt < p.n_tt; tt += p.cpb, ++it) {
        const int s = it % p.nstages;
        const uint32_t ph = (it / p.nstages) & 1;
        bool ok = mbar_wait(&hdr->full[s], ph, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok) && (*abort_flag == 0);
        if (!ok) {
            if (lane == 0) {
                record_status(p.status, kStatusTimeout);
                *abort_flag = 1;
            }
            break;
        }
        const int t0 = tt * TT;
        const uint8_t *st = stages + s * p.stage_bytes;
        const E *xs = reinterpret_cast<const E *>(st + p.x_off) + lane * 8;   // row i <-> token t0-(W-1)+i
        const E *gs = reinterpret_cast<const E *>(st + p.dy_off) + lane * 8;  // row i <-> token t0+i
        const int8_t *nvs = reinterpret_cast<const int8_t *>(st + p.nv_off);
        // rings indexed by step r (token t0+r0+r): the x window and the dx accumulators
        float2 xw[W][4];
        float2 acc[W][4];
#pragma unroll
        for (int r = -(W - 1); r < 0; ++r) load8x2(xs + (r0 + r + W - 1) * kDC, xw[ring(r, W)]);
#pragma unroll
        for (int k = 0; k < W; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[k][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < RPW + W - 1; ++r) {
            const int j = r0 + r;
            float2 g[4];
            load8x2(gs + j * kDC, g);
            const int nv = nvs[j];
            // dx: the residual opens this token's slot; w[k] * dy[j] goes to token j-k
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[ring(r, W)][i] = g[i];
#pragma unroll
            for (int k = 0; k < W; ++k)
                if (k < nv) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[ring(r - k, W)][i] = fma2(wp[i][k], g[i], acc[ring(r - k, W)][i]);
                }
            if (r >= W - 1) {  // the token of step r-(W-1) has received all of its terms
                const int tdx = t0 + j - (W - 1);
                if (cvalid && tdx < p.BT) store8x2(dx + static_cast<size_t>(tdx) * p.D + c, acc[ring(r - (W - 1), W)]);
            }
            if (r < RPW) {  // dw: dy[j] * x~[j-k] for the taps inside token j's document
                load8x2(xs + (j + W - 1) * kDC, xw[ring(r, W)]);
#pragma unroll
                for (int k = 0; k < W; ++k)
                    if (k < nv) {
                        if constexpr (std::is_same<Acc, float>::value) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 v = fma2(g[i], xw[ring(r - k, W)][i], make_float2(dwp[2 * i][k], dwp[2 * i + 1][k]));
                                dwp[2 * i][k] = v.x;
                                dwp[2 * i + 1][k] = v.y;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                dwp[2 * i][k] = fma(static_cast<double>(g[i].x), static_cast<double>(xw[ring(r - k, W)][i].x), dwp[2 * i][k]);
                                dwp[2 * i + 1][k] = fma(static_cast<double>(g[i].y), static_cast<double>(xw[ring(r - k, W)][i].y), dwp[2 * i + 1][k]);
                            }
                        }
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hdr->empty[s]);
    }

    // dw: the consumer warps' partials meet in shared memory (the stages are idle now: every tile this CTA
    // loaded has been consumed), then one fp32 addition per (channel, tap) of the block
    named_bar(1, NCW * 32);
    Acc *red = reinterpret_cast<Acc *>(stages);  // [NCW][kDC][W]
    Acc *mine = red + (warp - 1) * (kDC * W) + lane * 8 * W;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < W; ++k) mine[i * W + k] = dwp[i][k];
    named_bar(1, NCW * 32);
    if (*abort_flag) return;
    for (int e = threadIdx.x - 32; e < kDC * W; e += NCW * 32) {
        const int ch = cb * kDC + e / W;
        if (ch >= p.D) continue;
        Acc sum = Acc(0);
#pragma unroll
        for (int q = 0; q < NCW; ++q) sum += red[q * (kDC * W) + e];
        atomicAdd(p.dw + static_cast<size_t>(cb) * kDC * W + e, static_cast<float>(sum));
    }
}

// ------------------------------------------------------------------ scalar paths (any shape / alignment)

template <typename E>
__global__ void static_fwd_scalar(const E *__restrict__ x, const E *__restrict__ w, E *__restrict__ y, int BT, int T,
                                  int D, int W, const int32_t *cu, int n_docs)
{
    grid_dependency_wait();
    const long long n = static_cast<long long>(BT) * D;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / D), d = static_cast<int>(i - static_cast<long long>(t) * D);
        const int nv = valid_taps(t, T, W, cu, n_docs);
        float acc = Elem<E>::to_f(x[i]);
        for (int k = 0; k < nv; ++k)
            acc = fmaf(Elem<E>::to_f(w[d * W + k]), Elem<E>::to_f(x[i - static_cast<long long>(k) * D]), acc);
        y[i] = Elem<E>::from_f(acc);
    }
}

template <typename E>
__global__ void static_bwd_dx_scalar(const E *__restrict__ w, const E *__restrict__ dy, E *__restrict__ dx, int BT,
                                     int T, int D, int W, const int32_t *cu, int n_docs)
{
    grid_dependency_wait();
    const long long n = static_cast<long long>(BT) * D;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i / D), d = static_cast<int>(i - static_cast<long long>(s) * D);
        float acc = Elem<E>::to_f(dy[i]);
        for (int k = 0; k < W && s + k < BT; ++k)
            if (k < valid_taps(s + k, T, W, cu, n_docs))
                acc = fmaf(Elem<E>::to_f(w[d * W + k]), Elem<E>::to_f(dy[i + static_cast<long long>(k) * D]), acc);
        dx[i] = Elem<E>::from_f(acc);
    }
}

template <typename E>
__global__ void static_bwd_dw_scalar(const E *__restrict__ x, const E *__restrict__ dy, float *__restrict__ dw, int BT,
                                     int T, int D, int W, const int32_t *cu, int n_docs)
{
    grid_dependency_wait();  // dw was zeroed two launches ago
    const long long n = static_cast<long long>(BT) * D;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / D), d = static_cast<int>(i - static_cast<long long>(t) * D);
        const int nv = valid_taps(t, T, W, cu, n_docs);
        const float g = Elem<E>::to_f(dy[i]);
        for (int k = 0; k < nv; ++k)
            atomicAdd(dw + d * W + k, g * Elem<E>::to_f(x[i - static_cast<long long>(k) * D]));
    }
}

// fp32 inputs: one thread per (channel, tap) sums every token in fp64 and stores once
__global__ void static_bwd_dw_scalar_f64(const float *__restrict__ x, const float *__restrict__ dy,
                                         float *__restrict__ dw, int BT, int T, int D, int W, const int32_t *cu,
                                         int n_docs)
{
    grid_dependency_wait();  // dw was zeroed two launches ago
    const int n = D * W;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
        const int d = e / W, k = e - d * W;
        double acc = 0.0;
        for (int t = 0; t < BT; ++t)
            if (k < valid_taps(t, T, W, cu, n_docs))
                acc = fma(static_cast<double>(dy[static_cast<size_t>(t) * D + d]),
                          static_cast<double>(x[static_cast<size_t>(t - k) * D + d]), acc);
        dw[e] = static_cast<float>(acc);
    }
}

__global__ void static_zero(float *a, int n)
{
    grid_dependency_wait();
    grid_dependents_launch();  // the backward kernel may start its prologue
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) a[i] = 0.f;
}

// ------------------------------------------------------------------ decode step

// V consecutive elements as fp32 (V = 16 bytes of elements on the vector path, 1 on the scalar path).
template <typename E, int V>
__device__ __forceinline__ void load_v(const E *p, float (&v)[V])
{
    load_n<E, V>(p, v);
}

// The filter values of a chunk's V channels, tap k of channel v at f[v][k].  HM says how the chunk meets
// the heads: 1 -- one head holds all V channels (H % V == 0): its W taps are read once; 2 -- every channel
// is its own head (H == 1): V*W consecutive values; 0 -- anything else, one value at a time.
template <typename E, int V, int HM, int WM>
__device__ __forceinline__ void decode_filter(const E *wb, int c, int W, int H, float (&f)[V][WM])
{
    if constexpr (HM == 1) {
        float t[WM];
        const E *p = wb + (c / H) * W;
#pragma unroll
        for (int k = 0; k < WM; ++k) t[k] = k < W ? Elem<E>::to_f(p[k]) : 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int k = 0; k < WM; ++k) f[v][k] = t[k];
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int k = 0; k < WM; ++k)
                f[v][k] = k < W ? Elem<E>::to_f(wb[(HM == 2 ? (c + v) : (c + v) / H) * W + k]) : 0.f;
    }
}

template <typename E, int V, int HM, int W>
__global__ void __launch_bounds__(256) decode_step_kernel(const E *__restrict__ x, const E *__restrict__ w,
                                                          E *__restrict__ hist, const int32_t *__restrict__ pos,
                                                          E *__restrict__ y, int B, int D, int H, int *status)
{
    grid_dependents_launch();
    grid_dependency_wait();
    const int chunks = D / V;
    const int G = D / H;
    static_assert(W >= 1 && W <= 8, "filter width");
    const long long n = static_cast<long long>(B) * chunks;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(i / chunks);
        const int c = static_cast<int>(i - static_cast<long long>(b) * chunks) * V;
        // every ring slot is loaded at once, before the position is known (the addresses do not depend on
        // it); slot s then holds tap k = (pos - s) mod (W-1) (W-1 where that is 0), used when k <= pos
        E *hb = hist + static_cast<size_t>(b) * (W - 1) * D + c;
        float hv[W > 1 ? W - 1 : 1][V];
#pragma unroll
        for (int sl = 0; sl + 1 < W; ++sl) load_v<E, V>(hb + static_cast<size_t>(sl) * D, hv[sl]);
        float xv[V], acc[V];
        load_v<E, V>(x + static_cast<size_t>(b) * D + c, xv);
        float f[V][W];
        decode_filter<E, V, HM, W>(w + static_cast<size_t>(b) * G * W, c, W, H, f);
        int p = pos[b];
        if (p < 0) {  // not a position: treated as a document start, and reported
            record_status(status, kStatusInvalid);
            p = 0;
        }
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = fmaf(f[v][0], xv[v], xv[v]);
        if constexpr (W > 1) {
            const int pm = p % (W - 1);
#pragma unroll
            for (int sl = 0; sl + 1 < W; ++sl) {
                int k = pm - sl;
                k = k <= 0 ? k + (W - 1) : k;  // 1 .. W-1
                if (k <= p) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        float fk = f[v][1];
#pragma unroll
                        for (int kk = 2; kk < W; ++kk) fk = k == kk ? f[v][kk] : fk;
                        acc[v] = fmaf(fk, hv[sl][v], acc[v]);
                    }
                }
            }
        }
        store_n<E, V>(y + static_cast<size_t>(b) * D + c, acc);
        // every history read of this chunk is done: this token's input takes the oldest slot
        if (W > 1) store_n<E, V>(hb + static_cast<size_t>(p % (W - 1)) * D, xv);
    }
}

// ------------------------------------------------------------------ host side

template <typename E, int W>
static dsc_status launch_static_fwd(const StaticArgs &a, const DeviceInfo &dev)
{
    using Tl = stc::Tile<E, false>;
    stc::Plan pl;
    if (!stc::make_plan(a, false, Tl::TT, Tl::NCW, W, Tl::kStageCap, dev, &pl)) return DSC_ERR_UNSUPPORTED;
    const CUtensorMapDataType tdt = sizeof(E) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const unsigned long long BT = static_cast<unsigned long long>(a.B) * a.T;
    CUtensorMap tm_x;
    if (!encode_tmap_2d(&tm_x, a.x, tdt, a.D, BT, static_cast<unsigned long long>(a.D) * sizeof(E), kDC, pl.x_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_UNSUPPORTED;
    auto kern = static_fwd_tma<E, W>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    return launch_overlapped(kern, pl.grid, pl.threads, pl.smem, a.stream, tm_x, stc::make_params(a, pl, a.y, nullptr));
}

template <typename E, int W>
static dsc_status launch_static_bwd(const StaticArgs &a, const DeviceInfo &dev)
{
    using Tl = stc::Tile<E, true>;
    stc::Plan pl;
    if (!stc::make_plan(a, true, Tl::TT, Tl::NCW, W, Tl::kStageCap, dev, &pl)) return DSC_ERR_UNSUPPORTED;
    const CUtensorMapDataType tdt = sizeof(E) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const unsigned long long BT = static_cast<unsigned long long>(a.B) * a.T;
    const unsigned long long row = static_cast<unsigned long long>(a.D) * sizeof(E);
    CUtensorMap tm_x, tm_dy;
    if (!encode_tmap_2d(&tm_x, a.x, tdt, a.D, BT, row, kDC, pl.x_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&tm_dy, a.dy, tdt, a.D, BT, row, kDC, pl.g_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_UNSUPPORTED;
    auto kern = static_bwd_tma<E, W>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem) != cudaSuccess)
        return DSC_ERR_CUDA;
    const int nw = a.D * a.W;
    dsc_status s = launch_overlapped(static_zero, static_cast<unsigned>((nw + 255) / 256), 256u, 0, a.stream, a.dw, nw);
    if (s != DSC_OK) return s;
    return launch_overlapped(kern, pl.grid, pl.threads, pl.smem, a.stream, tm_x, tm_dy,
                             stc::make_params(a, pl, a.dx, a.dw));
}

template <typename E>
static dsc_status static_fwd_t(const StaticArgs &a, const DeviceInfo &dev)
{
    dsc_status s = DSC_ERR_INVALID_ARG;
    switch (a.W) {
    case 1: s = launch_static_fwd<E, 1>(a, dev); break;
    case 2: s = launch_static_fwd<E, 2>(a, dev); break;
    case 3: s = launch_static_fwd<E, 3>(a, dev); break;
    case 4: s = launch_static_fwd<E, 4>(a, dev); break;
    case 5: s = launch_static_fwd<E, 5>(a, dev); break;
    case 6: s = launch_static_fwd<E, 6>(a, dev); break;
    case 7: s = launch_static_fwd<E, 7>(a, dev); break;
    case 8: s = launch_static_fwd<E, 8>(a, dev); break;
    default: return DSC_ERR_INVALID_ARG;
    }
    if (s != DSC_ERR_UNSUPPORTED) return s;
    const long long n = static_cast<long long>(a.B) * a.T * a.D;
    long long blocks = (n + 255) / 256;
    if (blocks > static_cast<long long>(dev.sm_count) * 8) blocks = static_cast<long long>(dev.sm_count) * 8;
    return launch_overlapped(static_fwd_scalar<E>, static_cast<unsigned>(blocks), 256u, 0, a.stream,
                             static_cast<const E *>(a.x), static_cast<const E *>(a.w), static_cast<E *>(a.y),
                             a.B * a.T, a.T, a.D, a.W, a.cu, a.n_docs);
}

template <typename E>
static dsc_status static_bwd_t(const StaticArgs &a, const DeviceInfo &dev)
{
    dsc_status s = DSC_ERR_INVALID_ARG;
    switch (a.W) {
    case 1: s = launch_static_bwd<E, 1>(a, dev); break;
    case 2: s = launch_static_bwd<E, 2>(a, dev); break;
    case 3: s = launch_static_bwd<E, 3>(a, dev); break;
    case 4: s = launch_static_bwd<E, 4>(a, dev); break;
    case 5: s = launch_static_bwd<E, 5>(a, dev); break;
    case 6: s = launch_static_bwd<E, 6>(a, dev); break;
    case 7: s = launch_static_bwd<E, 7>(a, dev); break;
    case 8: s = launch_static_bwd<E, 8>(a, dev); break;
    default: return DSC_ERR_INVALID_ARG;
    }
    if (s != DSC_ERR_UNSUPPORTED) return s;
    const long long n = static_cast<long long>(a.B) * a.T * a.D;
    long long blocks = (n + 255) / 256;
    if (blocks > static_cast<long long>(dev.sm_count) * 8) blocks = static_cast<long long>(dev.sm_count) * 8;
    const int nw = a.D * a.W;
    s = launch_overlapped(static_zero, static_cast<unsigned>((nw + 255) / 256), 256u, 0, a.stream, a.dw, nw);
    if (s != DSC_OK) return s;
    s = launch_overlapped(static_bwd_dx_scalar<E>, static_cast<unsigned>(blocks), 256u, 0, a.stream,
                          static_cast<const E *>(a.w), static_cast<const E *>(a.dy), static_cast<E *>(a.dx), a.B * a.T,
                          a.T, a.D, a.W, a.cu, a.n_docs);
    if (s != DSC_OK) return s;
    // dx and dw are independent; the dw kernel follows the zeroing in stream order
    if constexpr (std::is_same<E, float>::value)
        return launch_overlapped(static_bwd_dw_scalar_f64, static_cast<unsigned>((nw + 127) / 128), 128u, 0, a.stream,
                                 a.x == nullptr ? nullptr : static_cast<const float *>(a.x),
                                 static_cast<const float *>(a.dy), a.dw, a.B * a.T, a.T, a.D, a.W, a.cu, a.n_docs);
    else
        return launch_overlapped(static_bwd_dw_scalar<E>, static_cast<unsigned>(blocks), 256u, 0, a.stream,
                                 static_cast<const E *>(a.x), static_cast<const E *>(a.dy), a.dw, a.B * a.T, a.T, a.D,
                                 a.W, a.cu, a.n_docs);
}

dsc_status static_fwd(const StaticArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    return a.dt == DSC_BF16 ? static_fwd_t<__nv_bfloat16>(a, dev) : static_fwd_t<float>(a, dev);
}

dsc_status static_bwd(const StaticArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    return a.dt == DSC_BF16 ? static_bwd_t<__nv_bfloat16>(a, dev) : static_bwd_t<float>(a, dev);
}

template <typename E, int V, int W>
static dsc_status decode_launch(const DecodeArgs &a, unsigned nb, int *st, bool vec)
{
    const E *x = static_cast<const E *>(a.x), *w = static_cast<const E *>(a.w);
    E *h = static_cast<E *>(a.hist), *y = static_cast<E *>(a.y);
    if (!vec) return launch_overlapped(decode_step_kernel<E, 1, 0, W>, nb, 256u, 0, a.stream, x, w, h, a.pos, y, a.B, a.D, a.H, st);
    if (a.H % V == 0)
        return launch_overlapped(decode_step_kernel<E, V, 1, W>, nb, 256u, 0, a.stream, x, w, h, a.pos, y, a.B, a.D, a.H, st);
    if (a.H == 1)
        return launch_overlapped(decode_step_kernel<E, V, 2, W>, nb, 256u, 0, a.stream, x, w, h, a.pos, y, a.B, a.D, a.H, st);
    return launch_overlapped(decode_step_kernel<E, V, 0, W>, nb, 256u, 0, a.stream, x, w, h, a.pos, y, a.B, a.D, a.H, st);
}

template <typename E>
static dsc_status decode_t(const DecodeArgs &a, const DeviceInfo &dev)
{
    constexpr int V = 16 / sizeof(E);
    const bool vec = a.D % V == 0 && aligned16(a.x) && aligned16(a.y) && aligned16(a.hist);
    const long long n = static_cast<long long>(a.B) * (vec ? a.D / V : a.D);
    long long blocks = (n + 255) / 256;
    if (blocks > static_cast<long long>(dev.sm_count) * 16) blocks = static_cast<long long>(dev.sm_count) * 16;
    int *st = device_status_word();
    if (!st) return DSC_ERR_CUDA;
    const unsigned nb = static_cast<unsigned>(blocks);
    switch (a.W) {
    case 1: return decode_launch<E, V, 1>(a, nb, st, vec);
    case 2: return decode_launch<E, V, 2>(a, nb, st, vec);
    case 3: return decode_launch<E, V, 3>(a, nb, st, vec);
    case 4: return decode_launch<E, V, 4>(a, nb, st, vec);
    case 5: return decode_launch<E, V, 5>(a, nb, st, vec);
    case 6: return decode_launch<E, V, 6>(a, nb, st, vec);
    case 7: return decode_launch<E, V, 7>(a, nb, st, vec);
    case 8: return decode_launch<E, V, 8>(a, nb, st, vec);
    default: return DSC_ERR_INVALID_ARG;
    }
}

dsc_status decode_step(const DecodeArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    return a.dt == DSC_BF16 ? decode_t<__nv_bfloat16>(a, dev) : decode_t<float>(a, dev);
}

}  // namespace dsc
