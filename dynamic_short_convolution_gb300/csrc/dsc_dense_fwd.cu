// dsc_dense_fwd.cu -- forward pass, materialised (H = 1) and head-wise (H > 1)
// filters: y[t,d] = x[t,d] + sum_{k<W} w[t, d/H, k] * x~[t-k, d]
// (notes on "Dynamic Short Convolutions Improve Transformers",
// "Parameterization" eq. 2 with the residual of eq. 3; the kernel reads x and
// w once and writes y once, as section "Efficient training" describes).
//
// TMA path: per tile the producer warp stages x rows [t0-(W-1), t0+TT) -- the
// causal halo plus the tile, rows before token 0 arrive zero-filled -- and
// the tile's filter rows, and computes each token's valid-tap count from the
// packed-document offsets.  Each consumer warp walks its RPW tokens with a
// register sliding window of the last W x rows, so every x element is read
// from shared memory once per warp.  fp32 accumulation, one 16-byte vector
// store per lane and token.
#include "dsc_dense_common.cuh"

namespace dsc {

template <typename E, int W, int HPT, bool WIDE>
__global__ void __launch_bounds__(32 * (1 + TileCfg<E, HPT, false, WIDE>::NCW), 1)
    dense_fwd_tma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const DenseParams p)
{
    using Cfg = TileCfg<E, HPT, false, WIDE>;
    constexpr int TT = Cfg::TT, RPW = Cfg::RPW, NCW = Cfg::NCW;
    constexpr int NWV = HPT * W;  // filter values per lane and token

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

    if (warp == 0) {
        // ---------------- producer: stage tiles, compute valid-tap counts
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_w);
        }
        int issued[kMaxStages];
#pragma unroll
        for (int s = 0; s < kMaxStages; ++s) issued[s] = -1;
        bool aborted = false;
        DocCursor cursor;  // this CTA's tiles come in increasing token order
        int it = 0;
        for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++it) {
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
            const int tt = tile / p.n_cb, cb = tile - tt * p.n_cb;
            const int t0 = tt * TT;
            uint8_t *st = stages + s * p.stage_bytes;
            int8_t *nv = reinterpret_cast<int8_t *>(st + p.nv_off);
            for (int r = lane; r < TT; r += 32) {
                const int t = t0 + r;
                nv[r] = static_cast<int8_t>(t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&hdr->full[s], p.tx_bytes);
                tma_load_2d(st + p.x_off, &tm_x, &hdr->full[s], cb * kDC, t0 - (W - 1));
                for (int b = 0; b < p.w_nboxes; ++b)
                    tma_load_2d(st + p.w_off + b * p.w_box_stride, &tm_w, &hdr->full[s],
                                cb * p.w_blk + b * p.w_box, t0);
                issued[s] = it;
            }
        }
        if (aborted && lane == 0) {
            // let every copy this CTA started land before the CTA exits
            for (int s = 0; s < p.nstages; ++s)
                if (issued[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued[s] / p.nstages) & 1, kDrainLimitNs);
        }
    } else {
        // ---------------- consumers
        const int r0 = (warp - 1) * RPW;
        const int wstart = ((lane * 8) >> p.hshift) * W;  // first filter value of this lane's channels
        const int wb = wstart / p.w_box;
        const int wo = wstart - wb * p.w_box;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++it) {
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
            const int tt = tile / p.n_cb, cb = tile - tt * p.n_cb;
            const int t0 = tt * TT;
            const uint8_t *st = stages + s * p.stage_bytes;
            const E *xs = reinterpret_cast<const E *>(st + p.x_off) + lane * 8;  // row i <-> token t0-(W-1)+i
            const E *ws = reinterpret_cast<const E *>(st + p.w_off + wb * p.w_box_stride) + wo;
            const int8_t *nvs = reinterpret_cast<const int8_t *>(st + p.nv_off);
            const int c = cb * kDC + lane * 8;
            const bool cvalid = c < p.D;
            E *y = reinterpret_cast<E *>(p.out0);

            // x window as a ring: the row of step r (token t0+r0+r) sits in slot ring(r, W)
            float2 xw[W][4];
#pragma unroll
            for (int r = -(W - 1); r < 0; ++r) load8x2(xs + (r0 + r + W - 1) * kDC, xw[ring(r, W)]);
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const int j = r0 + r;  // tile-local token
                load8x2(xs + (j + W - 1) * kDC, xw[ring(r, W)]);
                float wv[NWV];
                load_n<E, NWV>(ws + j * p.w_box, wv);
                float2 wp[4][W];
                filter_pairs<HPT, W>(wv, wp);
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

// Scalar path for any shape the TMA path cannot take: one thread per output element.
template <typename E>
__global__ void dense_fwd_scalar(const E *__restrict__ x, const E *__restrict__ w, E *__restrict__ y, int BT, int T,
                                 int D, int W, int H, const int32_t *cu, int n_docs)
{
    const long long n = static_cast<long long>(BT) * D;
    const int G = D / H;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / D), d = static_cast<int>(i - static_cast<long long>(t) * D);
        const int nv = valid_taps(t, T, W, cu, n_docs);
        const E *wt = w + (static_cast<long long>(t) * G + d / H) * W;
        float acc = Elem<E>::to_f(x[i]);
        for (int k = 0; k < nv; ++k) acc = fmaf(Elem<E>::to_f(wt[k]), Elem<E>::to_f(x[i - static_cast<long long>(k) * D]), acc);
        y[i] = Elem<E>::from_f(acc);
    }
}

template <typename E, int W, int HPT, bool WIDE = false>
static dsc_status launch_fwd_tma(const DenseArgs &a, const DeviceInfo &dev)
{
    using Cfg = TileCfg<E, HPT, false, WIDE>;
    DensePlan plan;
    if (!make_dense_plan(a, false, Cfg::TT, Cfg::RPW, Cfg::kStageCap, dev, &plan)) return DSC_ERR_UNSUPPORTED;
    const CUtensorMapDataType tdt =
        sizeof(E) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const unsigned long long BT = static_cast<unsigned long long>(a.B) * a.T;
    const unsigned long long G = a.D / a.H;
    CUtensorMap tm_x, tm_w;
    if (!encode_tmap_2d(&tm_x, a.x, tdt, a.D, BT, static_cast<unsigned long long>(a.D) * sizeof(E), kDC,
                        plan.x_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_UNSUPPORTED;
    if (!encode_tmap_2d(&tm_w, a.w, tdt, G * a.W, BT, G * a.W * sizeof(E), plan.w_box, plan.g_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_UNSUPPORTED;  // descriptor rejected: the scalar path takes the call
    auto kern = dense_fwd_tma<E, W, HPT, WIDE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes);
    if (e != cudaSuccess) return DSC_ERR_CUDA;
    const DenseParams q = dense_params(a, plan, a.y, nullptr);
    return launch_overlapped(kern, plan.grid, plan.threads, plan.smem_bytes, a.stream, tm_x, tm_w, q);
}

// Tokens the busiest CTA of a one-CTA-per-SM grid carries with tiles of tt tokens.
static long long busiest_cta_tokens(const DenseArgs &a, int tt, int sm_count)
{
    const long long n_tiles = ((static_cast<long long>(a.B) * a.T + tt - 1) / tt) * ((a.D + kDC - 1) / kDC);
    return ((n_tiles + sm_count - 1) / sm_count) * tt;
}

// bf16, H >= 8: 64-token tiles, unless 48-token tiles balance the grid better
// by more than 2% (measured: 64-token tiles are 9% faster on 4 x 8192 packed
// tokens x 3072 channels, 48-token tiles 4% faster on 8 x 2048 x 2048, where
// the last wave of 64-token tiles is half empty).
template <typename E, int W>
static dsc_status fwd_headwise(const DenseArgs &a, const DeviceInfo &dev)
{
    if constexpr (sizeof(E) == 2) {
        const long long n48 = busiest_cta_tokens(a, 48, dev.sm_count);
        const long long n64 = busiest_cta_tokens(a, 64, dev.sm_count);
        if (n48 * 50 >= n64 * 49) return launch_fwd_tma<E, W, 1, true>(a, dev);
    }
    return launch_fwd_tma<E, W, 1>(a, dev);
}

template <typename E, int W>
static dsc_status fwd_by_hpt(const DenseArgs &a, const DeviceInfo &dev)
{
    switch (a.H) {
    case 1: return launch_fwd_tma<E, W, 8>(a, dev);
    case 2: return launch_fwd_tma<E, W, 4>(a, dev);
    case 4: return launch_fwd_tma<E, W, 2>(a, dev);
    default: return fwd_headwise<E, W>(a, dev);
    }
}

template <typename E>
static dsc_status fwd_tma(const DenseArgs &a, const DeviceInfo &dev)
{
    switch (a.W) {
    case 1: return fwd_by_hpt<E, 1>(a, dev);
    case 2: return fwd_by_hpt<E, 2>(a, dev);
    case 3: return fwd_by_hpt<E, 3>(a, dev);
    case 4: return fwd_by_hpt<E, 4>(a, dev);
    case 5: return fwd_by_hpt<E, 5>(a, dev);
    case 6: return fwd_by_hpt<E, 6>(a, dev);
    case 7: return fwd_by_hpt<E, 7>(a, dev);
    case 8: return fwd_by_hpt<E, 8>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

template <typename E>
static dsc_status fwd_scalar(const DenseArgs &a, const DeviceInfo &dev)
{
    const long long n = static_cast<long long>(a.B) * a.T * a.D;
    long long blocks = (n + 255) / 256;
    const long long cap = static_cast<long long>(dev.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    dense_fwd_scalar<E><<<static_cast<int>(blocks), 256, 0, a.stream>>>(
        static_cast<const E *>(a.x), static_cast<const E *>(a.w), static_cast<E *>(a.y), a.B * a.T, a.T, a.D, a.W,
        a.H, a.cu, a.n_docs);
    return launched();
}

// Path selection: the TMA kernel whenever its alignment rules hold, else the scalar kernel.
dsc_status dense_fwd(const DenseArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    const dsc_status s = a.dt == DSC_BF16 ? fwd_tma<__nv_bfloat16>(a, dev) : fwd_tma<float>(a, dev);
    if (s != DSC_ERR_UNSUPPORTED) return s;
    return a.dt == DSC_BF16 ? fwd_scalar<__nv_bfloat16>(a, dev) : fwd_scalar<float>(a, dev);
}

}  // namespace dsc
