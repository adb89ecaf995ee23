// dsc_dense_bwd.cu -- backward pass of the materialised / head-wise dynamic
// short convolution, one pass producing both gradients:
//   dx[s,d]   = dy[s,d] + sum_{k<W, s+k in s's document} w[s+k, d/H, k] * dy[s+k, d]
//   dw[t,g,k] = sum_{d : d/H = g} dy[t,d] * x~[t-k, d]
// (the derivative of eq. 2 + eq. 3 in the notes on "Dynamic Short
// Convolutions Improve Transformers", "Parameterization" / "Placement").
//
// TMA path: per tile of TT tokens the producer stages x rows [t0-(W-1), t0+TT)
// (past halo for dw) and dy / w rows [t0, t0+TT+W-1) (future halo for dx);
// rows outside the tensor arrive zero-filled.  A consumer warp walks its
// tokens in ascending order once: a register window of the last W x rows
// gives dw (head sums across lanes with __shfl_xor), and a W-slot ring of dx
// accumulators receives w[t,k] * dy[t] for the token t-k; the slot of token
// t-(W-1) is complete after step t and is stored.
#include "dsc_dense_common.cuh"

namespace dsc {

template <typename E, int W, int HPT>
__global__ void __launch_bounds__(32 * (1 + TileCfg<E, HPT, true>::NCW), 1)
    dense_bwd_tma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                  const __grid_constant__ CUtensorMap tm_w, const DenseParams p)
{
    using Cfg = TileCfg<E, HPT, true>;
    constexpr int TT = Cfg::TT, RPW = Cfg::RPW, NCW = Cfg::NCW;
    constexpr int GR = TT + W - 1;  // dy / w rows per tile
    constexpr int NWV = HPT * W;

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
        // ---------------- producer
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_dy);
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
            for (int r = lane; r < GR; r += 32) {
                const int t = t0 + r;
                nv[r] = static_cast<int8_t>(t < p.BT ? cursor.taps(t, p.T, W, p.cu, p.n_docs) : W);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&hdr->full[s], p.tx_bytes);
                tma_load_2d(st + p.x_off, &tm_x, &hdr->full[s], cb * kDC, t0 - (W - 1));
                tma_load_2d(st + p.dy_off, &tm_dy, &hdr->full[s], cb * kDC, t0);
                for (int b = 0; b < p.w_nboxes; ++b)
                    tma_load_2d(st + p.w_off + b * p.w_box_stride, &tm_w, &hdr->full[s],
                                cb * p.w_blk + b * p.w_box, t0);
                issued[s] = it;
            }
        }
        if (aborted && lane == 0) {
            for (int s = 0; s < p.nstages; ++s)
                if (issued[s] >= 0) (void)mbar_wait(&hdr->full[s], (issued[s] / p.nstages) & 1, kDrainLimitNs);
        }
    } else {
        // ---------------- consumers
        const int r0 = (warp - 1) * RPW;
        const int wstart = ((lane * 8) >> p.hshift) * W;
        const int wb = wstart / p.w_box;
        const int wo = wstart - wb * p.w_box;
        const int lanes_per_head = p.hshift > 3 ? 1 << (p.hshift - 3) : 1;  // lanes sharing a head: H/8 for H >= 8
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
            const E *xs = reinterpret_cast<const E *>(st + p.x_off) + lane * 8;    // row i <-> token t0-(W-1)+i
            const E *gs = reinterpret_cast<const E *>(st + p.dy_off) + lane * 8;   // row i <-> token t0+i
            const E *ws = reinterpret_cast<const E *>(st + p.w_off + wb * p.w_box_stride) + wo;
            const int8_t *nvs = reinterpret_cast<const int8_t *>(st + p.nv_off);
            const int c = cb * kDC + lane * 8;
            const bool cvalid = c < p.D;
            E *dx = reinterpret_cast<E *>(p.out0);
            E *dw = reinterpret_cast<E *>(p.out1);
            const int head = c >> p.hshift;  // global head of this lane's first channel

            // Rings indexed by step r (token t0+r0+r): the x window (slot ring(r, W) holds the x row of
            // step r) and the dx accumulators (slot ring(r, W) collects the gradient of step r's token).
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
                const int j = r0 + r;  // tile-local token of this step
                float2 g[4];
                load8x2(gs + j * kDC, g);
                float wv[NWV];
                load_n<E, NWV>(ws + j * p.w_box, wv);
                float2 wp[4][W];
                filter_pairs<HPT, W>(wv, wp);
                const int nv = nvs[j];
                // dx: the residual opens this token's slot; w[j,k] * dy[j] goes to token j-k
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[ring(r, W)][i] = g[i];
                if (nv == W) {
#pragma unroll
                    for (int k = 0; k < W; ++k)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[ring(r - k, W)][i] = fma2(wp[i][k], g[i], acc[ring(r - k, W)][i]);
                } else {
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        if (k < nv) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                acc[ring(r - k, W)][i] = fma2(wp[i][k], g[i], acc[ring(r - k, W)][i]);
                        }
                }
                if (r >= W - 1) {  // the token of step r-(W-1) has received all of its terms
                    const int tdx = t0 + j - (W - 1);
                    if (cvalid && tdx < p.BT) store8x2(dx + static_cast<size_t>(tdx) * p.D + c, acc[ring(r - (W - 1), W)]);
                }
                if (r < RPW) {  // dw of token j: sum over each head's channels of dy * x~
                    load8x2(xs + (j + W - 1) * kDC, xw[ring(r, W)]);
                    float part[HPT][W];
#pragma unroll
                    for (int k = 0; k < W; ++k) {
                        const float2(&xk)[4] = xw[ring(r - k, W)];
                        if constexpr (HPT == 8) {  // one channel per head: plain products
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 pr = mul2(g[i], xk[i]);
                                part[2 * i][k] = pr.x;
                                part[2 * i + 1][k] = pr.y;
                            }
                        } else {
                            constexpr int PPH = 4 / HPT;  // channel pairs per head
#pragma unroll
                            for (int h = 0; h < HPT; ++h) {
                                float2 sacc = mul2(g[h * PPH], xk[h * PPH]);
#pragma unroll
                                for (int i = 1; i < PPH; ++i) sacc = fma2(g[h * PPH + i], xk[h * PPH + i], sacc);
                                part[h][k] = sacc.x + sacc.y;
                            }
                        }
                    }
                    if (nv != W) {
#pragma unroll
                        for (int h = 0; h < HPT; ++h)
#pragma unroll
                            for (int k = 0; k < W; ++k) part[h][k] = k < nv ? part[h][k] : 0.f;
                    }
                    if constexpr (HPT == 1) {
                        for (int off = 1; off < lanes_per_head; off <<= 1) {
#pragma unroll
                            for (int k = 0; k < W; ++k) part[0][k] += __shfl_xor_sync(0xffffffffu, part[0][k], off);
                        }
                    }
                    const int t = t0 + j;
                    const bool leader = (HPT > 1) || ((lane & (lanes_per_head - 1)) == 0);
                    if (cvalid && leader && t < p.BT) {
                        float o[NWV];
#pragma unroll
                        for (int h = 0; h < HPT; ++h)
#pragma unroll
                            for (int k = 0; k < W; ++k) o[h * W + k] = part[h][k];
                        store_n<E, NWV>(dw + (static_cast<size_t>(t) * p.G + head) * W, o);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdr->empty[s]);
        }
    }
}

// Scalar path for any shape the TMA path cannot take.
template <typename E>
__global__ void dense_bwd_dx_scalar(const E *__restrict__ w, const E *__restrict__ dy, E *__restrict__ dx, int BT,
                                    int T, int D, int W, int H, const int32_t *cu, int n_docs)
{
    const long long n = static_cast<long long>(BT) * D;
    const int G = D / H;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i / D), d = static_cast<int>(i - static_cast<long long>(s) * D);
        float acc = Elem<E>::to_f(dy[i]);
        for (int k = 0; k < W && s + k < BT; ++k) {
            const int t = s + k;
            if (k < valid_taps(t, T, W, cu, n_docs))
                acc = fmaf(Elem<E>::to_f(w[(static_cast<long long>(t) * G + d / H) * W + k]),
                           Elem<E>::to_f(dy[static_cast<long long>(t) * D + d]), acc);
        }
        dx[i] = Elem<E>::from_f(acc);
    }
}

template <typename E>
__global__ void dense_bwd_dw_scalar(const E *__restrict__ x, const E *__restrict__ dy, E *__restrict__ dw, int BT,
                                    int T, int D, int W, int H, const int32_t *cu, int n_docs)
{
    const int G = D / H;
    const long long n = static_cast<long long>(BT) * G * W;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int k = static_cast<int>(i % W);
        const long long tg = i / W;
        const int g = static_cast<int>(tg % G);
        const int t = static_cast<int>(tg / G);
        float acc = 0.f;
        if (k < valid_taps(t, T, W, cu, n_docs)) {
            for (int d = g * H; d < (g + 1) * H; ++d)
                acc = fmaf(Elem<E>::to_f(dy[static_cast<long long>(t) * D + d]),
                           Elem<E>::to_f(x[static_cast<long long>(t - k) * D + d]), acc);
        }
        dw[i] = Elem<E>::from_f(acc);
    }
}

template <typename E, int W, int HPT>
static dsc_status launch_bwd_tma(const DenseArgs &a, const DeviceInfo &dev)
{
    using Cfg = TileCfg<E, HPT, true>;
    DensePlan plan;
    if (!make_dense_plan(a, true, Cfg::TT, Cfg::RPW, Cfg::kStageCap, dev, &plan)) return DSC_ERR_UNSUPPORTED;
    const CUtensorMapDataType tdt =
        sizeof(E) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const unsigned long long BT = static_cast<unsigned long long>(a.B) * a.T;
    const unsigned long long G = a.D / a.H;
    const unsigned long long row = static_cast<unsigned long long>(a.D) * sizeof(E);
    CUtensorMap tm_x, tm_dy, tm_w;
    if (!encode_tmap_2d(&tm_x, a.x, tdt, a.D, BT, row, kDC, plan.x_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&tm_dy, a.dy, tdt, a.D, BT, row, kDC, plan.g_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&tm_w, a.w, tdt, G * a.W, BT, G * a.W * sizeof(E), plan.w_box, plan.g_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return DSC_ERR_UNSUPPORTED;  // descriptor rejected: the scalar path takes the call
    auto kern = dense_bwd_tma<E, W, HPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes);
    if (e != cudaSuccess) return DSC_ERR_CUDA;
    const DenseParams q = dense_params(a, plan, a.dx, a.dw);
    return launch_overlapped(kern, plan.grid, plan.threads, plan.smem_bytes, a.stream, tm_x, tm_dy, tm_w, q);
}

template <typename E, int W>
static dsc_status bwd_by_hpt(const DenseArgs &a, const DeviceInfo &dev)
{
    switch (a.H) {
    case 1: return launch_bwd_tma<E, W, 8>(a, dev);
    case 2: return launch_bwd_tma<E, W, 4>(a, dev);
    case 4: return launch_bwd_tma<E, W, 2>(a, dev);
    default: return launch_bwd_tma<E, W, 1>(a, dev);
    }
}

template <typename E>
static dsc_status bwd_tma(const DenseArgs &a, const DeviceInfo &dev)
{
    switch (a.W) {
    case 1: return bwd_by_hpt<E, 1>(a, dev);
    case 2: return bwd_by_hpt<E, 2>(a, dev);
    case 3: return bwd_by_hpt<E, 3>(a, dev);
    case 4: return bwd_by_hpt<E, 4>(a, dev);
    case 5: return bwd_by_hpt<E, 5>(a, dev);
    case 6: return bwd_by_hpt<E, 6>(a, dev);
    case 7: return bwd_by_hpt<E, 7>(a, dev);
    case 8: return bwd_by_hpt<E, 8>(a, dev);
    default: return DSC_ERR_INVALID_ARG;
    }
}

template <typename E>
static dsc_status bwd_scalar(const DenseArgs &a, const DeviceInfo &dev)
{
    const long long BT = static_cast<long long>(a.B) * a.T;
    const long long cap = static_cast<long long>(dev.sm_count) * 8;
    long long b1 = (BT * a.D + 255) / 256;
    long long b2 = (BT * (a.D / a.H) * a.W + 255) / 256;
    if (b1 > cap) b1 = cap;
    if (b2 > cap) b2 = cap;
    dense_bwd_dx_scalar<E><<<static_cast<int>(b1), 256, 0, a.stream>>>(
        static_cast<const E *>(a.w), static_cast<const E *>(a.dy), static_cast<E *>(a.dx), static_cast<int>(BT), a.T,
        a.D, a.W, a.H, a.cu, a.n_docs);
    dsc_status s = launched();
    if (s != DSC_OK) return s;
    dense_bwd_dw_scalar<E><<<static_cast<int>(b2), 256, 0, a.stream>>>(
        static_cast<const E *>(a.x), static_cast<const E *>(a.dy), static_cast<E *>(a.dw), static_cast<int>(BT), a.T,
        a.D, a.W, a.H, a.cu, a.n_docs);
    return launched();
}

dsc_status dense_bwd(const DenseArgs &a)
{
    DeviceInfo dev;
    if (!device_info(&dev)) return DSC_ERR_CUDA;
    const dsc_status s = a.dt == DSC_BF16 ? bwd_tma<__nv_bfloat16>(a, dev) : bwd_tma<float>(a, dev);
    if (s != DSC_ERR_UNSUPPORTED) return s;
    return a.dt == DSC_BF16 ? bwd_scalar<__nv_bfloat16>(a, dev) : bwd_scalar<float>(a, dev);
}

}  // namespace dsc
