// dsc_abi.cu -- the extern "C" entry points of libdsc.so: argument
// validation, path selection, the device status word and small utilities.
// The operations are defined in dsc.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "dsc_device.cuh"
#include "dsc_internal.h"

namespace dsc {

// One status word per device (static device memory: no allocation).  Kernels
// record the first error of any launch here; dsc_sync_status takes it (reads
// and clears it in one atomic exchange) into g_status_taken.
__device__ int g_status_word;
__device__ int g_status_taken;

static std::mutex g_mu;
static constexpr int kMaxDevices = 64;
static DeviceInfo g_dev[kMaxDevices] = {};
static bool g_dev_ok[kMaxDevices] = {};
static std::atomic<unsigned long long> g_wait_ns{1000000000ull};  // about one second
static std::atomic<unsigned long long> g_launches{0};

void count_launch(unsigned n) { g_launches.fetch_add(n); }

// cuCtxGetCurrent through the runtime's driver entry point (no libcuda link).
using PfnCtxGetCurrent = CUresult (*)(CUcontext *);
static PfnCtxGetCurrent ctx_get_current_fn()
{
    static PfnCtxGetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PfnCtxGetCurrent>(p);
    });
    return fn;
}

static CUcontext current_context()
{
    CUcontext c = nullptr;
    auto fn = ctx_get_current_fn();
    if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
}

void *symbol_address(SymbolCache *cache, const void *symbol)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SymbolCache::kDevices) return nullptr;
    std::lock_guard<std::mutex> lk(cache->mu);
    const CUcontext cur = current_context();
    if (cache->addr[dev] && cur != nullptr && cache->ctx[dev] == cur) return cache->addr[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
    cache->ctx[dev] = current_context();  // the runtime call above made the device's context current
    cache->addr[dev] = p;
    return p;
}

static SymbolCache g_status_cache, g_taken_cache;

int *device_status_word() { return static_cast<int *>(symbol_address(&g_status_cache, &g_status_word)); }

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }

bool device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return false;
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library links no libcuda at build time.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, unsigned long long inner,
                    unsigned long long outer, unsigned long long row_bytes, unsigned box_inner, unsigned box_outer,
                    CUtensorMapSwizzle swizzle)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ small kernels

__global__ void validate_cu_kernel(const int32_t *cu, int n_docs, long long BT, int *status)
{
    bool bad = false;
    for (int i = threadIdx.x; i <= n_docs; i += blockDim.x) {
        const long long v = cu[i];
        if (i == 0 && v != 0) bad = true;
        if (i == n_docs && v != BT) bad = true;
        if (i > 0 && v <= static_cast<long long>(cu[i - 1])) bad = true;
    }
    if (bad) record_status(status, kStatusInvalid);
}

// Read and clear the status word in one atomic step, so an error that a kernel on
// another stream records meanwhile is never lost.
__global__ void take_status_kernel(int *st, int *taken) { *taken = atomicExch(st, 0); }

// A wait on an mbarrier that nothing ever arrives at: exercises the bounded
// wait and the timeout status without hanging anything.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, int *status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) record_status(status, kStatusTimeout);
}

}  // namespace dsc

using namespace dsc;

// ------------------------------------------------------------------ validation helpers

static bool dims_ok(int B, int T, int D, int W)
{
    if (B < 1 || T < 1 || D < 1 || W < 1 || W > 8) return false;
    const long long n = static_cast<long long>(B) * T * D;
    return n < (1LL << 31);
}

static bool cu_ok(const int32_t *cu, int n_docs) { return cu == nullptr || n_docs >= 1; }

static bool elem_aligned(const void *p, int esize)
{
    return p != nullptr && (reinterpret_cast<unsigned long long>(p) % static_cast<unsigned>(esize)) == 0;
}

extern "C" {

int dsc_version(void) { return 10000; }

const char *dsc_status_string(dsc_status s)
{
    switch (s) {
    case DSC_OK: return "DSC_OK";
    case DSC_ERR_INVALID_ARG: return "DSC_ERR_INVALID_ARG";
    case DSC_ERR_UNSUPPORTED: return "DSC_ERR_UNSUPPORTED";
    case DSC_ERR_CUDA: return "DSC_ERR_CUDA";
    case DSC_ERR_TIMEOUT: return "DSC_ERR_TIMEOUT";
    }
    return "DSC_ERR_UNKNOWN";
}

dsc_status dsc_fwd(const void *x, const void *w, void *y, int B, int T, int D, int W, int H, dsc_dtype dt,
                   const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    const int es = dt == DSC_BF16 ? 2 : 4;
    if (!dims_ok(B, T, D, W) || H < 1 || D % H != 0 || !cu_ok(cu_seqlens, n_docs)) return DSC_ERR_INVALID_ARG;
    if (!elem_aligned(x, es) || !elem_aligned(w, es) || !elem_aligned(y, es)) return DSC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * T * (D / H) * W >= (1LL << 31)) return DSC_ERR_INVALID_ARG;
    DenseArgs a;
    a.x = x; a.w = w; a.y = y;
    a.B = B; a.T = T; a.D = D; a.W = W; a.H = H; a.dt = dt;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return dense_fwd(a);
}

dsc_status dsc_bwd(const void *x, const void *w, const void *dy, void *dx, void *dw, int B, int T, int D, int W,
                   int H, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    const int es = dt == DSC_BF16 ? 2 : 4;
    if (!dims_ok(B, T, D, W) || H < 1 || D % H != 0 || !cu_ok(cu_seqlens, n_docs)) return DSC_ERR_INVALID_ARG;
    if (!elem_aligned(x, es) || !elem_aligned(w, es) || !elem_aligned(dy, es) || !elem_aligned(dx, es) ||
        !elem_aligned(dw, es))
        return DSC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * T * (D / H) * W >= (1LL << 31)) return DSC_ERR_INVALID_ARG;
    DenseArgs a;
    a.x = x; a.w = w; a.dy = dy; a.dx = dx; a.dw = dw;
    a.B = B; a.T = T; a.D = D; a.W = W; a.H = H; a.dt = dt;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return dense_bwd(a);
}

static dsc_status lowrank_check(const void *x, const void *z, const void *U, const float *bias, int B, int T, int D,
                                int W, int R, dsc_dtype dt, const int32_t *cu, int n_docs)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    if (!dims_ok(B, T, D, W) || R < 1 || !cu_ok(cu, n_docs)) return DSC_ERR_INVALID_ARG;
    if (!x || !z || !U || !bias) return DSC_ERR_INVALID_ARG;
    if (dt == DSC_F32) return DSC_ERR_UNSUPPORTED;
    if (D % 8 != 0 || R % 8 != 0 || R > 256) return DSC_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(z) || !aligned16(U) || !aligned16(bias)) return DSC_ERR_UNSUPPORTED;
    if (static_cast<long long>(D) * W * R >= (1LL << 31) || static_cast<long long>(B) * T * R >= (1LL << 31))
        return DSC_ERR_INVALID_ARG;
    return DSC_OK;
}

dsc_status dsc_lowrank_fwd(const void *x, const void *z, const void *U, const float *bias, void *y, int B, int T,
                           int D, int W, int R, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs,
                           cudaStream_t stream)
{
    dsc_status s = lowrank_check(x, z, U, bias, B, T, D, W, R, dt, cu_seqlens, n_docs);
    if (s != DSC_OK) return s;
    if (!y) return DSC_ERR_INVALID_ARG;
    if (!aligned16(y)) return DSC_ERR_UNSUPPORTED;
    LowrankArgs a;
    a.x = x; a.z = z; a.U = U; a.bias = bias; a.y = y;
    a.B = B; a.T = T; a.D = D; a.W = W; a.R = R;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return lowrank_fwd(a);
}

dsc_status dsc_lowrank_zproj_fwd(const void *x, const void *h, const void *W1, const float *b1, const void *U,
                                 const float *bias, void *y, int B, int T, int D, int Dm, int W, int R, dsc_dtype dt,
                                 const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    // x, U, bias and the shape as for dsc_lowrank_fwd (h stands in for z in the pointer checks)
    dsc_status s = lowrank_check(x, h, U, bias, B, T, D, W, R, dt, cu_seqlens, n_docs);
    if (s != DSC_OK) return s;
    if (!W1 || !y || Dm < 1) return DSC_ERR_INVALID_ARG;
    if (b1 != nullptr && !elem_aligned(b1, 4)) return DSC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * T * Dm >= (1LL << 31) || static_cast<long long>(R) * Dm >= (1LL << 31))
        return DSC_ERR_INVALID_ARG;
    if (Dm % 8 != 0 || R > 128) return DSC_ERR_UNSUPPORTED;
    if (!aligned16(W1) || !aligned16(y)) return DSC_ERR_UNSUPPORTED;
    LowrankZArgs a;
    a.x = x; a.h = h; a.W1 = W1; a.b1 = b1; a.U = U; a.bias = bias; a.y = y;
    a.B = B; a.T = T; a.D = D; a.Dm = Dm; a.W = W; a.R = R;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return lowrank_zproj_fwd(a);
}

size_t dsc_lowrank_bwd_workspace_bytes(int B, int T, int D, int W, int R)
{
    if (!dims_ok(B, T, D, W) || R < 1) return 0;
    return lowrank_bwd_workspace(B, T, D, W, R);
}

}  // extern "C"

// The backward's checks of everything but the workspace (shared with the allocation-free entry point).
dsc_status dsc::lowrank_bwd_validate(const void *x, const void *z, const void *U, const float *bias, const void *dy,
                                     void *dx, void *dz, float *dU, float *db, int B, int T, int D, int W, int R,
                                     dsc_dtype dt, const int32_t *cu_seqlens, int n_docs)
{
    dsc_status s = lowrank_check(x, z, U, bias, B, T, D, W, R, dt, cu_seqlens, n_docs);
    if (s != DSC_OK) return s;
    if (!dy || !dx || !dz || !dU || !db) return DSC_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(dx) || !aligned16(dz) || !aligned16(dU) || !aligned16(db))
        return DSC_ERR_UNSUPPORTED;
    return DSC_OK;
}

extern "C" {

dsc_status dsc_lowrank_bwd(const void *x, const void *z, const void *U, const float *bias, const void *dy, void *dx,
                           void *dz, float *dU, float *db, void *workspace, int B, int T, int D, int W, int R,
                           dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    dsc_status s = lowrank_bwd_validate(x, z, U, bias, dy, dx, dz, dU, db, B, T, D, W, R, dt, cu_seqlens, n_docs);
    if (s != DSC_OK) return s;
    const size_t ws = lowrank_bwd_workspace(B, T, D, W, R);
    if (ws > 0 && (workspace == nullptr || (reinterpret_cast<unsigned long long>(workspace) & 255ull) != 0))
        return DSC_ERR_INVALID_ARG;
    LowrankArgs a;
    a.x = x; a.z = z; a.U = U; a.bias = bias; a.dy = dy;
    a.dx = dx; a.dz = dz; a.dU = dU; a.db = db; a.workspace = workspace;
    a.B = B; a.T = T; a.D = D; a.W = W; a.R = R;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return lowrank_bwd(a);
}

dsc_status dsc_static_fwd(const void *x, const void *w, void *y, int B, int T, int D, int W, dsc_dtype dt,
                          const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    const int es = dt == DSC_BF16 ? 2 : 4;
    if (!dims_ok(B, T, D, W) || !cu_ok(cu_seqlens, n_docs)) return DSC_ERR_INVALID_ARG;
    if (!elem_aligned(x, es) || !elem_aligned(w, es) || !elem_aligned(y, es)) return DSC_ERR_INVALID_ARG;
    StaticArgs a;
    a.x = x; a.w = w; a.y = y;
    a.B = B; a.T = T; a.D = D; a.W = W; a.dt = dt;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return static_fwd(a);
}

dsc_status dsc_static_bwd(const void *x, const void *w, const void *dy, void *dx, float *dw, int B, int T, int D,
                          int W, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    const int es = dt == DSC_BF16 ? 2 : 4;
    if (!dims_ok(B, T, D, W) || !cu_ok(cu_seqlens, n_docs)) return DSC_ERR_INVALID_ARG;
    if (!elem_aligned(x, es) || !elem_aligned(w, es) || !elem_aligned(dy, es) || !elem_aligned(dx, es) ||
        !elem_aligned(dw, 4))
        return DSC_ERR_INVALID_ARG;
    StaticArgs a;
    a.x = x; a.w = w; a.dy = dy; a.dx = dx; a.dw = dw;
    a.B = B; a.T = T; a.D = D; a.W = W; a.dt = dt;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return static_bwd(a);
}

dsc_status dsc_proj_fwd(const void *h, const void *Wx, const void *Wg, const float *bg, void *y, int B, int T, int Dm,
                        int D, int W, int H, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs,
                        cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    if (!dims_ok(B, T, D, W) || Dm < 1 || H < 1 || D % H != 0 || !cu_ok(cu_seqlens, n_docs))
        return DSC_ERR_INVALID_ARG;
    if (!h || !Wx || !Wg || !y) return DSC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * T * Dm >= (1LL << 31)) return DSC_ERR_INVALID_ARG;
    if (bg != nullptr && !elem_aligned(bg, 4)) return DSC_ERR_INVALID_ARG;
    if (dt == DSC_F32) return DSC_ERR_UNSUPPORTED;
    if (D % 8 != 0 || Dm % 8 != 0 || !(H == 1 || H == 2 || H == 4 || H % 8 == 0)) return DSC_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(Wx) || !aligned16(Wg) || !aligned16(y)) return DSC_ERR_UNSUPPORTED;
    ProjArgs a;
    a.h = h; a.Wx = Wx; a.Wg = Wg; a.bg = bg; a.y = y;
    a.B = B; a.T = T; a.Dm = Dm; a.D = D; a.W = W; a.H = H;
    a.cu = cu_seqlens; a.n_docs = cu_seqlens ? n_docs : 0; a.stream = stream;
    return proj_fwd(a);
}

dsc_status dsc_decode_step(const void *x, const void *w, void *hist, const int32_t *pos, void *y, int B, int D, int W,
                           int H, dsc_dtype dt, cudaStream_t stream)
{
    if (dt != DSC_F32 && dt != DSC_BF16) return DSC_ERR_INVALID_ARG;
    const int es = dt == DSC_BF16 ? 2 : 4;
    if (!dims_ok(B, 1, D, W) || H < 1 || D % H != 0) return DSC_ERR_INVALID_ARG;
    if (!elem_aligned(x, es) || !elem_aligned(w, es) || !elem_aligned(y, es) || !elem_aligned(pos, 4))
        return DSC_ERR_INVALID_ARG;
    if (W > 1 && !elem_aligned(hist, es)) return DSC_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * (W - 1) * D >= (1LL << 31)) return DSC_ERR_INVALID_ARG;
    DecodeArgs a;
    a.x = x; a.w = w; a.hist = hist; a.pos = pos; a.y = y;
    a.B = B; a.D = D; a.W = W; a.H = H; a.dt = dt; a.stream = stream;
    return decode_step(a);
}

dsc_status dsc_validate_cu_seqlens(const int32_t *cu_seqlens, int n_docs, int B, int T, cudaStream_t stream)
{
    if (!cu_seqlens || n_docs < 1 || B < 1 || T < 1) return DSC_ERR_INVALID_ARG;
    int *st = device_status_word();
    if (!st) return DSC_ERR_CUDA;
    validate_cu_kernel<<<1, 256, 0, stream>>>(cu_seqlens, n_docs, static_cast<long long>(B) * T, st);
    return launched();
}

dsc_status dsc_sync_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DSC_ERR_CUDA;
    int *st = device_status_word();
    int *taken = static_cast<int *>(symbol_address(&g_taken_cache, &g_status_taken));
    if (!st || !taken) return DSC_ERR_CUDA;
    take_status_kernel<<<1, 1, 0, stream>>>(st, taken);
    if (cudaGetLastError() != cudaSuccess) return DSC_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, taken, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DSC_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DSC_ERR_CUDA;
    return static_cast<dsc_status>(v);
}

dsc_status dsc_test_wait_timeout(unsigned long long limit_ns, cudaStream_t stream)
{
    int *st = device_status_word();
    if (!st) return DSC_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, st);
    return launched();
}

unsigned long long dsc_launch_count(void) { return g_launches.load(); }

}  // extern "C"
