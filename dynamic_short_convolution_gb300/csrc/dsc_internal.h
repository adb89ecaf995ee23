// dsc_internal.h -- host-side plumbing shared by the libdsc translation units.
#pragma once

#include <cuda.h>
#include <mutex>
#include <cuda_runtime.h>

#include "dsc.h"

namespace dsc {

// Arguments of the materialised / head-wise forward and backward passes.
struct DenseArgs {
    const void *x = nullptr;
    const void *w = nullptr;
    const void *dy = nullptr;
    void *y = nullptr;
    void *dx = nullptr;
    void *dw = nullptr;
    int B = 0, T = 0, D = 0, W = 0, H = 0;
    dsc_dtype dt = DSC_BF16;
    const int32_t *cu = nullptr;
    int n_docs = 0;
    cudaStream_t stream = nullptr;
};

// Arguments of the low-rank forward and backward passes.
struct LowrankArgs {
    const void *x = nullptr;
    const void *z = nullptr;
    const void *U = nullptr;
    const float *bias = nullptr;
    const void *dy = nullptr;
    void *y = nullptr;
    void *dx = nullptr;
    void *dz = nullptr;
    float *dU = nullptr;
    float *db = nullptr;
    void *workspace = nullptr;
    int B = 0, T = 0, D = 0, W = 0, R = 0;
    const int32_t *cu = nullptr;
    int n_docs = 0;
    cudaStream_t stream = nullptr;
};

// Arguments of the static short convolution (filter w [D, W]; dw fp32 [D, W]).
struct StaticArgs {
    const void *x = nullptr;
    const void *w = nullptr;
    const void *dy = nullptr;
    void *y = nullptr;
    void *dx = nullptr;
    float *dw = nullptr;
    int B = 0, T = 0, D = 0, W = 0;
    dsc_dtype dt = DSC_BF16;
    const int32_t *cu = nullptr;
    int n_docs = 0;
    cudaStream_t stream = nullptr;
};

// Arguments of one decode step (x, y [B, D]; w [B, D/H, W]; hist [B, W-1, D]; pos [B]).
struct DecodeArgs {
    const void *x = nullptr;
    const void *w = nullptr;
    void *hist = nullptr;
    const int32_t *pos = nullptr;
    void *y = nullptr;
    int B = 0, D = 0, W = 0, H = 0;
    dsc_dtype dt = DSC_BF16;
    cudaStream_t stream = nullptr;
};

// Arguments of the projection with the convolution in its epilogue (h [B,T,Dm]; Wx [D,Dm]; Wg [(D/H)W, Dm];
// bg [(D/H)W] fp32 or nullptr; y [B,T,D]).
struct ProjArgs {
    const void *h = nullptr;
    const void *Wx = nullptr;
    const void *Wg = nullptr;
    const float *bg = nullptr;
    void *y = nullptr;
    int B = 0, T = 0, Dm = 0, D = 0, W = 0, H = 0;
    const int32_t *cu = nullptr;
    int n_docs = 0;
    cudaStream_t stream = nullptr;
};

dsc_status dense_fwd(const DenseArgs &a);
dsc_status dense_bwd(const DenseArgs &a);
// Low-rank forward whose code z = h W1^T is computed on chip from the layer input h.
struct LowrankZArgs {
    const void *x = nullptr;
    const void *h = nullptr;
    const void *W1 = nullptr;
    const float *b1 = nullptr;  // may be null
    const void *U = nullptr;
    const float *bias = nullptr;
    void *y = nullptr;
    int B = 0, T = 0, D = 0, Dm = 0, W = 0, R = 0;
    const int32_t *cu = nullptr;
    int n_docs = 0;
    cudaStream_t stream = nullptr;
};

dsc_status lowrank_fwd(const LowrankArgs &a);
dsc_status lowrank_zproj_fwd(const LowrankZArgs &a);
dsc_status lowrank_bwd(const LowrankArgs &a);
size_t lowrank_bwd_workspace(int B, int T, int D, int W, int R);
dsc_status lowrank_bwd_validate(const void *x, const void *z, const void *U, const float *bias, const void *dy, void *dx,
                                void *dz, float *dU, float *db, int B, int T, int D, int W, int R, dsc_dtype dt,
                                const int32_t *cu_seqlens, int n_docs);
struct DeviceInfo;
dsc_status lowrank_bwd_dudb(const LowrankArgs &a, const DeviceInfo &dev);  // second kernel of lowrank_bwd
dsc_status static_fwd(const StaticArgs &a);
dsc_status static_bwd(const StaticArgs &a);
dsc_status decode_step(const DecodeArgs &a);
dsc_status proj_fwd(const ProjArgs &a);

// Device address of a file-scope __device__ variable on the current device, looked up once per device
// and context (looked up again after the context changes, e.g. after cudaDeviceReset).
struct SymbolCache {
    static constexpr int kDevices = 64;
    std::mutex mu;
    CUcontext ctx[kDevices] = {};
    void *addr[kDevices] = {};
};
void *symbol_address(SymbolCache *cache, const void *symbol);

// Per-device status word (device address) and the current wait limit.
int *device_status_word();
unsigned long long wait_limit_ns();

// Device facts of the current device (cached per device).
struct DeviceInfo {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
};
bool device_info(DeviceInfo *out);

// 2-D tiled TMA descriptor: dims {inner, outer}, row pitch in bytes, box
// {box_inner, box_outer}, zero fill outside the tensor.
bool encode_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, unsigned long long inner,
                    unsigned long long outer, unsigned long long row_bytes, unsigned box_inner, unsigned box_outer,
                    CUtensorMapSwizzle swizzle);

// Count one kernel launch (process-wide; reported by dsc_launch_count).
void count_launch(unsigned n = 1);

inline dsc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSC_OK : DSC_ERR_CUDA; }

// Status of a launch that was just queued: counts it when it succeeded.
inline dsc_status launched(unsigned n = 1)
{
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(n);
    return cuda_status(e);
}

// Launch a kernel that may begin while the stream's previous kernel is still running (programmatic
// dependent launch).  The kernel itself orders every access that depends on that previous kernel behind
// grid_dependency_wait(); the previous kernel lets it start with grid_dependents_launch() or by exiting.
template <typename... KArgs, typename... Args>
inline dsc_status launch_overlapped(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return DSC_ERR_CUDA;
    }
    return launched();
}

inline unsigned align_up(unsigned v, unsigned a) { return (v + a - 1) / a * a; }

inline bool aligned16(const void *p) { return (reinterpret_cast<unsigned long long>(p) & 15ull) == 0; }

}  // namespace dsc
