/*
 * dsc.h -- C ABI of libdsc.so, the GB300 (sm_103a) dynamic short convolution.
 *
 * The operation (notes on "Dynamic Short Convolutions Improve Transformers",
 * section "Parameterization", eq. 2, applied as a residual as in eq. 3 of
 * section "Placement"):
 *
 *     y[t,d] = x[t,d] + sum_{k=0}^{W-1} w[t, g(d), k] * x~[t-k, d]
 *
 * a causal depthwise convolution along time whose filter is generated per
 * token.  g(d) = floor(d / H): H is the head SIZE -- H consecutive channels
 * share one filter ("head-wise parameterization"); H = 1 is the materialised
 * per-channel filter.  x~[j, d] = x[j, d] when token j lies in token t's
 * document, else 0: zero history before every sequence start and, with
 * packed documents, before every document start (the boundary rule of the
 * notes on "RubiConv - Efficient Boundary-Respecting Convolutions", section
 * "Key design 1").  The residual term x[t,d] is never masked.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout.  Row-major, contiguous, tokens on a flattened B*T axis:
 *     x, y, dy, dx     [B, T, D]
 *     w, dw            [B, T, D/H, W]     (tap index k innermost; k = 0 is the
 *                                          current token, k = j reaches back j)
 *     z, dz            [B, T, R]
 *     U, dU            [R, D*W]           (filter column n = d*W + k)
 *     bias, db         [D*W]              (fp32)
 *     cu_seqlens       [n_docs + 1] int32 offsets on the flattened axis
 *                      (0 = cu[0] < cu[1] < ... < cu[n_docs] = B*T).  Every
 *                      sequence start b*T is a document start whether or not it
 *                      is listed.  NULL: each sequence is one document.
 *  Ownership.  Every pointer is caller-owned DEVICE memory of the current
 *     device, 16-byte aligned for the vectorised paths (any element-aligned
 *     pointer is accepted and routed to a scalar path).  The library
 *     allocates no device memory and keeps no per-call state; it caches the
 *     SM count and kernel attributes per device.
 *  Semantics.  Outputs are OVERWRITTEN (never accumulated).  Calls are
 *     asynchronous on `stream` and return after the launches are queued.
 *     Inputs and outputs must not overlap.
 *  Precision.  bf16 (or fp32) storage, fp32 arithmetic, results rounded to
 *     nearest-even on store.
 *  Errors.  Arguments are validated before any launch; a rejected call
 *     launches nothing and returns DSC_ERR_INVALID_ARG or
 *     DSC_ERR_UNSUPPORTED.  A failed launch returns DSC_ERR_CUDA.  Kernels
 *     never trap: a device-side wait that exceeds its time limit records
 *     DSC_ERR_TIMEOUT in a device status word, which dsc_sync_status()
 *     reports.  Nothing aborts, exits or throws across this ABI.
 *  Malformed cu_seqlens (not increasing, wrong ends) cannot make a kernel
 *     read or write out of bounds; the results are then unspecified.
 *     dsc_validate_cu_seqlens() checks them on the device.
 */
#ifndef DSC_H
#define DSC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSC_OK = 0,
    DSC_ERR_INVALID_ARG = 1, /* bad size, null pointer, D % H != 0, ... */
    DSC_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. fp32 low-rank) */
    DSC_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    DSC_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up */
} dsc_status;

typedef enum { DSC_F32 = 0, DSC_BF16 = 1 } dsc_dtype;

/* Library version (major * 10000 + minor * 100 + patch). */
int dsc_version(void);

/* Human-readable name of a status code (static string). */
const char *dsc_status_string(dsc_status s);

/*
 * dsc_fwd -- forward pass, materialised (H = 1) or head-wise (H > 1) filter.
 *   "Parameterization", eq. 2, with the residual of eq. 3.
 *   x [B,T,D], w [B,T,D/H,W] in dtype dt; writes y [B,T,D].
 *   Requirements: B, T, D >= 1; 1 <= W <= 8; H >= 1 and D % H == 0;
 *   B*T*D < 2^31; cu_seqlens NULL or n_docs >= 1.
 *   Reads every input once and writes y once ("Efficient training": the
 *   kernel reads activations and weights once and keeps the convolution on
 *   chip).
 */
dsc_status dsc_fwd(const void *x, const void *w, void *y, int B, int T, int D, int W, int H, dsc_dtype dt,
                   const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_bwd -- backward pass of dsc_fwd for an upstream gradient dy.
 *   The derivative of eq. 2 + eq. 3:
 *     dx[s,d]   = dy[s,d] + sum_{k<W, s+k in s's document} w[s+k, g(d), k] dy[s+k, d]
 *     dw[t,g,k] = sum_{d : g(d) = g} dy[t,d] * x~[t-k, d]
 *   x, w, dy in dtype dt; writes dx [B,T,D] and dw [B,T,D/H,W] (both fully
 *   overwritten).  Same requirements as dsc_fwd.
 */
dsc_status dsc_bwd(const void *x, const void *w, const void *dy, void *dx, void *dw, int B, int T, int D, int W,
                   int H, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_lowrank_fwd -- forward pass with the low-rank filter generator fused.
 *   "Parameterization" (low-rank D -> R -> W*D, every transform with a bias)
 *   and "Efficient training" (the second projection fused into the kernel):
 *     w[t, d, k] = sum_r z[t,r] U[r, d*W+k] + bias[d*W+k]
 *   is formed on chip (tensor cores, fp32 accumulation) and never written to
 *   memory, then eq. 2 + eq. 3 with H = 1.
 *   x [B,T,D], z [B,T,R], U [R,D*W] in bf16, bias [D*W] fp32; writes y.
 *   Requirements: dt == DSC_BF16 (DSC_F32 -> DSC_ERR_UNSUPPORTED);
 *   D % 8 == 0; R % 8 == 0 and 8 <= R <= 256; 1 <= W <= 8; pointers 16-byte
 *   aligned.
 */
dsc_status dsc_lowrank_fwd(const void *x, const void *z, const void *U, const float *bias, void *y, int B, int T,
                           int D, int W, int R, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs,
                           cudaStream_t stream);

/*
 * dsc_lowrank_zproj_fwd -- dsc_lowrank_fwd with the generator's first
 *   projection on chip as well.  "Parameterization": the generator maps the
 *   layer input through D -> R -> W*D; "Placement": its first projection runs
 *   beside the Q/K/V projection, on the same input h.  Computes
 *     z[t, r]    = sum_i h[t, i] W1[r, i] + b1[r]
 *     w[t, d, k] = sum_r z[t, r] U[r, d*W+k] + bias[d*W+k]
 *   on the tensor cores (fp32 accumulation; z enters the second product
 *   rounded to bf16, as a stored activation would be) and never writes z or w
 *   to memory, then eq. 2 + eq. 3 with H = 1 on x.
 *   x [B,T,D], h [B,T,Dm], W1 [R,Dm] (row-major, as a linear layer's weight),
 *   U [R,D*W] in bf16; b1 [R] fp32 or NULL (no first bias; every transform of
 *   the generator carries a bias, and b1 U can equally be folded into bias);
 *   bias [D*W] fp32; writes y [B,T,D].  All caller-owned device memory.
 *   Requirements: those of dsc_lowrank_fwd, and Dm >= 1 with Dm % 8 == 0,
 *   R <= 128 (larger ranks -> DSC_ERR_UNSUPPORTED: compute z with a GEMM and
 *   call dsc_lowrank_fwd), B*T*Dm < 2^31.
 */
dsc_status dsc_lowrank_zproj_fwd(const void *x, const void *h, const void *W1, const float *b1, const void *U,
                                 const float *bias, void *y, int B, int T, int D, int Dm, int W, int R, dsc_dtype dt,
                                 const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * Bytes of caller-provided device workspace dsc_lowrank_bwd needs for these
 * sizes: 16 * (D*W + 256) rounded up to 1024, plus 2 * R * D*W rounded up to
 * 256; independent of B and T.  The call writes into it the generator bias
 * split into bf16 high and low halves (one 16-byte row per filter entry) and a
 * copy of U, both with the W taps of each group of 8 channels reordered
 * tap-major.
 */
size_t dsc_lowrank_bwd_workspace_bytes(int B, int T, int D, int W, int R);

/*
 * dsc_lowrank_bwd -- backward pass of dsc_lowrank_fwd.
 *   With G[t, d*W+k] = dy[t,d] * x~[t-k, d] (the gradient of the generated
 *   filter, formed on chip) and the filter recomputed on chip:
 *     dx  as in dsc_bwd with w = zU + bias
 *     dz[t,r] = sum_n G[t,n] U[r,n]        (bf16 [B,T,R])
 *     dU[r,n] = sum_t z[t,r] G[t,n]        (fp32 [R, D*W])
 *     db[n]   = sum_t G[t,n]               (fp32 [D*W])
 *   `workspace` must hold dsc_lowrank_bwd_workspace_bytes() bytes of device
 *   memory, 256-byte aligned (may be NULL when that size is 0); its contents on
 *   entry are ignored.  Same requirements as dsc_lowrank_fwd except the rank:
 *   R % 8 == 0 and 8 <= R <= 256 (other ranks return DSC_ERR_UNSUPPORTED
 *   before anything is launched).  dy, dx, dz, dU and db must be non-NULL and
 *   16-byte aligned (else DSC_ERR_INVALID_ARG).  dx and dz are deterministic;
 *   dU and db are sums of fp32 partials added in a run-dependent order.
 */
dsc_status dsc_lowrank_bwd(const void *x, const void *z, const void *U, const float *bias, const void *dy, void *dx,
                           void *dz, float *dU, float *db, void *workspace, int B, int T, int D, int W, int R,
                           dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_lowrank_bwd_noalloc -- dsc_lowrank_bwd for callers that cannot allocate
 * device memory: a plugin inside a host framework that owns the whole device
 * memory pool under a fixed memory plan, or a latency-critical loop that must
 * never enter the allocator.  The paper has no counterpart; this is an
 * interface convenience.  Same arguments and results as dsc_lowrank_bwd,
 * without `workspace`: the workspace lives in a fixed array of 8 MiB in the
 * library's static device memory, held by every GPU that loads the library
 * until the process exits.  Nothing is allocated or freed by the call, and no
 * allocating library routine is used.
 *   Limit: dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R) <= 8 MiB (about
 *   2 * R * D*W + 16 * D*W bytes); larger sizes return DSC_ERR_INVALID_ARG
 *   before anything is launched.
 *   The first call on a device looks up the array's device address (once per
 *   device and context, with that device current); make that first call
 *   before any stream capture.
 *   Every call uses the same array and rewrites it before reading it.  Calls
 *   that overlap on the GPU (for example on two streams) race on the array:
 *   serialise them.
 */
dsc_status dsc_lowrank_bwd_noalloc(const void *x, const void *z, const void *U, const float *bias, const void *dy,
                                   void *dx, void *dz, float *dU, float *db, int B, int T, int D, int W, int R,
                                   dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_static_fwd -- the static short convolution: one filter for every token
 *   ("Parameterization", eq. 1), applied with the residual of eq. 3 and the
 *   same zero history before sequence and document starts:
 *     y[t,d] = x[t,d] + sum_{k<W} w[d,k] * x~[t-k, d]
 *   x [B,T,D] and w [D,W] (tap k innermost) in dtype dt; writes y [B,T,D].
 *   Requirements as dsc_fwd (no H).  The fast path wants D % 8 == 0 and
 *   16-byte aligned pointers; other shapes take a slower element-wise path.
 */
dsc_status dsc_static_fwd(const void *x, const void *w, void *y, int B, int T, int D, int W, dsc_dtype dt,
                          const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_static_bwd -- backward pass of dsc_static_fwd for an upstream gradient dy:
 *     dx[s,d] = dy[s,d] + sum_{k<W, s+k in s's document} w[d,k] dy[s+k, d]
 *     dw[d,k] = sum over every token t of dy[t,d] * x~[t-k, d]
 *   x, w, dy in dtype dt; writes dx [B,T,D] (dtype dt) and dw [D,W] in fp32
 *   (both overwritten).  dw is summed with fp32 atomic additions, so the
 *   order of its additions, and its last bits, may vary from call to call.
 *   Requirements as dsc_static_fwd.
 */
dsc_status dsc_static_bwd(const void *x, const void *w, const void *dy, void *dx, float *dw, int B, int T, int D,
                          int W, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs, cudaStream_t stream);

/*
 * dsc_decode_step -- one inference step of eq. 2 + eq. 3 for B sequences, one
 *   new token each, against a per-sequence history of the last W-1 inputs.
 *   The notes list inference optimisation as open work ("Discussion and
 *   limitations"); this is the single-token form of dsc_fwd.
 *     x [B,D]        this step's inputs (dtype dt)
 *     w [B,D/H,W]    their filters (head size H as in dsc_fwd)
 *     pos [B] int32  the position of each token within its document
 *                    (0 = the document's first token); read only -- the
 *                    caller advances it
 *     hist [B,W-1,D] a ring of past inputs: slot (p mod (W-1)) holds the input
 *                    of the document's token at position p.  Read, then the
 *                    slot (pos mod (W-1)) is overwritten with x (W > 1; with
 *                    W == 1 hist is not touched and may be NULL)
 *     y [B,D]        y[b,d] = x[b,d] + sum_{k<W, k<=pos[b]} w[b,g(d),k] * x_{pos-k}
 *   History before a document start is zero because pos says where the
 *   document starts, so a new document needs no reset of hist.  A negative
 *   pos is treated as 0 and recorded as DSC_ERR_INVALID_ARG in the device
 *   status word.  Requirements: B, D >= 1; 1 <= W <= 8; D % H == 0;
 *   B*(W-1)*D < 2^31.  The fast path wants (16 / element size) | D and x, y,
 *   hist 16-byte aligned.
 */
dsc_status dsc_decode_step(const void *x, const void *w, void *hist, const int32_t *pos, void *y, int B, int D, int W,
                           int H, dsc_dtype dt, cudaStream_t stream);

/*
 * dsc_proj_fwd -- the projection that produces the convolution's input and its
 *   filter, with eq. 2 + eq. 3 applied in the projection GEMM's epilogue
 *   ("Placement": the filter generator's projection beside the Q/K/V
 *   projection; fusing the convolution into the matmul epilogue saves the
 *   round trip of x and w through memory):
 *     x[t,d]   = sum_j h[t,j] Wx[d,j]                     (never stored)
 *     w[t,g,k] = sum_j h[t,j] Wg[g*W + k, j] + bg[g*W+k]  (never stored)
 *     y[t,d]   = x[t,d] + sum_{k<W} w[t, d/H, k] * x~[t-k, d]
 *   with the zero history and document masking of dsc_fwd.
 *     h  [B,T,Dm]         the projection's input, bf16
 *     Wx [D,Dm]           one row per output channel (the layout of a linear
 *                         layer's weight), bf16
 *     Wg [(D/H)*W, Dm]    the generator: row g*W + k is tap k of head g, bf16
 *     bg [(D/H)*W]        the generator's bias, fp32; may be NULL (no bias)
 *     y  [B,T,D]          bf16, overwritten
 *   x and w are accumulated in fp32 on the tensor cores and used unrounded.
 *   Requirements: dt == DSC_BF16 (DSC_F32 -> DSC_ERR_UNSUPPORTED); D, Dm
 *   multiples of 8; D % H == 0 with H in {1, 2, 4} or a multiple of 8, and a
 *   tile of whole heads must fit 256 accumulator columns (H <= 128 for
 *   W <= 8; else DSC_ERR_UNSUPPORTED); 1 <= W <= 8; h, Wx, Wg, y 16-byte
 *   aligned, bg 4-byte aligned; B*T*max(D, Dm) < 2^31.
 */
dsc_status dsc_proj_fwd(const void *h, const void *Wx, const void *Wg, const float *bg, void *y, int B, int T, int Dm,
                        int D, int W, int H, dsc_dtype dt, const int32_t *cu_seqlens, int n_docs,
                        cudaStream_t stream);

/*
 * dsc_validate_cu_seqlens -- device-side check of packed-document offsets:
 * cu[0] == 0, strictly increasing, cu[n_docs] == B*T.  Asynchronous; a
 * violation is recorded as DSC_ERR_INVALID_ARG in the device status word,
 * read by dsc_sync_status().
 */
dsc_status dsc_validate_cu_seqlens(const int32_t *cu_seqlens, int n_docs, int B, int T, cudaStream_t stream);

/*
 * dsc_sync_status -- synchronise `stream`, then read and clear the device
 * status word of the current device.  Returns DSC_OK, DSC_ERR_TIMEOUT (a
 * kernel's bounded wait gave up), DSC_ERR_INVALID_ARG (a failed
 * dsc_validate_cu_seqlens, or a negative position given to dsc_decode_step)
 * or DSC_ERR_CUDA.  The word is shared by every stream of the device: with
 * calls in flight on several streams, a status may come from any of them.
 */
dsc_status dsc_sync_status(cudaStream_t stream);

/*
 * dsc_launch_count -- number of kernels this library has launched in this
 * process, on any device (a monotonically increasing counter; for
 * accounting in benchmarks).
 */
unsigned long long dsc_launch_count(void);

/*
 * dsc_test_wait_timeout -- test hook for the failure path.  Launches one tiny
 * kernel that waits on a shared-memory barrier nothing ever arrives at, with
 * the same bounded wait the product kernels use and the given limit in
 * nanoseconds; when the limit runs out it records DSC_ERR_TIMEOUT in the
 * device status word (read it with dsc_sync_status) and returns.  Nothing
 * hangs, traps or faults.  The paper has no counterpart; this exists so the
 * timeout path can be tested on a GPU.
 */
dsc_status dsc_test_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSC_H */
