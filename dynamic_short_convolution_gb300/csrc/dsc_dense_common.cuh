// dsc_dense_common.cuh -- tile plan shared by the materialised / head-wise
// forward and backward kernels.
//
// Work decomposition: a tile is TT consecutive tokens of the flattened B*T
// axis times a block of kDC = 256 channels (one warp covers the block, 8
// channels = one 16-byte bf16 vector per lane).  A persistent grid walks the
// tiles channel-block-fastest, so the tiles that share a halo run at the same
// time and the halo rows come from L2.  One producer warp stages every tile
// with TMA into a ring of shared-memory stages (mbarrier full/empty pairs);
// consumer warps each own RPW consecutive tokens of the tile.
#pragma once

#include "dsc_device.cuh"
#include "dsc_internal.h"

namespace dsc {

constexpr int kDC = 256;        // channels per tile
constexpr int kMaxStages = 8;   // shared-memory ring depth cap

// Tokens per tile (TT) and per consumer warp (RPW), by element type, heads
// per lane (HPT: 8 for H=1, 4 for H=2, 2 for H=4, 1 for H>=8) and direction.
// bf16 forward: 16 consumer warps; for H >= 8 tiles of 48 tokens (3 per warp,
// stages of 33 KB, a ring of 5) or, with WIDE, of 64 tokens (4 per warp,
// stages of 43 KB, 5 of them fit) -- the launcher picks one per call; for
// smaller H larger tiles (the filter rows grow with 1/H).  bf16 backward: 16
// consumer warps of 3 tokens for H >= 8, 4 warps of 4 tokens for H = 1 (the
// filter rows dominate a stage); stages of 59 KB, 3 fit.  Chosen by measured
// sweeps and A/B runs of the tile shape and ring depth on GB300.  fp32 halves
// the tokens.
template <typename E, int HPT, bool BWD, bool WIDE = false>
struct TileCfg {
    static constexpr bool kBf16 = sizeof(E) == 2;
    static constexpr int TTb = BWD ? (HPT == 1 ? 48 : HPT == 8 ? 16 : 32)
                                   : (HPT == 1 ? (WIDE ? 64 : 48) : HPT == 2 ? 64 : HPT == 4 ? 48 : 32);
    static constexpr int RPWb = BWD ? (HPT == 1 ? 3 : 4)
                                    : (HPT == 1 ? (WIDE ? 4 : 3) : HPT == 2 ? 4 : HPT == 4 ? 3 : 2);
    static constexpr int TT = kBf16 ? TTb : (BWD && HPT == 8 ? 8 : TTb / 2);
    static constexpr int RPW = kBf16 ? RPWb : (BWD ? (HPT == 1 ? 8 : 4) : RPWb);
    static constexpr int NCW = TT / RPW;  // consumer warps
    static constexpr int kStageCap = (!BWD && HPT == 1 && kBf16 && !WIDE) ? 5 : kMaxStages;
    static_assert(TT % RPW == 0, "whole warps per tile");
};

// Filter values of one lane's channel pairs: wp[i][k] = (w[head(2i), k], w[head(2i+1), k]).
template <int HPT, int W>
__device__ __forceinline__ void filter_pairs(const float (&wv)[HPT * W], float2 (&wp)[4][W])
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < W; ++k)
            wp[i][k] = make_float2(wv[((2 * i) * HPT / 8) * W + k], wv[((2 * i + 1) * HPT / 8) * W + k]);
}

// Host-side plan of one launch of the TMA path.
struct DensePlan {
    int esize = 2;
    int hpt = 1;          // heads per lane class
    int hshift = 0;       // log2(H)
    int TT = 0, RPW = 0, NCW = 0;
    int x_rows = 0;       // x rows staged per tile (TT + W - 1)
    int g_rows = 0;       // dy / w rows staged per tile (TT fwd, TT + W - 1 bwd)
    int w_blk = 0;        // filter values per token in one channel block
    int w_box = 0;        // inner extent of one w box (elements)
    int w_nboxes = 0;
    unsigned w_box_stride = 0;  // bytes between w boxes in a stage (128-byte aligned TMA destinations)
    unsigned x_off = 0, dy_off = 0, w_off = 0, nv_off = 0, stage_bytes = 0, tx_bytes = 0;
    int nstages = 0;
    int n_cb = 0, n_tiles = 0;
    int grid = 0, threads = 0;
    unsigned smem_bytes = 0;
};

inline int ilog2_exact(int v)
{
    int s = 0;
    while ((1 << s) < v) ++s;
    return (1 << s) == v ? s : -1;
}

// Decide whether the TMA path can take these arguments and lay out its stages.
// Returns false (use the scalar path) when a TMA alignment or size rule fails.
inline bool make_dense_plan(const DenseArgs &a, bool bwd, int TT, int RPW, int stage_cap, const DeviceInfo &dev,
                            DensePlan *p)
{
    const int esize = (a.dt == DSC_BF16) ? 2 : 4;
    p->esize = esize;
    const int hs = ilog2_exact(a.H);
    if (hs < 0 || a.H > kDC) return false;
    if ((static_cast<long long>(a.D) * esize) % 16 != 0) return false;
    const long long G = a.D / a.H;
    if ((G * a.W * esize) % 16 != 0) return false;  // w row pitch must be a TMA stride
    if (!aligned16(a.x) || !aligned16(a.w)) return false;
    if (bwd && (!aligned16(a.dy) || !aligned16(a.dx) || !aligned16(a.dw))) return false;
    if (!bwd && !aligned16(a.y)) return false;
    p->hshift = hs;
    p->hpt = a.H >= 8 ? 1 : 8 / a.H;
    const int nwv = p->hpt * a.W;  // filter values one lane reads per token
    p->w_blk = (kDC / a.H) * a.W;
    int box = 0;
    for (int c = p->w_blk < 256 ? p->w_blk : 256; c >= 1; --c) {
        if (p->w_blk % c == 0 && c % nwv == 0 && (c * esize) % 16 == 0) { box = c; break; }
    }
    if (box == 0) return false;
    p->w_box = box;
    p->w_nboxes = p->w_blk / box;
    p->TT = TT;
    p->RPW = RPW;
    p->NCW = TT / RPW;
    p->x_rows = TT + a.W - 1;
    p->g_rows = bwd ? TT + a.W - 1 : TT;
    const unsigned x_bytes = static_cast<unsigned>(kDC * esize * p->x_rows);
    const unsigned dy_bytes = bwd ? static_cast<unsigned>(kDC * esize * p->g_rows) : 0u;
    const unsigned w_box_bytes = static_cast<unsigned>(box * esize * p->g_rows);
    p->w_box_stride = align_up(w_box_bytes, 128);
    const unsigned w_bytes = p->w_box_stride * p->w_nboxes;
    unsigned off = 0;
    p->x_off = off;
    off = align_up(off + x_bytes, 1024);
    p->dy_off = off;
    off = align_up(off + dy_bytes, 1024);
    p->w_off = off;
    off = align_up(off + w_bytes, 128);
    p->nv_off = off;
    off = align_up(off + static_cast<unsigned>(p->g_rows), 1024);
    p->stage_bytes = off;
    p->tx_bytes = x_bytes + dy_bytes + w_box_bytes * p->w_nboxes;  // bytes the copies deliver
    const unsigned header = 2048;  // barriers + abort flag, then slack to align the stages to 1024 B
    const int fit = static_cast<int>((static_cast<unsigned>(dev.max_smem_optin) - header) / p->stage_bytes);
    if (fit < 2) return false;
    p->nstages = fit < stage_cap ? fit : stage_cap;
    p->smem_bytes = header + p->nstages * p->stage_bytes;
    const long long BT = static_cast<long long>(a.B) * a.T;
    p->n_cb = (a.D + kDC - 1) / kDC;
    const long long n_tt = (BT + TT - 1) / TT;
    const long long n_tiles = n_tt * p->n_cb;
    if (n_tiles > 0x7fffffffLL) return false;
    p->n_tiles = static_cast<int>(n_tiles);
    p->threads = 32 * (1 + p->NCW);
    p->grid = dev.sm_count;  // one CTA per SM (the ring takes most of shared memory)
    if (p->grid > p->n_tiles) p->grid = p->n_tiles;
    return true;
}

// Parameters the dense kernels read (passed by value).
struct DenseParams {
    void *out0;            // fwd: y; bwd: dx
    void *out1;            // bwd: dw
    const int32_t *cu;
    int n_docs;
    int BT, T, D, G;       // G = D / H
    int hshift;
    int n_cb, n_tiles;
    int w_blk, w_box, w_nboxes;
    unsigned w_box_stride;
    unsigned x_off, dy_off, w_off, nv_off, stage_bytes, tx_bytes;
    int nstages;
    int *status;
    unsigned long long wait_ns;
};

inline DenseParams dense_params(const DenseArgs &a, const DensePlan &p, void *out0, void *out1)
{
    DenseParams q;
    q.out0 = out0;
    q.out1 = out1;
    q.cu = a.cu;
    q.n_docs = a.n_docs;
    q.BT = a.B * a.T;
    q.T = a.T;
    q.D = a.D;
    q.G = a.D / a.H;
    q.hshift = p.hshift;
    q.n_cb = p.n_cb;
    q.n_tiles = p.n_tiles;
    q.w_blk = p.w_blk;
    q.w_box = p.w_box;
    q.w_nboxes = p.w_nboxes;
    q.w_box_stride = p.w_box_stride;
    q.x_off = p.x_off;
    q.dy_off = p.dy_off;
    q.w_off = p.w_off;
    q.nv_off = p.nv_off;
    q.stage_bytes = p.stage_bytes;
    q.tx_bytes = p.tx_bytes;
    q.nstages = p.nstages;
    q.status = device_status_word();
    q.wait_ns = wait_limit_ns();
    return q;
}

// Shared-memory header: full[kMaxStages], empty[kMaxStages], abort flag.
struct RingHeader {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int abort_flag;
};

// First stage: 1 KB past the header, rounded up to a 1024-byte shared address.
__device__ __forceinline__ uint8_t *stage_base(uint8_t *smem)
{
    uint8_t *b = smem + 1024;
    return b + ((1024u - (smem_u32(b) & 1023u)) & 1023u);
}

}  // namespace dsc
