/*
 * dsc_oracle.c -- plain, slow fp64 CPU oracle for the dynamic short convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * What it computes (notes on "Dynamic Short Convolutions Improve
 * Transformers", section "Parameterization", eqs. 1-3, and section
 * "Efficient training"):
 *
 *   eq. 2 + residual of eq. 3:
 *     y[t,d] = x[t,d] + sum_{k<W} w[t, g(d), k] * xt(t, t-k, d)
 *   with g(d) = floor(d / H) (H = head size: H consecutive channels share one
 *   filter; H = 1 is the materialised per-channel form), and
 *     xt(t, j, d) = x[j, d] if j >= docstart(t) else 0
 *   (zero history before a sequence start and before a packed-document start;
 *   the latter rule is from the notes on "RubiConv - Efficient
 *   Boundary-Respecting Convolutions", section "Key design 1").
 *
 *   low-rank form ("Parameterization", D -> R -> W*D with a bias):
 *     Wt[t, d*W + k] = sum_r z[t,r] U[r, d*W + k] + bias[d*W + k]
 *   then the materialised conv above with w[t,d,k] = Wt[t, d*W+k].
 *
 *   The backward pass is the plain derivative of that bilinear map with an
 *   upstream gradient dy:
 *     dx[s,d]   = dy[s,d] + sum_{k<W, s+k<BT, s>=docstart(s+k)} w[s+k,g(d),k] dy[s+k,d]
 *     dw[t,g,k] = sum_{d: g(d)=g} dy[t,d] * xt(t, t-k, d)
 *   low-rank, with G[t, d*W+k] = dy[t,d] * xt(t, t-k, d):
 *     dz[t,r] = sum_n G[t,n] U[r,n],  dU[r,n] = sum_t z[t,r] G[t,n],
 *     db[n]   = sum_t G[t,n].
 *
 *   Also: the static form (eq. 1, one filter w[d,k] for all tokens) with the
 *   same residual and masking, its backward (dw summed over every token), and
 *   one decode step of eq. 2 + 3 against a per-sequence history ring.
 *
 *   Projected form ("Placement": the filter generator's projection sits beside
 *   the Q/K/V projection, and the convolution consumes both outputs):
 *     x[t,d]   = sum_j h[t,j] Wx[d,j]
 *     w[t,g,k] = sum_j h[t,j] Wg[g*W + k, j] + bg[g*W + k]
 *   then eq. 2 + residual of eq. 3 on that x and w.
 *
 * Tokens are indexed on the flattened B*T axis; docstart(t) >= (t / T) * T
 * always, so sequences never see each other.  Every product and sum is done
 * in IEEE double from inputs converted exactly (fp32, bf16 or fp64 storage).
 * OpenMP only splits independent output rows/columns across threads; it
 * changes no arithmetic.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { DSCO_F32 = 0, DSCO_BF16 = 1, DSCO_F64 = 2 };

/* Exact conversion of one stored element to double. */
static double load(const void *p, int dt, int64_t i)
{
    if (dt == DSCO_F32)
        return (double)((const float *)p)[i];
    if (dt == DSCO_F64)
        return ((const double *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16; /* bf16 = high half of fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int dsco_version(void) { return 1; }

/*
 * Per-token document start on the flattened axis.  The start of the token's
 * own sequence, raised to the largest packed-document offset cu[i] <= t.
 * cu may be NULL (each sequence is one document).
 */
void dsco_docstarts(int64_t B, int64_t T, const int32_t *cu, int64_t n_docs, int64_t *ds)
{
    for (int64_t t = 0; t < B * T; ++t) {
        int64_t s = (t / T) * T;
        if (cu) {
            for (int64_t i = 0; i <= n_docs; ++i)
                if ((int64_t)cu[i] <= t && (int64_t)cu[i] > s)
                    s = cu[i];
        }
        ds[t] = s;
    }
}

/* xt(t, j, d): x[j,d] when j lies in token t's document, else 0. */
static double xt(const void *x, int dt, int64_t D, const int64_t *ds, int64_t t, int64_t j, int64_t d)
{
    return (j >= ds[t]) ? load(x, dt, j * D + d) : 0.0;
}

/* Forward, materialised (H = 1) or head-wise weights w[BT, D/H, W]; rows [r0, r1). */
void dsco_fwd_rows(const void *x, const void *w, int dt, int64_t BT, int64_t D, int W, int64_t H,
                   const int64_t *ds, int64_t r0, int64_t r1, double *y)
{
    const int64_t G = D / H;
    (void)BT;
#pragma omp parallel for schedule(static)
    for (int64_t t = r0; t < r1; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            double acc = load(x, dt, t * D + d);
            for (int k = 0; k < W; ++k)
                acc += load(w, dt, (t * G + d / H) * W + k) * xt(x, dt, D, ds, t, t - k, d);
            y[(t - r0) * D + d] = acc;
        }
    }
}

/*
 * Backward, materialised or head-wise.  dx rows [r0, r1) into dx (may be NULL),
 * dw rows [r0, r1) into dw [(r1-r0), D/H, W] (may be NULL).
 */
void dsco_bwd_rows(const void *x, const void *w, const void *dy, int dt, int64_t BT, int64_t D, int W,
                   int64_t H, const int64_t *ds, int64_t r0, int64_t r1, double *dx, double *dw)
{
    const int64_t G = D / H;
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t s = r0; s < r1; ++s) {
            for (int64_t d = 0; d < D; ++d) {
                double acc = load(dy, dt, s * D + d);
                for (int k = 0; k < W; ++k) {
                    int64_t t = s + k;
                    if (t < BT && s >= ds[t])
                        acc += load(w, dt, (t * G + d / H) * W + k) * load(dy, dt, t * D + d);
                }
                dx[(s - r0) * D + d] = acc;
            }
        }
    }
    if (dw) {
#pragma omp parallel for schedule(static)
        for (int64_t t = r0; t < r1; ++t) {
            for (int64_t g = 0; g < G; ++g) {
                for (int k = 0; k < W; ++k) {
                    double acc = 0.0;
                    for (int64_t d = g * H; d < (g + 1) * H; ++d)
                        acc += load(dy, dt, t * D + d) * xt(x, dt, D, ds, t, t - k, d);
                    dw[((t - r0) * G + g) * W + k] = acc;
                }
            }
        }
    }
}

/* Low-rank generated filter: Wt[t, n] = sum_r z[t,r] U[r,n] + bias[n], n = d*W + k. */
static double wlr(const void *z, const void *U, const void *bias, int bdt, int dt, int64_t R, int64_t NW,
                  int64_t t, int64_t n)
{
    double acc = load(bias, bdt, n);
    for (int64_t r = 0; r < R; ++r)
        acc += load(z, dt, t * R + r) * load(U, dt, r * NW + n);
    return acc;
}

/* Low-rank forward rows [r0, r1): the filter row is materialised in fp64, then eq. 2 + residual. */
void dsco_lowrank_fwd_rows(const void *x, const void *z, const void *U, const void *bias, int bdt, int dt, int64_t BT,
                           int64_t D, int W, int64_t R, const int64_t *ds, int64_t r0, int64_t r1, double *y)
{
    const int64_t NW = D * W;
    (void)BT;
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)NW);
#pragma omp for schedule(static)
        for (int64_t t = r0; t < r1; ++t) {
            for (int64_t n = 0; n < NW; ++n)
                wrow[n] = wlr(z, U, bias, bdt, dt, R, NW, t, n);
            for (int64_t d = 0; d < D; ++d) {
                double acc = load(x, dt, t * D + d);
                for (int k = 0; k < W; ++k)
                    acc += wrow[d * W + k] * xt(x, dt, D, ds, t, t - k, d);
                y[(t - r0) * D + d] = acc;
            }
        }
        free(wrow);
    }
}

/*
 * Low-rank forward with the generator's first projection ("Parameterization":
 * the generator maps the layer input through D -> R -> W*D; "Placement": its
 * first projection runs beside the Q/K/V projection): rows [r0, r1) of
 *   z[t, r]  = b1[r] + sum_i h[t, i] W1[r, i]            (the rank-R code; b1 may be NULL: no bias)
 *   Wt[t, n] = sum_r z[t, r] U[r, n] + bias[n]            n = d*W + k
 *   y[t, d]  = x[t, d] + sum_k Wt[t, d*W+k] * x~[t-k, d]
 * all in fp64.  h [BT, Dm], W1 [R, Dm], x [BT, D], U [R, D*W] share one
 * storage type; bias and b1 have their own (bdt).
 */
void dsco_lowrank_zproj_fwd_rows(const void *x, const void *h, const void *W1, const void *b1, const void *U,
                                 const void *bias, int bdt, int dt, int64_t BT, int64_t Dm, int64_t D, int W, int64_t R,
                                 const int64_t *ds, int64_t r0, int64_t r1, double *y)
{
    const int64_t NW = D * W;
    (void)BT;
#pragma omp parallel
    {
        double *zr = (double *)malloc(sizeof(double) * (size_t)R);
        double *wrow = (double *)malloc(sizeof(double) * (size_t)NW);
#pragma omp for schedule(static)
        for (int64_t t = r0; t < r1; ++t) {
            for (int64_t r = 0; r < R; ++r) {
                double acc = b1 ? load(b1, bdt, r) : 0.0;
                for (int64_t i = 0; i < Dm; ++i) acc += load(h, dt, t * Dm + i) * load(W1, dt, r * Dm + i);
                zr[r] = acc;
            }
            for (int64_t n = 0; n < NW; ++n) {
                double acc = load(bias, bdt, n);
                for (int64_t r = 0; r < R; ++r) acc += zr[r] * load(U, dt, r * NW + n);
                wrow[n] = acc;
            }
            for (int64_t d = 0; d < D; ++d) {
                double acc = load(x, dt, t * D + d);
                for (int k = 0; k < W; ++k)
                    acc += wrow[d * W + k] * xt(x, dt, D, ds, t, t - k, d);
                y[(t - r0) * D + d] = acc;
            }
        }
        free(zr);
        free(wrow);
    }
}

/* G[t, d*W+k] = dy[t,d] * xt(t, t-k, d): the gradient of the loss w.r.t. the generated filter. */
static double gfil(const void *x, const void *dy, int dt, int64_t D, int W, const int64_t *ds, int64_t t, int64_t n)
{
    int64_t d = n / W, k = n % W;
    return load(dy, dt, t * D + d) * xt(x, dt, D, ds, t, t - k, d);
}

/*
 * Low-rank backward, per-row outputs for rows [r0, r1):
 *   dx rows (may be NULL) and dz rows [(r1-r0), R] (may be NULL).
 */
void dsco_lowrank_bwd_rows(const void *x, const void *z, const void *U, const void *bias, int bdt, const void *dy, int dt,
                           int64_t BT, int64_t D, int W, int64_t R, const int64_t *ds, int64_t r0, int64_t r1,
                           double *dx, double *dz)
{
    const int64_t NW = D * W;
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t s = r0; s < r1; ++s) {
            for (int64_t d = 0; d < D; ++d) {
                double acc = load(dy, dt, s * D + d);
                for (int k = 0; k < W; ++k) {
                    int64_t t = s + k;
                    if (t < BT && s >= ds[t])
                        acc += wlr(z, U, bias, bdt, dt, R, NW, t, d * W + k) * load(dy, dt, t * D + d);
                }
                dx[(s - r0) * D + d] = acc;
            }
        }
    }
    if (dz) {
#pragma omp parallel for schedule(static)
        for (int64_t t = r0; t < r1; ++t) {
            for (int64_t r = 0; r < R; ++r) {
                double acc = 0.0;
                for (int64_t n = 0; n < NW; ++n)
                    acc += gfil(x, dy, dt, D, W, ds, t, n) * load(U, dt, r * NW + n);
                dz[(t - r0) * R + r] = acc;
            }
        }
    }
}

/*
 * Low-rank backward, parameter gradients for a list of filter columns n = cols[i]:
 *   dU[r, i] = sum_t z[t,r] G[t, n]   (dU laid out [R, ncols], may be NULL)
 *   db[i]    = sum_t G[t, n]          (may be NULL)
 * Sums run over every token of the flattened axis.
 */
void dsco_lowrank_bwd_params(const void *x, const void *z, const void *dy, int dt, int64_t BT, int64_t D, int W,
                             int64_t R, const int64_t *ds, const int64_t *cols, int64_t ncols, double *dU, double *db)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < ncols; ++i) {
        const int64_t n = cols[i];
        if (db) {
            double acc = 0.0;
            for (int64_t t = 0; t < BT; ++t)
                acc += gfil(x, dy, dt, D, W, ds, t, n);
            db[i] = acc;
        }
        if (dU) {
            for (int64_t r = 0; r < R; ++r) {
                double acc = 0.0;
                for (int64_t t = 0; t < BT; ++t)
                    acc += load(z, dt, t * R + r) * gfil(x, dy, dt, D, W, ds, t, n);
                dU[r * ncols + i] = acc;
            }
        }
    }
}

/*
 * Static short convolution (eq. 1: one filter w[d][k] for every token), with the residual placement of
 * eq. 3 and the same zero history before each document start:
 *   y[t,d] = x[t,d] + sum_{k<W} w[d,k] * xt(t, t-k, d)
 * rows [r0, r1); w is [D, W].
 */
void dsco_static_fwd_rows(const void *x, const void *w, int dt, int64_t BT, int64_t D, int W, const int64_t *ds,
                          int64_t r0, int64_t r1, double *y)
{
    (void)BT;
#pragma omp parallel for schedule(static)
    for (int64_t t = r0; t < r1; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            double acc = load(x, dt, t * D + d);
            for (int k = 0; k < W; ++k)
                acc += load(w, dt, d * W + k) * xt(x, dt, D, ds, t, t - k, d);
            y[(t - r0) * D + d] = acc;
        }
    }
}

/*
 * Static backward.  dx rows [r0, r1) (dx may be NULL):
 *   dx[s,d] = dy[s,d] + sum_{k<W, s+k<BT, s>=docstart(s+k)} w[d,k] dy[s+k,d]
 * dw [D, W] over every token of the flattened axis (dw may be NULL):
 *   dw[d,k] = sum_t dy[t,d] * xt(t, t-k, d)
 */
void dsco_static_bwd(const void *x, const void *w, const void *dy, int dt, int64_t BT, int64_t D, int W,
                     const int64_t *ds, int64_t r0, int64_t r1, double *dx, double *dw)
{
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t s = r0; s < r1; ++s) {
            for (int64_t d = 0; d < D; ++d) {
                double acc = load(dy, dt, s * D + d);
                for (int k = 0; k < W; ++k) {
                    int64_t t = s + k;
                    if (t < BT && s >= ds[t])
                        acc += load(w, dt, d * W + k) * load(dy, dt, t * D + d);
                }
                dx[(s - r0) * D + d] = acc;
            }
        }
    }
    if (dw) {
#pragma omp parallel for schedule(static)
        for (int64_t d = 0; d < D; ++d) {
            for (int k = 0; k < W; ++k) {
                double acc = 0.0;
                for (int64_t t = 0; t < BT; ++t)
                    acc += load(dy, dt, t * D + d) * xt(x, dt, D, ds, t, t - k, d);
                dw[d * W + k] = acc;
            }
        }
    }
}

/*
 * One decode step of eq. 2 + eq. 3 for B sequences, each at one new token.  x[b, D] is the token's
 * input, w[b, D/H, W] its filter, pos[b] its position within its document, and hist[b, W-1, D] a ring
 * whose slot (p mod (W-1)) holds the input of the document's token at position p:
 *   y[b,d] = x[b,d] + w[b,g(d),0] x[b,d] + sum_{1<=k<W, k<=pos[b]} w[b,g(d),k] hist[b, (pos[b]-k) mod (W-1), d]
 * (a history token before the document start contributes zero).  Only y is computed here; the ring
 * update (slot pos[b] mod (W-1) := x[b]) is a copy.
 */
void dsco_decode_step(const void *x, const void *w, const void *hist, const int32_t *pos, int dt, int64_t B,
                      int64_t D, int W, int64_t H, double *y)
{
    const int64_t G = D / H;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        const int64_t p = pos[b];
        for (int64_t d = 0; d < D; ++d) {
            const double xv = load(x, dt, b * D + d);
            double acc = xv + load(w, dt, (b * G + d / H) * W + 0) * xv;
            for (int k = 1; k < W; ++k) {
                if (p - k < 0)
                    continue;
                const int64_t slot = (p - k) % (W - 1);
                acc += load(w, dt, (b * G + d / H) * W + k) * load(hist, dt, (b * (W - 1) + slot) * D + d);
            }
            y[b * D + d] = acc;
        }
    }
}

/*
 * Projected forward rows [r0, r1): for every output token t, the W input rows
 * x[t-k] (those inside t's document) and the filter row w[t] are computed in
 * fp64 from h, Wx, Wg and bg (bg may be NULL: no generator bias), then eq. 2 +
 * residual.  h [BT, Dm], Wx [D, Dm], Wg [(D/H)*W, Dm] share one storage type;
 * bg has its own (bdt).
 */
void dsco_proj_fwd_rows(const void *h, const void *Wx, const void *Wg, const void *bg, int bdt, int dt, int64_t BT,
                        int64_t Dm, int64_t D, int W, int64_t H, const int64_t *ds, int64_t r0, int64_t r1,
                        double *y)
{
    const int64_t G = D / H, NG = G * W;
    (void)BT;
#pragma omp parallel
    {
        double *xr = (double *)malloc(sizeof(double) * (size_t)(W * D)); /* xr[k*D + d] = x[t-k, d] */
        double *wr = (double *)malloc(sizeof(double) * (size_t)NG);       /* wr[g*W + k] = w[t, g, k] */
#pragma omp for schedule(static)
        for (int64_t t = r0; t < r1; ++t) {
            for (int k = 0; k < W; ++k) {
                const int64_t j = t - k;
                for (int64_t d = 0; d < D; ++d) {
                    double acc = 0.0;
                    if (j >= ds[t])
                        for (int64_t i = 0; i < Dm; ++i)
                            acc += load(h, dt, j * Dm + i) * load(Wx, dt, d * Dm + i);
                    xr[k * D + d] = acc;
                }
            }
            for (int64_t n = 0; n < NG; ++n) {
                double acc = bg ? load(bg, bdt, n) : 0.0;
                for (int64_t i = 0; i < Dm; ++i)
                    acc += load(h, dt, t * Dm + i) * load(Wg, dt, n * Dm + i);
                wr[n] = acc;
            }
            for (int64_t d = 0; d < D; ++d) {
                double acc = xr[d];
                for (int k = 0; k < W; ++k)
                    acc += wr[(d / H) * W + k] * xr[k * D + d];
                y[(t - r0) * D + d] = acc;
            }
        }
        free(xr);
        free(wr);
    }
}
