/*
 * acnn_oracle.c -- plain, slow fp64 CPU oracle for the fused 2-D convolution
 * layer and its companion ops.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it is written straight from the definitions on the pages:
 *
 *   P1  "inferencelayer -- src/rtdetr_gpu.rs" (docs.rs): IM2COL_SRC (tap order
 *       and zero padding), RtDetrGpu::conv (output size), MAXPOOL_SRC,
 *       AVGPOOL_SRC, UPSAMPLE_SRC, CONCAT_SRC, ADDACT_SRC (activations and the
 *       add-then-activate residual).
 *   P3  "@framecast/rt 1.0.0 -- package/rt.js": wgslConv (per-channel PReLU
 *       and the activate-then-add residual), wgslPrepQuarter (RGBA8 unpack,
 *       BGR order, timestep plane, bilinear 1/4), wgslFlowOut (bilinear x8),
 *       wgslDeconv (4x4/s2/p1 transposed conv, gather form), wgslPrepFull and
 *       wgslFlowOut's warp, blend and RGBA8 pack (the one op computed in
 *       binary32, because a float there decides an output byte).
 *
 * Every value is a double.  Where the GPU path stores activations in a
 * narrower type, the caller rounds with oracle_round_storage() between ops
 * (round-to-nearest-even, the reading taken where the pages are silent).
 *
 * Loops are the definitions written out; the only parallelism is a static
 * split of independent output rows (n, oy) over pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { O_NHWC = 0, O_NCHW = 1 };
enum { O_ACT_NONE = 0, O_ACT_RELU = 1, O_ACT_SILU = 2, O_ACT_PRELU = 3 };
enum { O_RES_NONE = 0, O_RES_ADD_THEN_ACT = 1, O_RES_ACT_THEN_ADD = 2 };
enum { O_F32 = 0, O_F16 = 1, O_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* indexing                                                                  */
/* ------------------------------------------------------------------------ */

/* Flat index of activation element (n, c, y, x) in an N x C x H x W tensor
 * stored NHWC (channels innermost, P1) or NCHW (planes, P3). */
static size_t act_index(int layout, int C, int H, int W, int n, int c, int y, int x)
{
    if (layout == O_NHWC)
        return (((size_t)n * H + y) * W + x) * C + c;
    return (((size_t)n * C + c) * H + y) * W + x;
}

/* Flat index of conv weight (co, ci, ky, kx).  With NHWC activations the
 * weight is OHWI, so that k = (ky, kx, ci) -- the (dy, dx, c) order of P1's
 * IM2COL_SRC.  With NCHW activations it is OIHW, P3 wgslConv's [CO,CI,3,3]. */
static size_t wgt_index(int layout, int C_in, int KH, int KW, int co, int ci, int ky, int kx)
{
    if (layout == O_NHWC)
        return (((size_t)co * KH + ky) * KW + kx) * C_in + ci;
    return (((size_t)co * C_in + ci) * KH + ky) * KW + kx;
}

/* ------------------------------------------------------------------------ */
/* activations: P1 ADDACT_SRC (relu = max(v,0), silu = v/(1+exp(-v))) and    */
/* P3 wgslConv (prelu = select(alpha*a, a, a >= 0))                          */
/* ------------------------------------------------------------------------ */
double oracle_act(int act, double v, double alpha)
{
    switch (act) {
    case O_ACT_RELU: return v > 0.0 ? v : 0.0;
    case O_ACT_SILU: return v / (1.0 + exp(-v));
    case O_ACT_PRELU: return v >= 0.0 ? v : alpha * v;
    default: return v;
    }
}

/* ------------------------------------------------------------------------ */
/* row-parallel driver                                                       */
/* ------------------------------------------------------------------------ */
typedef void (*row_fn)(const void* args, int row);
typedef struct { row_fn fn; const void* args; int rows, tid, nthreads; } row_job;

static void* row_worker(void* p)
{
    const row_job* j = (const row_job*)p;
    for (int r = j->tid; r < j->rows; r += j->nthreads)
        j->fn(j->args, r);
    return NULL;
}

static void for_rows(row_fn fn, const void* args, int rows, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = rows > 0 ? rows : 1;
    if (nthreads == 1) {
        for (int r = 0; r < rows; ++r) fn(args, r);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    row_job* jobs = (row_job*)malloc(sizeof(row_job) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].args = args; jobs[t].rows = rows;
        jobs[t].tid = t; jobs[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, row_worker, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
}

/* ------------------------------------------------------------------------ */
/* conv2d_fused                                                              */
/* ------------------------------------------------------------------------ */
typedef struct {
    int layout, N, H, W, C_in, C_out, KH, KW, S, P, OH, OW, act, res_mode;
    const double *x, *wgt, *bias, *alpha, *res;
    double* y;
    const int* pts; /* sampled mode: (n, oy, ox) triples */
} conv_args;

/* One output element.  P1 RtDetrGpu::conv is im2col then a GEMM with the bias
 * and activation in its epilogue: the accumulator starts from the bias and
 * takes every tap k = (ky, kx, ci) in that order; taps that fall outside the
 * input read zero (IM2COL_SRC writes 0.0 there).  The residual is added before
 * the activation (P1: addact(relu) after the block's last conv) or after it
 * (P3 wgslConv: dst = prelu(acc) + res). */
static double conv_point(const conv_args* a, int n, int co, int oy, int ox)
{
    double acc = a->bias ? a->bias[co] : 0.0;
    for (int ky = 0; ky < a->KH; ++ky) {
        int iy = oy * a->S + ky - a->P;
        if (iy < 0 || iy >= a->H) continue;
        for (int kx = 0; kx < a->KW; ++kx) {
            int ix = ox * a->S + kx - a->P;
            if (ix < 0 || ix >= a->W) continue;
            for (int ci = 0; ci < a->C_in; ++ci)
                acc += a->x[act_index(a->layout, a->C_in, a->H, a->W, n, ci, iy, ix)] *
                       a->wgt[wgt_index(a->layout, a->C_in, a->KH, a->KW, co, ci, ky, kx)];
        }
    }
    double al = (a->act == O_ACT_PRELU && a->alpha) ? a->alpha[co] : 0.0;
    if (a->res_mode == O_RES_NONE || !a->res)
        return oracle_act(a->act, acc, al);
    double r = a->res[act_index(a->layout, a->C_out, a->OH, a->OW, n, co, oy, ox)];
    if (a->res_mode == O_RES_ADD_THEN_ACT)
        return oracle_act(a->act, acc + r, al);
    return oracle_act(a->act, acc, al) + r;
}

static void conv_row(const void* p, int row)
{
    const conv_args* a = (const conv_args*)p;
    int n = row / a->OH, oy = row % a->OH;
    for (int ox = 0; ox < a->OW; ++ox)
        for (int co = 0; co < a->C_out; ++co)
            a->y[act_index(a->layout, a->C_out, a->OH, a->OW, n, co, oy, ox)] =
                conv_point(a, n, co, oy, ox);
}

static void conv_pts_row(const void* p, int i)
{
    const conv_args* a = (const conv_args*)p;
    int n = a->pts[3 * i], oy = a->pts[3 * i + 1], ox = a->pts[3 * i + 2];
    for (int co = 0; co < a->C_out; ++co)
        a->y[(size_t)i * a->C_out + co] = conv_point(a, n, co, oy, ox);
}

/* Output size rule of P1 RtDetrGpu::conv: oh = (h + 2p - kh)/s + 1 (floor). */
int oracle_conv_out(int in, int k, int s, int p) { return (in + 2 * p - k) / s + 1; }

int oracle_conv2d(int layout, int N, int H, int W, int C_in, int C_out, int KH, int KW,
                  int S, int P, const double* x, const double* wgt, const double* bias,
                  const double* alpha, const double* res, int res_mode, int act, double* y,
                  int nthreads)
{
    conv_args a = {layout, N, H, W, C_in, C_out, KH, KW, S, P,
                   oracle_conv_out(H, KH, S, P), oracle_conv_out(W, KW, S, P), act, res_mode,
                   x, wgt, bias, alpha, res, y, NULL};
    if (a.OH <= 0 || a.OW <= 0) return -1;
    for_rows(conv_row, &a, N * a.OH, nthreads);
    return 0;
}

/* Same definition at a list of output pixels: y[i*C_out + co] for the pixel
 * (n, oy, ox) = pts[3i .. 3i+2].  Used to check full-size outputs one by one. */
int oracle_conv2d_points(int layout, int N, int H, int W, int C_in, int C_out, int KH, int KW,
                         int S, int P, const double* x, const double* wgt, const double* bias,
                         const double* alpha, const double* res, int res_mode, int act,
                         const int* pts, int npts, double* y, int nthreads)
{
    conv_args a = {layout, N, H, W, C_in, C_out, KH, KW, S, P,
                   oracle_conv_out(H, KH, S, P), oracle_conv_out(W, KW, S, P), act, res_mode,
                   x, wgt, bias, alpha, res, y, pts};
    for_rows(conv_pts_row, &a, npts, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* pooling: P1 MAXPOOL_SRC (-inf padding: out-of-range taps are skipped) and  */
/* AVGPOOL_SRC ((a+b+c+d)*0.25 over a 2x2/s2 window, even inputs)            */
/* ------------------------------------------------------------------------ */
typedef struct {
    int kind, layout, N, C, H, W, K, S, P, OH, OW;
    const double* x;
    double* y;
} pool_args;

static void pool_row(const void* p, int row)
{
    const pool_args* a = (const pool_args*)p;
    int n = row / a->OH, oy = row % a->OH;
    for (int ox = 0; ox < a->OW; ++ox)
        for (int c = 0; c < a->C; ++c) {
            double v;
            if (a->kind == 0) {
                v = -INFINITY;
                for (int dy = 0; dy < a->K; ++dy) {
                    int iy = oy * a->S + dy - a->P;
                    if (iy < 0 || iy >= a->H) continue;
                    for (int dx = 0; dx < a->K; ++dx) {
                        int ix = ox * a->S + dx - a->P;
                        if (ix < 0 || ix >= a->W) continue;
                        double t = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, iy, ix)];
                        if (t > v) v = t;
                    }
                }
            } else {
                double s = 0.0;
                for (int dy = 0; dy < a->K; ++dy)
                    for (int dx = 0; dx < a->K; ++dx)
                        s += a->x[act_index(a->layout, a->C, a->H, a->W, n, c,
                                            oy * a->S + dy, ox * a->S + dx)];
                v = s * (1.0 / (a->K * a->K));
            }
            a->y[act_index(a->layout, a->C, a->OH, a->OW, n, c, oy, ox)] = v;
        }
}

/* kind 0 = max (any K, S, P); kind 1 = average over fully in-range windows
 * (P must be 0, as in AVGPOOL_SRC).  Output size as for conv. */
int oracle_pool2d(int kind, int layout, int N, int C, int H, int W, int K, int S, int P,
                  const double* x, double* y, int nthreads)
{
    if (kind == 1 && P != 0) return -1;
    pool_args a = {kind, layout, N, C, H, W, K, S, P,
                   oracle_conv_out(H, K, S, P), oracle_conv_out(W, K, S, P), x, y};
    if (a.OH <= 0 || a.OW <= 0) return -1;
    for_rows(pool_row, &a, N * a.OH, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* resize                                                                    */
/* ------------------------------------------------------------------------ */
typedef struct {
    int mode, layout, N, C, H, W, OH, OW;
    const double* x;
    double* y;
} resize_args;

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Bilinear with align_corners=false, as P3 wgslPrepQuarter / wgslFlowOut
 * write it: src = (dst + 0.5) * (in/out) - 0.5, x0 = floor(src), f = src - x0,
 * both taps clamped to the image, mix(mix(v00, v10, fx), mix(v01, v11, fx), fy)
 * with mix(a, b, t) = a*(1-t) + b*t. */
static double bilinear_at(const resize_args* a, int n, int c, int oy, int ox)
{
    double sy = (oy + 0.5) * ((double)a->H / a->OH) - 0.5;
    double sx = (ox + 0.5) * ((double)a->W / a->OW) - 0.5;
    double fy0 = floor(sy), fx0 = floor(sx);
    double fy = sy - fy0, fx = sx - fx0;
    int y0 = (int)fy0, x0 = (int)fx0;
    int ya = clampi(y0, 0, a->H - 1), yb = clampi(y0 + 1, 0, a->H - 1);
    int xa = clampi(x0, 0, a->W - 1), xb = clampi(x0 + 1, 0, a->W - 1);
    double v00 = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, ya, xa)];
    double v10 = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, ya, xb)];
    double v01 = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, yb, xa)];
    double v11 = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, yb, xb)];
    double top = v00 * (1.0 - fx) + v10 * fx;
    double bot = v01 * (1.0 - fx) + v11 * fx;
    return top * (1.0 - fy) + bot * fy;
}

static void resize_row(const void* p, int row)
{
    const resize_args* a = (const resize_args*)p;
    int n = row / a->OH, oy = row % a->OH;
    for (int ox = 0; ox < a->OW; ++ox)
        for (int c = 0; c < a->C; ++c) {
            double v;
            if (a->mode == 0) {
                /* nearest, P1 UPSAMPLE_SRC: y[oy, ox] = x[oy/2, ox/2] for 2x;
                 * for any size the source index is floor(dst * in / out). */
                int iy = (int)(((long long)oy * a->H) / a->OH);
                int ix = (int)(((long long)ox * a->W) / a->OW);
                v = a->x[act_index(a->layout, a->C, a->H, a->W, n, c, iy, ix)];
            } else {
                v = bilinear_at(a, n, c, oy, ox);
            }
            a->y[act_index(a->layout, a->C, a->OH, a->OW, n, c, oy, ox)] = v;
        }
}

/* mode 0 = nearest, mode 1 = bilinear (align_corners=false). */
int oracle_resize2d(int mode, int layout, int N, int C, int H, int W, int OH, int OW,
                    const double* x, double* y, int nthreads)
{
    if (OH <= 0 || OW <= 0 || H <= 0 || W <= 0) return -1;
    resize_args a = {mode, layout, N, C, H, W, OH, OW, x, y};
    for_rows(resize_row, &a, N * OH, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* concat: P1 CONCAT_SRC -- per pixel y = [a | b] along channels.            */
/* ------------------------------------------------------------------------ */
int oracle_concat(int layout, int N, int H, int W, int Ca, int Cb, const double* a,
                  const double* b, double* y)
{
    int C = Ca + Cb;
    for (int n = 0; n < N; ++n)
        for (int yy = 0; yy < H; ++yy)
            for (int xx = 0; xx < W; ++xx)
                for (int c = 0; c < C; ++c)
                    y[act_index(layout, C, H, W, n, c, yy, xx)] =
                        c < Ca ? a[act_index(layout, Ca, H, W, n, c, yy, xx)]
                               : b[act_index(layout, Cb, H, W, n, c - Ca, yy, xx)];
    return 0;
}

/* ------------------------------------------------------------------------ */
/* deconv: P3 wgslDeconv, gather form.  Weight layout [CI, CO, K, K].        */
/* y[co, oy, ox] = b[co] + sum over taps (ky, kx) with ty = oy + P - ky >= 0,  */
/* ty % S == 0, iy = ty / S < IH (same along x) of sum_ci x[ci, iy, ix] *     */
/* w[ci, co, ky, kx].  Output size (IH - 1)*S - 2P + K (= 2*IH for 4/2/1).    */
/* ------------------------------------------------------------------------ */
typedef struct {
    int layout, N, C_in, C_out, H, W, K, S, P, OH, OW, act;
    const double *x, *wgt, *bias, *alpha;
    double* y;
} deconv_args;

static void deconv_row(const void* p, int row)
{
    const deconv_args* a = (const deconv_args*)p;
    int n = row / a->OH, oy = row % a->OH;
    for (int ox = 0; ox < a->OW; ++ox)
        for (int co = 0; co < a->C_out; ++co) {
            double acc = a->bias ? a->bias[co] : 0.0;
            for (int ky = 0; ky < a->K; ++ky) {
                int ty = oy + a->P - ky;
                if (ty < 0 || ty % a->S != 0) continue;
                int iy = ty / a->S;
                if (iy >= a->H) continue;
                for (int kx = 0; kx < a->K; ++kx) {
                    int tx = ox + a->P - kx;
                    if (tx < 0 || tx % a->S != 0) continue;
                    int ix = tx / a->S;
                    if (ix >= a->W) continue;
                    for (int ci = 0; ci < a->C_in; ++ci)
                        acc += a->x[act_index(a->layout, a->C_in, a->H, a->W, n, ci, iy, ix)] *
                               a->wgt[(((size_t)ci * a->C_out + co) * a->K + ky) * a->K + kx];
                }
            }
            double al = (a->act == O_ACT_PRELU && a->alpha) ? a->alpha[co] : 0.0;
            a->y[act_index(a->layout, a->C_out, a->OH, a->OW, n, co, oy, ox)] =
                oracle_act(a->act, acc, al);
        }
}

int oracle_deconv2d(int layout, int N, int H, int W, int C_in, int C_out, int K, int S, int P,
                    const double* x, const double* wgt, const double* bias,
                    const double* alpha, int act, double* y, int nthreads)
{
    deconv_args a = {layout, N, C_in, C_out, H, W, K, S, P,
                     (H - 1) * S - 2 * P + K, (W - 1) * S - 2 * P + K, act,
                     x, wgt, bias, alpha, y};
    if (a.OH <= 0 || a.OW <= 0) return -1;
    for_rows(deconv_row, &a, N * a.OH, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* frame prep: P3 wgslPrepQuarter.  Two RGBA8 frames (byte order R,G,B,A per  */
/* pixel, unpacked /255) -> 7 planes [B0,G0,R0,B1,G1,R1,t] at (H/4, W/4),     */
/* each colour plane a bilinear 1/4 downsample (align_corners=false) of the  */
/* full-resolution plane.                                                    */
/* ------------------------------------------------------------------------ */
int oracle_prep_quarter(int H, int W, const uint8_t* rgba0, const uint8_t* rgba1, double t,
                        double* y)
{
    int QH = H / 4, QW = W / 4;
    if (QH <= 0 || QW <= 0) return -1;
    double* plane = (double*)malloc(sizeof(double) * (size_t)H * W);
    for (int f = 0; f < 2; ++f) {
        const uint8_t* src = f == 0 ? rgba0 : rgba1;
        for (int k = 0; k < 3; ++k) {
            int byte = 2 - k; /* plane order B, G, R */
            for (size_t i = 0; i < (size_t)H * W; ++i) plane[i] = src[4 * i + byte] / 255.0;
            resize_args a = {1, O_NCHW, 1, 1, H, W, QH, QW, plane, y + (size_t)(3 * f + k) * QH * QW};
            for (int r = 0; r < QH; ++r) resize_row(&a, r);
        }
    }
    for (size_t i = 0; i < (size_t)QH * QW; ++i) y[(size_t)6 * QH * QW + i] = t;
    free(plane);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* flow out: P3 wgslFlowOut (the stage after the deconv of the frame stack),  */
/* with wgslPrepFull's full-resolution planes read straight from the RGBA8    */
/* frames.  The page computes it in binary32 and truncates to bytes, so a     */
/* float decides an integer here: this function computes in float, one       */
/* operation at a time in the order below (gcc -ffp-contract=off: no fused    */
/* multiply-adds).                                                           */
/*                                                                          */
/*   t = tmp8, 5 planes (flow0 x,y, flow1 x,y, mask) at (H/8, W/8)           */
/*   for output pixel (x, y):                                                */
/*     sx = (x + 0.5) * 0.125 - 0.5, sy likewise  (align_corners=false x8)   */
/*     up(c) = bilinear of plane c at (sx, sy): x0 = floor(sx), fx = sx - x0, */
/*             taps clamped into the plane, mix(a, b, f) = a*(1-f) + b*f,    */
/*             first along x on rows y0 and y0+1, then along y              */
/*     flow0 = 8 * (up(0), up(1)), flow1 = 8 * (up(2), up(3))                */
/*     m = 1 / (1 + exp(-up(4)))                                             */
/*     w_f = bilinear of frame f's B, G, R (byte / 255) at                   */
/*           (x + flow_f.x, y + flow_f.y), taps clamped into the frame       */
/*           (grid_sample, border, align_corners=true)                      */
/*     bgr = w0 * m + w1 * (1 - m)                                           */
/*     out = bytes R, G, B, 255 with each = (uint)(clamp(v, 0, 1) * 255)     */
/*                                                                          */
/* The page's WGSL exp is a binary32 function whose rounding the page does   */
/* not fix; here it is the C library's double exp rounded to float (within    */
/* an ulp of e^x).  Any binary32 exp of similar accuracy moves a byte only     */
/* where clamp(v, 0, 1) * 255 lies within a few ulp of an integer.           */
/* ------------------------------------------------------------------------ */
static float flow_exp(float x)
{
    return (float)exp((double)x);
}

static float flow_mix(float a, float b, float f)
{
    const float u = a * (1.0f - f);
    const float v = b * f;
    return u + v;
}

typedef struct {
    int H, W;
    const float* t;
    const uint8_t* f0;
    const uint8_t* f1;
    const float* res; /* optional refine residual [3][H/4][W/4] (B, G, R) */
    float* pre;       /* [3][H][W] clamped R, G, B in [0, 1] before the byte scale */
    uint8_t* out;     /* [H][W][4] */
} flow_args;

static float flow_up(const flow_args* a, int c, float sx, float sy)
{
    const int TH = a->H / 8, TW = a->W / 8;
    const float* pl = a->t + (size_t)c * TH * TW;
    const float fx0 = floorf(sx), fy0 = floorf(sy);
    const int x0 = (int)fx0, y0 = (int)fy0;
    const float fx = sx - fx0, fy = sy - fy0;
    const int xa = clampi(x0, 0, TW - 1), xb = clampi(x0 + 1, 0, TW - 1);
    const int ya = clampi(y0, 0, TH - 1), yb = clampi(y0 + 1, 0, TH - 1);
    const float top = flow_mix(pl[(size_t)ya * TW + xa], pl[(size_t)ya * TW + xb], fx);
    const float bot = flow_mix(pl[(size_t)yb * TW + xa], pl[(size_t)yb * TW + xb], fx);
    return flow_mix(top, bot, fy);
}

/* Bilinear B, G, R of an RGBA8 frame at pixel-space (px, py), clamped taps. */
static void flow_warp(const flow_args* a, const uint8_t* f, float px, float py, float bgr[3])
{
    const float fx0 = floorf(px), fy0 = floorf(py);
    const float fx = px - fx0, fy = py - fy0;
    /* clamp in float first: a flow can put the tap far outside the int range */
    const float cx0 = fx0 < -1.0f ? -1.0f : (fx0 > (float)a->W ? (float)a->W : fx0);
    const float cy0 = fy0 < -1.0f ? -1.0f : (fy0 > (float)a->H ? (float)a->H : fy0);
    const int x0 = (int)cx0, y0 = (int)cy0;
    const int xa = clampi(x0, 0, a->W - 1), xb = clampi(x0 + 1, 0, a->W - 1);
    const int ya = clampi(y0, 0, a->H - 1), yb = clampi(y0 + 1, 0, a->H - 1);
    for (int k = 0; k < 3; ++k) {
        const int byte = 2 - k; /* B, G, R */
        const float p00 = (float)f[((size_t)ya * a->W + xa) * 4 + byte] / 255.0f;
        const float p01 = (float)f[((size_t)ya * a->W + xb) * 4 + byte] / 255.0f;
        const float p10 = (float)f[((size_t)yb * a->W + xa) * 4 + byte] / 255.0f;
        const float p11 = (float)f[((size_t)yb * a->W + xb) * 4 + byte] / 255.0f;
        bgr[k] = flow_mix(flow_mix(p00, p01, fx), flow_mix(p10, p11, fx), fy);
    }
}

static void flow_row(const void* p, int y)
{
    const flow_args* a = (const flow_args*)p;
    for (int x = 0; x < a->W; ++x) {
        const float sx = ((float)x + 0.5f) * 0.125f - 0.5f;
        const float sy = ((float)y + 0.5f) * 0.125f - 0.5f;
        const float u0 = flow_up(a, 0, sx, sy) * 8.0f, v0 = flow_up(a, 1, sx, sy) * 8.0f;
        const float u1 = flow_up(a, 2, sx, sy) * 8.0f, v1 = flow_up(a, 3, sx, sy) * 8.0f;
        const float m = 1.0f / (1.0f + flow_exp(-flow_up(a, 4, sx, sy)));
        float w0[3], w1[3];
        flow_warp(a, a->f0, (float)x + u0, (float)y + v0, w0);
        flow_warp(a, a->f1, (float)x + u1, (float)y + v1, w1);
        const float om = 1.0f - m;
        /* refine residual: its x4 bilinear upsample (align_corners=false,
         * clamped taps), added before the clamp */
        float rv[3] = {0.0f, 0.0f, 0.0f};
        if (a->res) {
            const int RH = a->H / 4, RW = a->W / 4;
            const float rx = ((float)x + 0.5f) * 0.25f - 0.5f;
            const float ry = ((float)y + 0.5f) * 0.25f - 0.5f;
            const float fx0 = floorf(rx), fy0 = floorf(ry);
            const float fx = rx - fx0, fy = ry - fy0;
            const int xa = clampi((int)fx0, 0, RW - 1), xb = clampi((int)fx0 + 1, 0, RW - 1);
            const int ya = clampi((int)fy0, 0, RH - 1), yb = clampi((int)fy0 + 1, 0, RH - 1);
            for (int k = 0; k < 3; ++k) {
                const float* pl = a->res + (size_t)k * RH * RW;
                const float top = flow_mix(pl[(size_t)ya * RW + xa], pl[(size_t)ya * RW + xb], fx);
                const float bot = flow_mix(pl[(size_t)yb * RW + xa], pl[(size_t)yb * RW + xb], fx);
                rv[k] = flow_mix(top, bot, fy);
            }
        }
        uint8_t* o = a->out + ((size_t)y * a->W + x) * 4;
        for (int k = 0; k < 3; ++k) { /* k: B, G, R -> byte 2 - k */
            const float u = w0[k] * m;
            const float v = w1[k] * om;
            float c = u + v;
            if (a->res) c = c + rv[k];
            c = c < 0.0f ? 0.0f : (c > 1.0f ? 1.0f : c);
            if (a->pre) a->pre[(size_t)(2 - k) * a->H * a->W + (size_t)y * a->W + x] = c;
            o[2 - k] = (uint8_t)(unsigned)(c * 255.0f);
        }
        o[3] = 255;
    }
}

/* H, W multiples of 8; tmp8 [5][H/8][W/8] float; frames [H][W][4] bytes;
 * res (optional) the refine residual [3][H/4][W/4] float (B, G, R); out
 * [H][W][4] bytes (R, G, B, 255); pre (optional) [3][H][W] the clamped R, G, B
 * values before the byte scale. */
int oracle_flow_out(int H, int W, const float* tmp8, const uint8_t* rgba0, const uint8_t* rgba1,
                    const float* res, uint8_t* out, float* pre, int nthreads)
{
    if (H <= 0 || W <= 0 || H % 8 || W % 8) return -1;
    flow_args a = {H, W, tmp8, rgba0, rgba1, res, pre, out};
    for_rows(flow_row, &a, H, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* t-factored frame stack (NEXT-3), P3 createRT's tfact path:                */
/*   FiLM (wgslFilm + filmParams): per timestep t a tiny MLP gives 2C values  */
/*   s = b2 + W2 relu(w0 t + b0); x' = x * (1 + s[c]) + s[C + c].            */
/*   Refine prep (wgslRefinePrep): 11 planes at (H/4, W/4), each the mean     */
/*   over the centre 2x2 of the 4x4 block (X = 4 hx + {1, 2}, Y likewise) of  */
/*   warped frame 0 (B, G, R), warped frame 1 (B, G, R), the sigmoid mask,    */
/*   and the four x8 flows scaled by 0.25 / 20.                               */
/*   Refine out (wgslRefineOut): conv3x3 C -> 3 with replicate (clamped)      */
/*   padding, bias, then 2 sigmoid(acc) - 1.                                  */
/* These values are not truncated to bytes, so they are computed in double.   */
/* ------------------------------------------------------------------------ */
int oracle_film(int C, int N, const double* x, double t, const double* w0, const double* b0,
                int HN, const double* w2, const double* b2, double* y)
{
    double* h = (double*)malloc(sizeof(double) * (size_t)HN);
    double* s = (double*)malloc(sizeof(double) * (size_t)2 * C);
    for (int j = 0; j < HN; ++j) {
        const double v = w0[j] * t + b0[j];
        h[j] = v > 0.0 ? v : 0.0;
    }
    for (int k = 0; k < 2 * C; ++k) {
        double acc = b2[k];
        for (int j = 0; j < HN; ++j) acc += w2[(size_t)k * HN + j] * h[j];
        s[k] = acc;
    }
    for (int c = 0; c < C; ++c)
        for (int i = 0; i < N; ++i)
            y[(size_t)c * N + i] = x[(size_t)c * N + i] * (1.0 + s[c]) + s[C + c];
    free(h);
    free(s);
    return 0;
}

static double rp_up(const double* t, int TH, int TW, int c, double sx, double sy)
{
    const double x0 = floor(sx), y0 = floor(sy), fx = sx - x0, fy = sy - y0;
    const double* pl = t + (size_t)c * TH * TW;
    const int xa = clampi((int)x0, 0, TW - 1), xb = clampi((int)x0 + 1, 0, TW - 1);
    const int ya = clampi((int)y0, 0, TH - 1), yb = clampi((int)y0 + 1, 0, TH - 1);
    const double top = pl[(size_t)ya * TW + xa] * (1 - fx) + pl[(size_t)ya * TW + xb] * fx;
    const double bot = pl[(size_t)yb * TW + xa] * (1 - fx) + pl[(size_t)yb * TW + xb] * fx;
    return top * (1 - fy) + bot * fy;
}

static void rp_warp(const uint8_t* f, int H, int W, double px, double py, double bgr[3])
{
    double x0 = floor(px), y0 = floor(py);
    const double fx = px - x0, fy = py - y0;
    if (x0 < -1) x0 = -1;
    if (x0 > W) x0 = W;
    if (y0 < -1) y0 = -1;
    if (y0 > H) y0 = H;
    const int xa = clampi((int)x0, 0, W - 1), xb = clampi((int)x0 + 1, 0, W - 1);
    const int ya = clampi((int)y0, 0, H - 1), yb = clampi((int)y0 + 1, 0, H - 1);
    for (int k = 0; k < 3; ++k) {
        const int byte = 2 - k;
        const double p00 = f[((size_t)ya * W + xa) * 4 + byte] / 255.0;
        const double p01 = f[((size_t)ya * W + xb) * 4 + byte] / 255.0;
        const double p10 = f[((size_t)yb * W + xa) * 4 + byte] / 255.0;
        const double p11 = f[((size_t)yb * W + xb) * 4 + byte] / 255.0;
        const double top = p00 * (1 - fx) + p01 * fx, bot = p10 * (1 - fx) + p11 * fx;
        bgr[k] = top * (1 - fy) + bot * fy;
    }
}

/* tmp8 [5][H/8][W/8]; frames [H][W][4]; y [11][H/4][W/4]. */
int oracle_refine_prep(int H, int W, const double* tmp8, const uint8_t* rgba0,
                       const uint8_t* rgba1, double* y)
{
    if (H <= 0 || W <= 0 || H % 8 || W % 8) return -1;
    const int TH = H / 8, TW = W / 8, QH = H / 4, QW = W / 4;
    const size_t P = (size_t)QH * QW;
    for (int hy = 0; hy < QH; ++hy)
        for (int hx = 0; hx < QW; ++hx) {
            double acc[11] = {0};
            for (int sy = 1; sy <= 2; ++sy)
                for (int sxp = 1; sxp <= 2; ++sxp) {
                    const int X = 4 * hx + sxp, Y = 4 * hy + sy;
                    const double gx = (X + 0.5) / 8.0 - 0.5, gy = (Y + 0.5) / 8.0 - 0.5;
                    const double u0 = rp_up(tmp8, TH, TW, 0, gx, gy) * 8.0;
                    const double v0 = rp_up(tmp8, TH, TW, 1, gx, gy) * 8.0;
                    const double u1 = rp_up(tmp8, TH, TW, 2, gx, gy) * 8.0;
                    const double v1 = rp_up(tmp8, TH, TW, 3, gx, gy) * 8.0;
                    const double m = 1.0 / (1.0 + exp(-rp_up(tmp8, TH, TW, 4, gx, gy)));
                    double w0[3], w1[3];
                    rp_warp(rgba0, H, W, X + u0, Y + v0, w0);
                    rp_warp(rgba1, H, W, X + u1, Y + v1, w1);
                    for (int k = 0; k < 3; ++k) {
                        acc[k] += w0[k];
                        acc[3 + k] += w1[k];
                    }
                    acc[6] += m;
                    acc[7] += u0;
                    acc[8] += v0;
                    acc[9] += u1;
                    acc[10] += v1;
                }
            const size_t o = (size_t)hy * QW + hx;
            for (int k = 0; k < 7; ++k) y[k * P + o] = acc[k] * 0.25;
            for (int k = 7; k < 11; ++k) y[k * P + o] = acc[k] * (0.25 * (0.25 / 20.0));
        }
    return 0;
}

/* x [C][HH][HW]; w [3][C][3][3]; b [3]; y [3][HH][HW]. */
int oracle_refine_out(int C, int HH, int HW, const double* x, const double* w, const double* b,
                      double* y)
{
    for (int co = 0; co < 3; ++co)
        for (int oy = 0; oy < HH; ++oy)
            for (int ox = 0; ox < HW; ++ox) {
                double acc = b[co];
                for (int ci = 0; ci < C; ++ci)
                    for (int ky = 0; ky < 3; ++ky) {
                        const int iy = clampi(oy + ky - 1, 0, HH - 1);
                        for (int kx = 0; kx < 3; ++kx) {
                            const int ix = clampi(ox + kx - 1, 0, HW - 1);
                            acc += x[((size_t)ci * HH + iy) * HW + ix] *
                                   w[(((size_t)co * C + ci) * 3 + ky) * 3 + kx];
                        }
                    }
                y[((size_t)co * HH + oy) * HW + ox] = 2.0 / (1.0 + exp(-acc)) - 1.0;
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* storage rounding: round-to-nearest-even to binary32, binary16 or bfloat16. */
/* A format with p significand bits (implicit bit included) and minimum       */
/* normal exponent emin has, for |v| in [2^e, 2^(e+1)), the quantum            */
/* 2^(max(e, emin) - p + 1); below 2^emin the quantum stays 2^(emin - p + 1)   */
/* (subnormals).  Rounding |v| / quantum to the nearest integer, ties to even, */
/* then scaling back is exact in double.  Results above the largest finite    */
/* value after rounding become infinity.                                      */
/* ------------------------------------------------------------------------ */
static double round_to_format(double v, int p, int emin, double maxfinite)
{
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    frexp(v, &e); /* v = m * 2^e, 0.5 <= |m| < 1, so |v| in [2^(e-1), 2^e) */
    int ex = e - 1;
    if (ex < emin) ex = emin;
    double q = ldexp(1.0, ex - p + 1);
    double r = nearbyint(v / q) * q; /* default rounding mode: to nearest, ties to even */
    if (fabs(r) > maxfinite) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round_value(double v, int dtype)
{
    switch (dtype) {
    case O_F32: return round_to_format(v, 24, -126, 3.4028234663852886e38);
    case O_F16: return round_to_format(v, 11, -14, 65504.0);
    case O_BF16: return round_to_format(v, 8, -126, 3.3895313892515355e38);
    default: return v;
    }
}

void oracle_round_storage(double* v, size_t n, int dtype)
{
    for (size_t i = 0; i < n; ++i) v[i] = oracle_round_value(v[i], dtype);
}
