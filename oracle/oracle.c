/*
 * Plain CPU oracle for the fused NHWC convolution layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library, and it includes nothing from it.
 *
 * What it computes is the plain definition of the layer, written out as
 * nested loops in the order a reader checks it against:
 *
 *   - the convolution is a cross-correlation (no kernel flip), the convention
 *     of the PyTorch layers the nanoinfer page checks its engine against
 *     ("nanoinfer", parity section) and that its im2col identity assumes
 *     ("nanoinfer", "1x1 convolutions are already a GEMM");
 *   - padding is zero outside the image, with one pad per axis applied on both
 *     sides (the keyword-spotting stem of "nanoinfer", "Asymmetric padding
 *     collapsed to one axis": a 10x4 kernel with padding (5, 1));
 *   - the output size follows the PyTorch rule floor((H + 2p - k) / S) + 1;
 *   - the epilogue adds the bias, then applies ReLU or Mish, where
 *     Mish(x) = x * tanh(ln(1 + e^x)) ("YOLOv4, optimized for Wormhole",
 *     section 7, the Mish / HardMish definition table);
 *   - int8 layers accumulate exactly, add an int32 bias, and requantise per
 *     output channel with symmetric scales and no zero point ("nanoinfer",
 *     post-training quantization: symmetric per-output-channel weight scales);
 *     the multiplier M[co] = s_x * s_w[co] / s_y is formed once in double and
 *     rounded once to float, the accumulator is rounded to float, multiplied
 *     by M[co] in one float multiply, rounded half-to-even to an integer and
 *     saturated to [-128, 127].
 *
 * Float layers are evaluated in double from the exact values of their fp32 or
 * bf16 inputs; int8 layers in int64.  Parallelism (OpenMP over output rows)
 * does not change any result: every output element is computed by one thread
 * in a fixed loop order.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math: the
 * requantisation must round exactly as IEEE single precision does).
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_MISH = 2 };

/* Output extent of one spatial axis: floor((in + 2*pad - k) / stride) + 1,
 * or -1 when no output position fits (the PyTorch shape rule). */
int oracle_output_dim(int in, int k, int pad, int stride)
{
    if (in < 0 || k < 1 || pad < 0 || stride < 1) return -1;
    int span = in + 2 * pad - k;
    if (span < 0) return -1;
    return span / stride + 1;
}

/* softplus(v) = ln(1 + e^v), evaluated without overflow. */
static double softplus(double v)
{
    return fmax(v, 0.0) + log1p(exp(-fabs(v)));
}

/* Mish(v) = v * tanh(softplus(v)). */
double oracle_mish(double v)
{
    return v * tanh(softplus(v));
}

static double activate(double v, int act)
{
    if (act == ORACLE_ACT_RELU) return v > 0.0 ? v : 0.0;
    if (act == ORACLE_ACT_MISH) return oracle_mish(v);
    return v;
}

/* Index helpers for the NHWC input/output and OHWI weight layouts. */
static size_t nhwc(int n, int h, int w, int c, int H, int W, int C)
{
    return (((size_t)n * H + h) * W + w) * C + c;
}

static size_t ohwi(int co, int r, int s, int j, int KH, int KW, int CPG)
{
    return (((size_t)co * KH + r) * KW + s) * CPG + j;
}

/* One output element of a float layer, before the epilogue: the sum over the
 * taps (r, s) and the input channels j of this output channel's group. */
static double point_f64(const double *x, const double *w, int n, int oh, int ow,
                        int co, int H, int W, int Cin, int Cout, int KH, int KW,
                        int stride, int pad_h, int pad_w, int groups)
{
    int cin_g = Cin / groups;
    int cout_g = Cout / groups;
    int g0 = (co / cout_g) * cin_g; /* first input channel of co's group */
    double acc = 0.0;
    for (int r = 0; r < KH; r++) {
        int ih = oh * stride - pad_h + r;
        if (ih < 0 || ih >= H) continue; /* zero padding */
        for (int s = 0; s < KW; s++) {
            int iw = ow * stride - pad_w + s;
            if (iw < 0 || iw >= W) continue;
            for (int j = 0; j < cin_g; j++)
                acc += x[nhwc(n, ih, iw, g0 + j, H, W, Cin)] *
                       w[ohwi(co, r, s, j, KH, KW, cin_g)];
        }
    }
    return acc;
}

static int64_t point_i64(const int8_t *x, const int8_t *w, int n, int oh, int ow,
                         int co, int H, int W, int Cin, int Cout, int KH, int KW,
                         int stride, int pad_h, int pad_w, int groups)
{
    int cin_g = Cin / groups;
    int cout_g = Cout / groups;
    int g0 = (co / cout_g) * cin_g;
    int64_t acc = 0;
    for (int r = 0; r < KH; r++) {
        int ih = oh * stride - pad_h + r;
        if (ih < 0 || ih >= H) continue;
        for (int s = 0; s < KW; s++) {
            int iw = ow * stride - pad_w + s;
            if (iw < 0 || iw >= W) continue;
            for (int j = 0; j < cin_g; j++)
                acc += (int64_t)x[nhwc(n, ih, iw, g0 + j, H, W, Cin)] *
                       (int64_t)w[ohwi(co, r, s, j, KH, KW, cin_g)];
        }
    }
    return acc;
}

static int check_args(int N, int H, int W, int Cin, int Cout, int KH, int KW,
                      int stride, int pad_h, int pad_w, int groups,
                      int *OH, int *OW)
{
    if (N < 0 || H < 1 || W < 1 || Cin < 1 || Cout < 1 || groups < 1) return -1;
    if (Cin % groups != 0 || Cout % groups != 0) return -1;
    *OH = oracle_output_dim(H, KH, pad_h, stride);
    *OW = oracle_output_dim(W, KW, pad_w, stride);
    if (*OH < 1 || *OW < 1) return -1;
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Float layer: y = act(conv(x, w) + b), all in double.  b may be NULL
 * (no bias).  Returns 0, or -1 on an invalid shape. */
int oracle_conv_f64(const double *x, const double *w, const double *b, double *y,
                    int N, int H, int W, int Cin, int Cout, int KH, int KW,
                    int stride, int pad_h, int pad_w, int groups, int act,
                    int nthreads)
{
    int OH, OW;
    if (check_args(N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                   &OH, &OW))
        return -1;
    set_threads(nthreads);
    long rows = (long)N * OH;
#pragma omp parallel for schedule(dynamic)
    for (long row = 0; row < rows; row++) {
        int n = (int)(row / OH), oh = (int)(row % OH);
        for (int ow = 0; ow < OW; ow++)
            for (int co = 0; co < Cout; co++) {
                double v = point_f64(x, w, n, oh, ow, co, H, W, Cin, Cout, KH,
                                     KW, stride, pad_h, pad_w, groups);
                if (b) v += b[co];
                y[nhwc(n, oh, ow, co, OH, OW, Cout)] = activate(v, act);
            }
    }
    return 0;
}

/* Float layer at selected output points only: pts holds npts quadruples
 * (n, oh, ow, co); vals[i] receives act(conv + b) at point i. */
int oracle_conv_f64_points(const double *x, const double *w, const double *b,
                           const int32_t *pts, long npts, double *vals,
                           int N, int H, int W, int Cin, int Cout, int KH, int KW,
                           int stride, int pad_h, int pad_w, int groups, int act,
                           int nthreads)
{
    int OH, OW;
    if (check_args(N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                   &OH, &OW))
        return -1;
    for (long i = 0; i < npts; i++) {
        const int32_t *p = pts + 4 * i;
        if (p[0] < 0 || p[0] >= N || p[1] < 0 || p[1] >= OH || p[2] < 0 ||
            p[2] >= OW || p[3] < 0 || p[3] >= Cout)
            return -1;
    }
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < npts; i++) {
        const int32_t *p = pts + 4 * i;
        double v = point_f64(x, w, p[0], p[1], p[2], p[3], H, W, Cin, Cout, KH,
                             KW, stride, pad_h, pad_w, groups);
        if (b) v += b[p[3]];
        vals[i] = activate(v, act);
    }
    return 0;
}

/* Requantisation multipliers: M[co] = float(s_x * s_w[co] / s_y), the
 * product and quotient taken in double and rounded once to float. */
int oracle_requant_multipliers(float in_scale, float out_scale,
                               const float *w_scales, int Cout, float *M)
{
    if (!(out_scale > 0.0f) || !(in_scale > 0.0f)) return -1;
    for (int co = 0; co < Cout; co++) {
        if (!(w_scales[co] > 0.0f)) return -1;
        M[co] = (float)((double)in_scale * (double)w_scales[co] /
                        (double)out_scale);
    }
    return 0;
}

/* q = sat_[-128,127]( rne( float(v) * M ) ), each step rounded to nearest,
 * ties to even, as IEEE single precision does; then ReLU as max(q, 0). */
int oracle_requant_one(int64_t v, float M, int relu)
{
    float fv = (float)v;        /* integer -> float, round to nearest even */
    volatile float p = fv * M;  /* one single-precision multiply */
    float r = nearbyintf(p);    /* round half to even (FE_TONEAREST) */
    if (r > 127.0f) r = 127.0f;
    if (r < -128.0f) r = -128.0f;
    int q = (int)r;
    if (relu && q < 0) q = 0;
    return q;
}

/* Raw int8 accumulators (int64, no bias), for invariant checks. */
int oracle_conv_i8_acc(const int8_t *x, const int8_t *w, int64_t *acc,
                       int N, int H, int W, int Cin, int Cout, int KH, int KW,
                       int stride, int pad_h, int pad_w, int groups, int nthreads)
{
    int OH, OW;
    if (check_args(N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                   &OH, &OW))
        return -1;
    set_threads(nthreads);
    long rows = (long)N * OH;
#pragma omp parallel for schedule(dynamic)
    for (long row = 0; row < rows; row++) {
        int n = (int)(row / OH), oh = (int)(row % OH);
        for (int ow = 0; ow < OW; ow++)
            for (int co = 0; co < Cout; co++)
                acc[nhwc(n, oh, ow, co, OH, OW, Cout)] =
                    point_i64(x, w, n, oh, ow, co, H, W, Cin, Cout, KH, KW,
                              stride, pad_h, pad_w, groups);
    }
    return 0;
}

/* int8 layer: y = requant(conv(x, w) + b) with M[co] from
 * oracle_requant_multipliers.  b (int32) may be NULL. */
int oracle_conv_i8(const int8_t *x, const int8_t *w, const int32_t *b,
                   const float *M, int8_t *y, int N, int H, int W, int Cin,
                   int Cout, int KH, int KW, int stride, int pad_h, int pad_w,
                   int groups, int relu, int nthreads)
{
    int OH, OW;
    if (check_args(N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                   &OH, &OW))
        return -1;
    if (fegetround() != FE_TONEAREST) fesetround(FE_TONEAREST);
    set_threads(nthreads);
    long rows = (long)N * OH;
#pragma omp parallel for schedule(dynamic)
    for (long row = 0; row < rows; row++) {
        int n = (int)(row / OH), oh = (int)(row % OH);
        for (int ow = 0; ow < OW; ow++)
            for (int co = 0; co < Cout; co++) {
                int64_t v = point_i64(x, w, n, oh, ow, co, H, W, Cin, Cout, KH,
                                      KW, stride, pad_h, pad_w, groups);
                if (b) v += b[co];
                y[nhwc(n, oh, ow, co, OH, OW, Cout)] =
                    (int8_t)oracle_requant_one(v, M[co], relu);
            }
    }
    return 0;
}

/* int8 layer at selected output points (n, oh, ow, co). */
int oracle_conv_i8_points(const int8_t *x, const int8_t *w, const int32_t *b,
                          const float *M, const int32_t *pts, long npts,
                          int8_t *vals, int N, int H, int W, int Cin, int Cout,
                          int KH, int KW, int stride, int pad_h, int pad_w,
                          int groups, int relu, int nthreads)
{
    int OH, OW;
    if (check_args(N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, groups,
                   &OH, &OW))
        return -1;
    for (long i = 0; i < npts; i++) {
        const int32_t *p = pts + 4 * i;
        if (p[0] < 0 || p[0] >= N || p[1] < 0 || p[1] >= OH || p[2] < 0 ||
            p[2] >= OW || p[3] < 0 || p[3] >= Cout)
            return -1;
    }
    if (fegetround() != FE_TONEAREST) fesetround(FE_TONEAREST);
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < npts; i++) {
        const int32_t *p = pts + 4 * i;
        int64_t v = point_i64(x, w, p[0], p[1], p[2], p[3], H, W, Cin, Cout, KH,
                              KW, stride, pad_h, pad_w, groups);
        if (b) v += b[p[3]];
        vals[i] = (int8_t)oracle_requant_one(v, M[p[3]], relu);
    }
    return 0;
}

/* Number of threads an OpenMP region started now would use. */
int oracle_max_threads(int nthreads)
{
    set_threads(nthreads);
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Max pooling with stride 1 and an output the size of the input: a k x k
 * window (k odd) centred on every pixel, positions outside the image left out
 * of the max (they never win it).  These are the three pools (k = 5, 9, 13)
 * of the YOLOv4 SPP block ("YOLOv4, optimized for Wormhole", section 9, K3).
 * Evaluated directly over the whole window -- not as the cascade of smaller
 * windows the fast kernel uses, so that the cascade identity is checked
 * rather than assumed.  x, y NHWC, C channels; exact for any input values.
 */
int oracle_maxpool_same(const double *x, double *y, int N, int H, int W, int C, int k, int nthreads)
{
    if (!x || !y || N < 0 || H < 1 || W < 1 || C < 1 || k < 1 || (k % 2) == 0)
        return -1;
    set_threads(nthreads);
    const int r = k / 2;
    const long long rows = (long long)N * H;
#pragma omp parallel for schedule(static)
    for (long long nh = 0; nh < rows; ++nh) {
        const int n = (int)(nh / H), h = (int)(nh % H);
        for (int w = 0; w < W; ++w)
            for (int c = 0; c < C; ++c) {
                double m = -INFINITY;
                for (int i = h - r; i <= h + r; ++i) {
                    if (i < 0 || i >= H)
                        continue;
                    for (int j = w - r; j <= w + r; ++j) {
                        if (j < 0 || j >= W)
                            continue;
                        const double v = x[(((long long)n * H + i) * W + j) * C + c];
                        if (v > m)
                            m = v;
                    }
                }
                y[(((long long)n * H + h) * W + w) * C + c] = m;
            }
    }
    return 0;
}
