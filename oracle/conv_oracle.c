/*
 * CPU oracle for the INT8 Conv2d forward pass (fprop) -- TEST INFRASTRUCTURE.
 *
 * This file is the plain, slow, obviously correct definition that the GPU
 * implicit-GEMM kernels are checked against.  It shares no code with the
 * GPU path.  Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline and reference legs may load it; the product path never
 * calls it.
 *
 * What it computes (written out from the pages, not from any listing):
 *  - Output extent per axis (kernel-benchmark trace, page 4, first analysis
 *    paragraph):  P = floor((H + 2*pad - dil*(R-1) - 1) / stride) + 1.
 *  - Direct convolution on plain NCHW activations and KCRS filters (the
 *    nn.Conv2d weight order used on page 4), with zero padding:
 *        acc[n][k][p][q] = sum_{c<C} sum_{r<R} sum_{s<S}
 *              [0 <= h < H and 0 <= w < W] * x[n][c][h][w] * f[k][c][r][s],
 *        h = p*stride_h - pad_h + r*dil_h,  w = q*stride_w - pad_w + s*dil_w
 *    (page 4, implicit-GEMM paragraph: k -> (ic, kh, kw), ih = oh*stride +
 *    kh*dil - pad; out-of-bounds taps contribute zero).  The sum is taken in
 *    int64 so it cannot overflow.
 *  - The alpha-only clamp epilogue of the CUTLASS configuration on page 1
 *    (LinearCombinationClamp<int8, 8, int32, float, OnlyAlphaScaling>):
 *        y = clamp(rint(alpha * (float)acc32), -128, 127)
 *    where acc32 is the int32 accumulator, (float) rounds to nearest even,
 *    the product is one single-precision multiply (no FMA, no double), and
 *    rint rounds half to even.
 *
 *  - The per-output-channel epilogue (the "row-wise scaling" of the
 *    weight-only quantisation issue on page 2, with a bias and a ReLU fused
 *    before the clamp):
 *        y = clamp(rint(relu(alpha_k * (float)acc32 + bias_k)), -128, 127)
 *    alpha_k the scale of output channel k (or the one alpha), one fp32
 *    multiply, then one fp32 add of bias_k (round to nearest even each, no
 *    FMA), relu(v) = max(v, 0) when asked for.  With alpha_k = alpha, no bias
 *    and no ReLU it is the clamp epilogue above.
 *
 *  - The fp32 direct convolution of the kernel-benchmark trace (page 4):
 *    nn.Conv2d on fp32 NCHW input and KCRS weight with an optional bias,
 *    the same tap indexing and zero padding as above, which the trace checks
 *    against the framework's own convolution with atol = rtol = 1e-4:
 *        y[n][k][p][q] = bias[k] + sum_{c,r,s} x[n][c][h][w] * w[k][c][r][s]
 *    evaluated here in double (each fp32 product is exact in double), with
 *    the magnitude sum |bias[k]| + sum |x * w| beside it: any fp32
 *    evaluation of the same sum, in any order, lies within
 *    (C*R*S + 1) * 2^-24 / (1 - (C*R*S + 1) * 2^-24) times that magnitude of
 *    the exact value (the standard bound for recursive summation).
 *
 * Built with -ffp-contract=off and without fast-math so the epilogue is the
 * IEEE single-precision sequence described above on both x86-64 and AArch64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#pragma STDC FP_CONTRACT OFF

/* Optional planted mistakes, used only by the test that proves the oracle's
 * pins catch plausible errors.  ORACLE_MUTATION == 0 is the real oracle. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

typedef struct {
    int64_t N, C, H, W, K, R, S;
    int64_t pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
} oracle_shape;

enum { ORACLE_OK = 0, ORACLE_EINVAL = 1, ORACLE_ERANGE = 2, ORACLE_ENOMEM = 3 };

/* Output extent along one spatial axis (page 4's formula).  A negative
 * numerator means the dilated filter does not fit: the extent is 0. */
int64_t oracle_out_extent(int64_t in, int64_t pad, int64_t dil, int64_t k, int64_t stride)
{
    if (in < 1 || pad < 0 || dil < 1 || k < 1 || stride < 1) return -1;
    int64_t num = in + 2 * pad - dil * (k - 1) - 1;
#if ORACLE_MUTATION == 8
    num = in + 2 * pad - dil * k - 1;          /* planted: effective extent off by one dilation */
#endif
    if (num < 0) return 0;
    return num / stride + 1;
}

static int shape_ok(const oracle_shape *s)
{
    if (!s) return 0;
    if (s->N < 1 || s->C < 1 || s->H < 1 || s->W < 1 || s->K < 1 || s->R < 1 || s->S < 1) return 0;
    if (s->pad_h < 0 || s->pad_w < 0 || s->stride_h < 1 || s->stride_w < 1 || s->dil_h < 1 || s->dil_w < 1) return 0;
    return 1;
}

/* One accumulator, straight from the definition. */
static int64_t acc_at(const int8_t *x, const int8_t *f, const oracle_shape *s,
                      int64_t n, int64_t k, int64_t p, int64_t q)
{
    int64_t sum = 0;
    for (int64_t c = 0; c < s->C; ++c) {
#if ORACLE_MUTATION == 7
        if (c == s->C - 1) break;              /* planted: last input channel dropped */
#endif
        for (int64_t r = 0; r < s->R; ++r) {
            int64_t h = p * s->stride_h - s->pad_h + r * s->dil_h;
#if ORACLE_MUTATION == 2
            h = p * s->stride_h + s->pad_h + r * s->dil_h;   /* planted: padding sign flipped */
#elif ORACLE_MUTATION == 3
            h = p * s->stride_h - s->pad_h + r * s->dil_w;   /* planted: dilation axes crossed */
#endif
            for (int64_t t = 0; t < s->S; ++t) {
                int64_t w = q * s->stride_w - s->pad_w + t * s->dil_w;
#if ORACLE_MUTATION == 4
                w = q - s->pad_w + t * s->dil_w;              /* planted: column stride ignored */
#endif
                if (h < 0 || h >= s->H || w < 0 || w >= s->W) continue;
                int64_t xv = x[((n * s->C + c) * s->H + h) * s->W + w];
                int64_t fi = ((k * s->C + c) * s->R + r) * s->S + t;
#if ORACLE_MUTATION == 1
                if (s->R == s->S) fi = ((k * s->C + c) * s->R + t) * s->S + r;  /* planted: filter taps transposed */
                else fi = ((k * s->C + c) * s->R + r) * s->S + (s->S - 1 - t);  /* planted: filter columns mirrored */
#endif
                int64_t fv = f[fi];
                sum += xv * fv;
            }
        }
    }
    return sum;
}

typedef struct {
    const int8_t *x, *f;
    int64_t *acc;
    const oracle_shape *s;
    int64_t P, Q;
    int64_t first, last; /* range of (n, k) pairs */
} job_t;

static void *run_job(void *arg)
{
    job_t *j = (job_t *)arg;
    const oracle_shape *s = j->s;
    for (int64_t nk = j->first; nk < j->last; ++nk) {
        int64_t n = nk / s->K, k = nk % s->K;
        int64_t *out = j->acc + nk * j->P * j->Q;
        for (int64_t p = 0; p < j->P; ++p)
            for (int64_t q = 0; q < j->Q; ++q)
                out[p * j->Q + q] = acc_at(j->x, j->f, s, n, k, p, q);
    }
    return NULL;
}

/* Full convolution.  x: NCHW int8, f: KCRS int8, acc: NKPQ int64 (caller
 * allocates N*K*P*Q).  Work is split over (n, k) pairs across nthreads
 * threads; each accumulator is computed by exactly one thread. */
int oracle_conv2d_acc(const int8_t *x, const int8_t *f, int64_t *acc, const oracle_shape *s, int nthreads)
{
    if (!x || !f || !acc || !shape_ok(s)) return ORACLE_EINVAL;
    int64_t P = oracle_out_extent(s->H, s->pad_h, s->dil_h, s->R, s->stride_h);
    int64_t Q = oracle_out_extent(s->W, s->pad_w, s->dil_w, s->S, s->stride_w);
    if (P <= 0 || Q <= 0) return ORACLE_OK;
    int64_t pairs = s->N * s->K;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = (int)pairs;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return ORACLE_ENOMEM; }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (job_t){x, f, acc, s, P, Q, pairs * i / nthreads, pairs * (i + 1) / nthreads};
        if (i == 0) continue;
        if (pthread_create(&tid[i], NULL, run_job, &jobs[i]) == 0) { ++started; }
        else { run_job(&jobs[i]); tid[i] = 0; }
    }
    run_job(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (tid[i]) pthread_join(tid[i], NULL);
    (void)started;
    free(jobs);
    free(tid);
    return ORACLE_OK;
}

/* Accumulators at a list of output coordinates: pts holds npts rows of
 * (n, k, p, q).  Used to check full-size GPU outputs point by point. */
int oracle_conv2d_acc_points(const int8_t *x, const int8_t *f, const oracle_shape *s,
                             const int64_t *pts, int64_t npts, int64_t *out)
{
    if (!x || !f || !pts || !out || !shape_ok(s) || npts < 0) return ORACLE_EINVAL;
    int64_t P = oracle_out_extent(s->H, s->pad_h, s->dil_h, s->R, s->stride_h);
    int64_t Q = oracle_out_extent(s->W, s->pad_w, s->dil_w, s->S, s->stride_w);
    for (int64_t i = 0; i < npts; ++i) {
        int64_t n = pts[4 * i], k = pts[4 * i + 1], p = pts[4 * i + 2], q = pts[4 * i + 3];
        if (n < 0 || n >= s->N || k < 0 || k >= s->K || p < 0 || p >= P || q < 0 || q >= Q) return ORACLE_EINVAL;
        out[i] = acc_at(x, f, s, n, k, p, q);
    }
    return ORACLE_OK;
}

/* The clamp epilogue on int32 accumulators held as int64.  Returns
 * ORACLE_ERANGE if any accumulator does not fit in int32 (the accumulator
 * type of the page-1 configuration); y is then left partly written. */
int oracle_requantize(const int64_t *acc, int64_t count, float alpha, int8_t *y)
{
    if ((!acc || !y) && count > 0) return ORACLE_EINVAL;
    for (int64_t i = 0; i < count; ++i) {
        if (acc[i] > INT32_MAX || acc[i] < INT32_MIN) return ORACLE_ERANGE;
        int32_t a32 = (int32_t)acc[i];
        volatile float v = (float)a32;         /* int32 -> fp32, round to nearest even */
        volatile float prod = alpha * v;       /* one fp32 multiply */
#if ORACLE_MUTATION == 5
        float r = roundf(prod);                /* planted: ties away from zero */
#else
        float r = rintf(prod);                 /* round half to even (default mode) */
#endif
        if (r > 127.0f) r = 127.0f;
#if ORACLE_MUTATION == 6
        if (r < -127.0f) r = -127.0f;          /* planted: symmetric clamp range */
#else
        if (r < -128.0f) r = -128.0f;
#endif
        y[i] = (int8_t)(int32_t)r;
    }
    return ORACLE_OK;
}

/* The per-output-channel epilogue on int32 accumulators held as int64 in
 * NKPQ order (count = N*K*PQ): alpha_k / bias_k are K floats each (alpha_k
 * NULL: the scalar alpha; bias_k NULL: no bias), relu non-zero: max(v, 0)
 * before the clamp.  ORACLE_ERANGE if an accumulator does not fit in int32. */
int oracle_requantize_channels(const int64_t *acc, int64_t N, int64_t K, int64_t PQ, float alpha,
                               const float *alpha_k, const float *bias_k, int relu, int8_t *y)
{
    if ((!acc || !y) && N * K * PQ > 0) return ORACLE_EINVAL;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
#if ORACLE_MUTATION == 11
            const int64_t kk = n % K;              /* planted: the channel's scale indexed by the image */
#else
            const int64_t kk = k;
#endif
            const float a = alpha_k ? alpha_k[kk] : alpha;
            const float b = bias_k ? bias_k[kk] : 0.0f;
            for (int64_t i = 0; i < PQ; ++i) {
                const int64_t idx = (n * K + k) * PQ + i;
                if (acc[idx] > INT32_MAX || acc[idx] < INT32_MIN) return ORACLE_ERANGE;
                volatile float v = (float)(int32_t)acc[idx];   /* int32 -> fp32, round to nearest even */
#if ORACLE_MUTATION == 9
                volatile float sum = a * (v + b);                /* planted: bias added before the scale */
#elif ORACLE_MUTATION == 12
                volatile float sum = fmaf(a, v, b);              /* planted: one fused multiply-add */
#else
                volatile float prod = a * v;                     /* one fp32 multiply */
                volatile float sum = prod + b;                   /* then one fp32 add */
#endif
                float r = sum;
                if (relu && r < 0.0f) r = 0.0f;
                r = rintf(r);                                    /* round half to even */
                if (r > 127.0f) r = 127.0f;
                if (r < -128.0f) r = -128.0f;
                y[idx] = (int8_t)(int32_t)r;
            }
        }
    return ORACLE_OK;
}

/* One fp32 direct-convolution output in double, and its magnitude sum. */
static void f64_at(const float *x, const float *wt, const float *bias, const oracle_shape *s,
                   int64_t n, int64_t k, int64_t p, int64_t q, double *out, double *mag)
{
    double sum = 0.0, abs_sum = 0.0;
    if (bias) {
#if ORACLE_MUTATION == 16
        const int64_t kb = n % s->K;           /* planted: bias indexed by the image */
#else
        const int64_t kb = k;
#endif
#if ORACLE_MUTATION != 13
        sum = (double)bias[kb];                /* (mutation 13 plants: bias ignored) */
#endif
        abs_sum = fabs((double)bias[kb]);
    }
    for (int64_t c = 0; c < s->C; ++c)
        for (int64_t r = 0; r < s->R; ++r) {
#if ORACLE_MUTATION == 15
            int64_t h = p - s->pad_h + r * s->dil_h;                   /* planted: row stride ignored */
#else
            int64_t h = p * s->stride_h - s->pad_h + r * s->dil_h;
#endif
            if (h < 0 || h >= s->H) continue;
            for (int64_t t = 0; t < s->S; ++t) {
#if ORACLE_MUTATION == 14
                int64_t w = q * s->stride_w - s->pad_w + t;            /* planted: column dilation ignored */
#else
                int64_t w = q * s->stride_w - s->pad_w + t * s->dil_w;
#endif
                if (w < 0 || w >= s->W) continue;
                double prod = (double)x[((n * s->C + c) * s->H + h) * s->W + w] *
                              (double)wt[((k * s->C + c) * s->R + r) * s->S + t];
                sum += prod;
                abs_sum += fabs(prod);
            }
        }
    *out = sum;
    *mag = abs_sum;
}

typedef struct {
    const float *x, *w, *bias;
    double *y, *mag;
    const oracle_shape *s;
    int64_t P, Q, first, last;
} f64_job_t;

static void *run_f64_job(void *arg)
{
    f64_job_t *j = (f64_job_t *)arg;
    const oracle_shape *s = j->s;
    for (int64_t nk = j->first; nk < j->last; ++nk) {
        int64_t n = nk / s->K, k = nk % s->K;
        for (int64_t p = 0; p < j->P; ++p)
            for (int64_t q = 0; q < j->Q; ++q) {
                int64_t i = (nk * j->P + p) * j->Q + q;
                f64_at(j->x, j->w, j->bias, s, n, k, p, q, &j->y[i], &j->mag[i]);
            }
    }
    return NULL;
}

/* fp32 direct convolution in double.  x: NCHW float, w: KCRS float, bias: K
 * floats or NULL; y and mag: NKPQ doubles (caller allocates N*K*P*Q each).
 * Threaded over (n, k) pairs like oracle_conv2d_acc. */
int oracle_conv2d_f64(const float *x, const float *w, const float *bias, double *y, double *mag,
                      const oracle_shape *s, int nthreads)
{
    if (!x || !w || !y || !mag || !shape_ok(s)) return ORACLE_EINVAL;
    int64_t P = oracle_out_extent(s->H, s->pad_h, s->dil_h, s->R, s->stride_h);
    int64_t Q = oracle_out_extent(s->W, s->pad_w, s->dil_w, s->S, s->stride_w);
    if (P <= 0 || Q <= 0) return ORACLE_OK;
    int64_t pairs = s->N * s->K;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = (int)pairs;
    f64_job_t *jobs = (f64_job_t *)calloc((size_t)nthreads, sizeof(f64_job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return ORACLE_ENOMEM; }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (f64_job_t){x, w, bias, y, mag, s, P, Q, pairs * i / nthreads, pairs * (i + 1) / nthreads};
        if (i == 0) continue;
        if (pthread_create(&tid[i], NULL, run_f64_job, &jobs[i]) != 0) { run_f64_job(&jobs[i]); tid[i] = 0; }
    }
    run_f64_job(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (tid[i]) pthread_join(tid[i], NULL);
    free(jobs);
    free(tid);
    return ORACLE_OK;
}

/* fp32 direct convolution in double at rows (n, k, p, q) of pts. */
int oracle_conv2d_f64_points(const float *x, const float *w, const float *bias, const oracle_shape *s,
                             const int64_t *pts, int64_t npts, double *y, double *mag)
{
    if (!x || !w || !pts || !y || !mag || !shape_ok(s) || npts < 0) return ORACLE_EINVAL;
    int64_t P = oracle_out_extent(s->H, s->pad_h, s->dil_h, s->R, s->stride_h);
    int64_t Q = oracle_out_extent(s->W, s->pad_w, s->dil_w, s->S, s->stride_w);
    for (int64_t i = 0; i < npts; ++i) {
        int64_t n = pts[4 * i], k = pts[4 * i + 1], p = pts[4 * i + 2], q = pts[4 * i + 3];
        if (n < 0 || n >= s->N || k < 0 || k >= s->K || p < 0 || p >= P || q < 0 || q >= Q) return ORACLE_EINVAL;
        f64_at(x, w, bias, s, n, k, p, q, &y[i], &mag[i]);
    }
    return ORACLE_OK;
}

int oracle_mutation_id(void) { return ORACLE_MUTATION; }
