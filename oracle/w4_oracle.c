/*
 * w4_oracle.c -- plain, slow, obviously correct CPU oracle for the W4A16
 * projection.  TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline).
 *
 * Passages followed:
 *  - "Building a Custom LLM Inference Runtime for Qwen2.5-Coder-7B on NVIDIA
 *    H100 Hopper Architecture", "Technical Specifications and Hardware
 *    Alignment": symmetric group-wise INT4 weights, group size 128, one FP16
 *    scale per group; model dimensions 3584 / 18944, 28 layers.
 *  - same page, "The INT8 vs. FP16 Activation Trade-off": activations stay
 *    FP16 (Path B).
 *  - "The Architecture of Modern Inference ...", "Data Integrity and
 *    Serialization: The .nanoqwen Format": symmetric INT4, group 128.
 * Readings where the pages are silent: q is two's-complement 4-bit, [-8, 7];
 * w = q * s; groups run along K within one output row; scales are stored
 * [N, K/128]; the sum is formed in FP64 with k ascending and rounded once
 * to binary16 with ties-to-even.
 */
#include "w4_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- IEEE 754-2008 binary16 ------------------------------------------- */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exponent field 0 encodes subnormals f * 2^-24; field 31 encodes inf/NaN;
 * otherwise the value is (1024 + f) * 2^(e - 25). */
double w4o_double_from_half(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);
    return sign ? -mag : mag;
}

uint16_t w4o_half_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs(v);
    /* 65504 is the largest finite half; the next step would be 65536, so
     * the midpoint 65520 and everything above round to infinity (the tie
     * goes to the even neighbour, 65536 = overflow). */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    /* a = m * 2^E with m in [0.5, 1): the unbiased binary16 exponent of a
     * is E - 1, clamped below at -14 (the subnormal range shares the
     * quantum of the smallest normal binade). */
    int E;
    (void)frexp(a, &E);
    int e = E - 1;
    if (e < -14)
        e = -14;
    /* quantum (one unit in the last place) of that binade: 2^(e - 10) */
    double n = ldexp(a, 10 - e); /* a / quantum, exact (power-of-two scale) */
    double fl = floor(n);
    double frac = n - fl;        /* exact: n < 2^11 */
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    /* r in [0, 2048]: r * 2^(e-10) is the rounded magnitude.  For the
     * subnormal binade (e = -14) the encoding is r itself (r = 1024 gives
     * 0x0400, the smallest normal); for a normal binade it is
     * (e + 15) << 10 | (r - 1024), where r = 2048 carries into the next
     * exponent. */
    unsigned bits;
    if (e == -14 && r < 1024.0)
        bits = (unsigned)r;
    else
        bits = ((unsigned)(e + 15) << 10) + (unsigned)(r - 1024.0);
    return (uint16_t)(sign | bits);
}

/* ---- bfloat16 -------------------------------------------------------------- */
/* bfloat16 (the upper half of IEEE 754 binary32): 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits.  Exponent field 0 encodes subnormals
 * f * 2^-133; field 255 encodes inf/NaN; otherwise the value is
 * (128 + f) * 2^(e - 134). */
double w4o_double_from_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 255;
    int f = b & 127;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133);
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + f), e - 134);
    return sign ? -mag : mag;
}

uint16_t w4o_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    /* largest finite: 255 * 2^120; the next step would be 256 * 2^120 =
     * 2^128, so the midpoint 255.5 * 2^120 and above round to infinity */
    if (a >= ldexp(255.5, 120))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    /* unbiased exponent of a, clamped below at -126 (subnormals share the
     * quantum of the smallest normal binade) */
    int E;
    (void)frexp(a, &E);
    int e = E - 1;
    if (e < -126)
        e = -126;
    double n = ldexp(a, 7 - e); /* a / 2^(e - 7), exact */
    double fl = floor(n);
    double frac = n - fl;
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    /* r in [0, 256]; r = 256 carries into the next exponent */
    unsigned bits;
    if (e == -126 && r < 128.0)
        bits = (unsigned)r;
    else
        bits = ((unsigned)(e + 127) << 7) + (unsigned)(r - 128.0);
    return (uint16_t)(sign | bits);
}

/* ---- INT8 activations (Path A) ------------------------------------------ */
/* Per-token symmetric INT8 quantisation in IEEE binary32 (the precision the
 * GPU takes the same integer decision in): amax = max_k |x|, sx = amax / 127,
 * xq = round-half-even(x / sx), clamped to [-127, 127]; sx = 0 (all-zero row)
 * gives xq = 0. */
void w4o_quantize_x8(const uint16_t* x, int64_t M, int64_t K, int8_t* xq, float* sx)
{
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            const float v = fabsf((float)w4o_double_from_half(x[m * K + k]));
            if (v > amax)
                amax = v;
        }
        const float scale = amax / 127.0f;
        sx[m] = scale;
        for (int64_t k = 0; k < K; ++k) {
            long r = 0;
            if (scale > 0.0f) {
                const float t = (float)w4o_double_from_half(x[m * K + k]) / scale;
                r = lrintf(t); /* default rounding mode: to nearest, ties to even */
                if (r > 127)
                    r = 127;
                if (r < -127)
                    r = -127;
            }
            xq[m * K + k] = (int8_t)r;
        }
    }
}

/* y[m,n] = half_rne( sum_g s[n,g] * sx[m] * sum_{k in g} xq[m,k] * q[n,k] ):
 * the integer group sums exactly (int64), the scaling and the sum over
 * groups in FP64.  acc as in w4o_linear.  Same return codes. */
int w4o_linear_q8(const uint16_t* x, const int8_t* q, const uint16_t* s,
                  int64_t M, int64_t N, int64_t K, uint16_t* y, double* acc)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -1;
    if (M == 0 || N == 0)
        return 0;
    if (!x || !q || !s || !y)
        return -1;
    for (int64_t i = 0; i < N * K; ++i)
        if (q[i] < -8 || q[i] > 7)
            return -2;
    int8_t* xq = (int8_t*)malloc((size_t)(M * K));
    float* sx = (float*)malloc((size_t)M * sizeof(float));
    if (!xq || !sx) {
        free(xq);
        free(sx);
        return -1;
    }
    w4o_quantize_x8(x, M, K, xq, sx);
    const int64_t G = K / 128;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double sum = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t isum = 0;
                for (int64_t k = 128 * g; k < 128 * g + 128; ++k)
                    isum += (int64_t)xq[m * K + k] * (int64_t)q[n * K + k];
                sum += w4o_double_from_half(s[n * G + g]) * (double)sx[m] * (double)isum;
            }
            y[m * N + n] = w4o_half_from_double(sum);
            if (acc)
                acc[m * N + n] = sum;
        }
    }
    free(xq);
    free(sx);
    return 0;
}

/* ---- the projection --------------------------------------------------- */
typedef struct {
    const uint16_t* x;
    const int8_t* q;
    const uint16_t* s;
    int64_t M, N, K;
    uint16_t* y;
    double* acc;
    int64_t n_begin, n_end;
    double (*x_value)(uint16_t);  /* activation decoding (x) */
    uint16_t (*y_bits)(double);   /* output rounding (y) */
} w4o_job;

static void* w4o_rows(void* arg)
{
    const w4o_job* jb = (const w4o_job*)arg;
    const int64_t K = jb->K, G = K / 128;
    for (int64_t n = jb->n_begin; n < jb->n_end; ++n) {
        const int8_t* qn = jb->q + n * K;
        const uint16_t* sn = jb->s + n * G;
        for (int64_t m = 0; m < jb->M; ++m) {
            const uint16_t* xm = jb->x + m * K;
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                /* w[n,k] = q[n,k] * s[n, k/128]; every product is exact in
                 * FP64 (11 + 4 + 11 significant bits). */
                double w = (double)qn[k] * w4o_double_from_half(sn[k / 128]);
                sum += jb->x_value(xm[k]) * w;
            }
            jb->y[m * jb->N + n] = jb->y_bits(sum);
            if (jb->acc)
                jb->acc[m * jb->N + n] = sum;
        }
    }
    return NULL;
}

int w4o_linear(const uint16_t* x, const int8_t* q, const uint16_t* s,
               int64_t M, int64_t N, int64_t K,
               uint16_t* y, double* acc, int nthreads)
{
    return w4o_linear_act(x, 0, q, s, M, N, K, y, acc, nthreads);
}

int w4o_linear_act(const uint16_t* x, int act, const int8_t* q, const uint16_t* s,
                   int64_t M, int64_t N, int64_t K,
                   uint16_t* y, double* acc, int nthreads)
{
    if (act != 0 && act != 1)
        return -1;
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return -1;
    if (M == 0 || N == 0)
        return 0;
    if (!x || !q || !s || !y)
        return -1;
    for (int64_t i = 0; i < N * K; ++i)
        if (q[i] < -8 || q[i] > 7)
            return -2;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > N)
        nthreads = (int)N;
    w4o_job* jobs = (w4o_job*)calloc((size_t)nthreads, sizeof(w4o_job));
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        w4o_job j = {x, q, s, M, N, K, y, acc,
                     N * t / nthreads, N * (t + 1) / nthreads,
                     act ? w4o_double_from_bf16 : w4o_double_from_half,
                     act ? w4o_bf16_from_double : w4o_half_from_double};
        jobs[t] = j;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, w4o_rows, &jobs[t]) != 0)
            break;
        started = t;
    }
    w4o_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
    /* rows of any thread that could not be started are done here */
    for (int t = started + 1; t < nthreads; ++t)
        w4o_rows(&jobs[t]);
    free(jobs);
    free(tid);
    return 0;
}

/* ---- the packed layout, written out from its definition -------------- */
int w4o_pack_layout(const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                    uint8_t* dst)
{
    if (N < 1 || K < 128 || K % 128 != 0 || !q || !s || !dst)
        return -1;
    for (int64_t i = 0; i < N * K; ++i)
        if (q[i] < -8 || q[i] > 7)
            return -2;
    const int64_t G = K / 128, bands = (N + 15) / 16;
    for (int64_t b = 0; b < bands; ++b) {
        for (int64_t g = 0; g < G; ++g) {
            uint8_t* tile = dst + (b * G + g) * 1056;
            memset(tile, 0, 1056);
            for (int L = 0; L < 32; ++L) {
                int r = L / 4, c = L % 4;
                for (int j = 0; j < 8; ++j) {
                    /* (row offset within band, k offset within group) of
                     * nibbles 0..7 of the word, as the definition lists */
                    const int row[8] = {r, r + 8, r, r + 8, r, r + 8, r, r + 8};
                    const int kk[8] = {16 * j + 4 * c,     16 * j + 4 * c,
                                       16 * j + 4 * c + 2, 16 * j + 4 * c + 2,
                                       16 * j + 4 * c + 1, 16 * j + 4 * c + 1,
                                       16 * j + 4 * c + 3, 16 * j + 4 * c + 3};
                    uint32_t word = 0;
                    for (int i = 0; i < 8; ++i) {
                        int64_t n = b * 16 + row[i];
                        int64_t k = g * 128 + kk[i];
                        uint32_t u = 8; /* padding row: q = 0 */
                        if (n < N)
                            u = (uint32_t)(q[n * K + k] + 8);
                        word |= u << (4 * i);
                    }
                    int off = (j < 4 ? 0 : 512) + 16 * L + 4 * (j % 4);
                    tile[off + 0] = (uint8_t)(word & 0xFF);
                    tile[off + 1] = (uint8_t)((word >> 8) & 0xFF);
                    tile[off + 2] = (uint8_t)((word >> 16) & 0xFF);
                    tile[off + 3] = (uint8_t)((word >> 24) & 0xFF);
                }
            }
            for (int p = 0; p < 8; ++p) {
                int64_t n0 = b * 16 + p, n1 = b * 16 + p + 8;
                uint16_t s0 = n0 < N ? s[n0 * G + g] : 0;
                uint16_t s1 = n1 < N ? s[n1 * G + g] : 0;
                tile[1024 + 4 * p + 0] = (uint8_t)(s0 & 0xFF);
                tile[1024 + 4 * p + 1] = (uint8_t)(s0 >> 8);
                tile[1024 + 4 * p + 2] = (uint8_t)(s1 & 0xFF);
                tile[1024 + 4 * p + 3] = (uint8_t)(s1 >> 8);
            }
        }
    }
    return 0;
}
