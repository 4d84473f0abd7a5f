/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY: the float64 CPU oracle for the
 * group-affine quantized projection.  See oracle.h for the contract, the
 * sources and the rule that no product code uses this file.
 *
 * What it computes, step by step, in the order the method states it:
 *   1. bf16 rounding (round to nearest, ties to even; signed zero kept on
 *      underflow; overflow to infinity) -- "cuda gemma4: images on the 12B"
 *      page, the commit on bf16(-2^-135).
 *   2. dequantization W = bf16(s*q + b), ONE rounding of the exact value --
 *      "Gemma 4 12B on the native Metal engine" page, the commit where each
 *      thread writes bf16(fma(scale, code, bias)) as mlx-lm dequantizes.
 *   3. the projection y[m,n] = sum_k W[n,k] * x[m,k] over the whole depth in
 *      double (the pages' tensor unit accumulates over the whole depth; the
 *      oracle's float64 sum stands for the exact sum).
 *   4. scaled embedding rows bf16(W[n,k] * scale) -- "cuda gemma4: images on
 *      the 12B" page, the embed_rows commit (the weight rounded first, then
 *      its product with the bf16 scale rounded again).
 *   5. the exact-codes form with producer-written group sums, and mlx_lm's
 *      GeGLU as bf16 operations (the fused gate/up epilogue) -- see oracle.h.
 *
 * The arithmetic is deliberately plain: no blocking, no vectorization, no
 * reordering of the sum.  Threads only split independent output rows.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* bf16 has 8 significant bits; its smallest subnormal is 2^-133 and its
 * largest finite value is (2 - 2^-7) * 2^127. */
#define BF16_MIN_ULP_EXP (-133)
#define BF16_SIG_BITS 8

static uint16_t bits_of_exact_bf16(double r, uint16_t sign) {
    /* r >= 0 is exactly representable in bf16 (or is +inf); a float holds it
     * exactly, and a bf16 pattern is the top half of that float's bits. */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return signbit(v) ? 0xFFC0u : 0x7FC0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    /* a = f * 2^e with f in [0.5, 1): the bf16 grid spacing around a is
     * 2^(e - 8), never finer than the subnormal spacing 2^-133. */
    int e = 0;
    (void)frexp(a, &e);
    int ulp_exp = e - BF16_SIG_BITS;
    if (ulp_exp < BF16_MIN_ULP_EXP) ulp_exp = BF16_MIN_ULP_EXP;
    double scaled = ldexp(a, -ulp_exp);       /* exact: a power-of-two scale */
    double rounded = nearbyint(scaled);       /* default mode: ties to even */
    double r = ldexp(rounded, ulp_exp);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max) return (uint16_t)(sign | 0x7F80u);
    return bits_of_exact_bf16(r, sign);
}

double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_bf16_from_f32_bits(const uint32_t* in, uint16_t* out, size_t n) {
    for (size_t i = 0; i < n; ++i) {
        float f;
        memcpy(&f, &in[i], sizeof f);
        out[i] = oracle_bf16_from_double((double)f);
    }
}

/* Round the exact real hi + lo (|lo| <= half an ulp of hi in double, as
 * TwoSum gives it) to bf16 once.  Rounding hi alone is correct unless hi sits
 * exactly on a midpoint between two bf16 values; there the sign of lo says on
 * which side the exact value lies, and lo == 0 means a true tie (to even). */
static uint16_t bf16_round_pair(double hi, double lo) {
    uint16_t r = oracle_bf16_from_double(hi);
    if (lo == 0.0 || isnan(hi) || isinf(hi)) return r;
    double a = fabs(hi);
    int e = 0;
    (void)frexp(a, &e);
    int ulp_exp = e - BF16_SIG_BITS;
    if (ulp_exp < BF16_MIN_ULP_EXP) ulp_exp = BF16_MIN_ULP_EXP;
    double scaled = ldexp(a, -ulp_exp);
    if (scaled - floor(scaled) != 0.5) return r; /* not a midpoint */
    double half = ldexp(0.5, ulp_exp);
    /* Pick the bf16 neighbour on lo's side of hi; both neighbours are exact
     * bf16 values, so this call does not round again. */
    return oracle_bf16_from_double(lo > 0.0 ? hi + half : hi - half);
}

uint16_t oracle_dequant_one(uint32_t q, uint16_t s, uint16_t b) {
    double sd = oracle_bf16_to_double(s);
    double bd = oracle_bf16_to_double(b);
    /* s has 8 significant bits and q at most 8, so s*q is exact in double. */
    double p = sd * (double)q;
    /* TwoSum (Knuth): hi + lo == p + b exactly. */
    double hi = p + bd;
    double bv = hi - p;
    double av = hi - bv;
    double lo = (p - av) + (bd - bv);
    if (isnan(hi) || isinf(hi)) return oracle_bf16_from_double(hi);
    return bf16_round_pair(hi, lo);
}

static int check_args(int bits, int group, int64_t N, int64_t K) {
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8)) return -1;
    if (!(group == 32 || group == 64 || group == 128)) return -2;
    if (N < 0 || K < 0 || (K % group) != 0) return -3;
    return 0;
}

int oracle_dequant(int bits, int group, int64_t N, int64_t K,
                   const uint8_t* codes, const uint16_t* scales,
                   const uint16_t* biases, uint16_t* w_out) {
    int rc = check_args(bits, group, N, K);
    if (rc) return rc;
    const int64_t G = K / group;
    const uint32_t qmax = (1u << bits) - 1u;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            uint32_t q = codes[n * K + k];
            if (q > qmax) return -4;
            int64_t j = k / group;
            w_out[n * K + k] = oracle_dequant_one(q, scales[n * G + j], biases[n * G + j]);
        }
    }
    return 0;
}

typedef struct {
    int bits, group;
    int64_t M, N, K, n0, n1;
    const uint16_t* x;
    const uint8_t* codes;
    const uint16_t* scales;
    const uint16_t* biases;
    double* y;
    int rc;
} qmm_job;

static void* qmm_rows(void* arg) {
    qmm_job* jb = (qmm_job*)arg;
    const int64_t K = jb->K, G = K / jb->group;
    const uint32_t qmax = (1u << jb->bits) - 1u;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!wrow) { jb->rc = -5; return NULL; }
    for (int64_t n = jb->n0; n < jb->n1; ++n) {
        /* Step 2: this row's weights, each rounded once to bf16. */
        for (int64_t k = 0; k < K; ++k) {
            uint32_t q = jb->codes[n * K + k];
            if (q > qmax) { jb->rc = -4; free(wrow); return NULL; }
            int64_t j = k / jb->group;
            wrow[k] = oracle_bf16_to_double(
                oracle_dequant_one(q, jb->scales[n * G + j], jb->biases[n * G + j]));
        }
        /* Step 3: each output is the depth-ordered sum of exact products. */
        for (int64_t m = 0; m < jb->M; ++m) {
            const uint16_t* xr = jb->x + m * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += wrow[k] * oracle_bf16_to_double(xr[k]);
            jb->y[m * jb->N + n] = acc;
        }
    }
    free(wrow);
    jb->rc = 0;
    return NULL;
}

int oracle_qmm(int bits, int group, int64_t M, int64_t N, int64_t K,
               const uint16_t* x, const uint8_t* codes,
               const uint16_t* scales, const uint16_t* biases,
               double* y_out, int nthreads) {
    int rc = check_args(bits, group, N, K);
    if (rc) return rc;
    if (M < 0) return -3;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    qmm_job* jobs = (qmm_job*)calloc((size_t)nthreads, sizeof(qmm_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -5; }
    for (int t = 0; t < nthreads; ++t) {
        qmm_job* jb = &jobs[t];
        jb->bits = bits; jb->group = group;
        jb->M = M; jb->N = N; jb->K = K;
        jb->n0 = N * t / nthreads;
        jb->n1 = N * (t + 1) / nthreads;
        jb->x = x; jb->codes = codes; jb->scales = scales; jb->biases = biases;
        jb->y = y_out;
    }
    if (nthreads == 1) {
        qmm_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&tids[t], NULL, qmm_rows, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(tids[t], NULL);
    }
    rc = 0;
    for (int t = 0; t < nthreads; ++t) if (jobs[t].rc) rc = jobs[t].rc;
    free(jobs);
    free(tids);
    return rc;
}

int oracle_qmm_groupsum(int bits, int group, int64_t M, int64_t N, int64_t K,
                        const uint16_t* x, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases,
                        double* y_gs, double* mag) {
    int rc = check_args(bits, group, N, K);
    if (rc) return rc;
    const int64_t G = K / group;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* xr = x + m * K;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, amag = 0.0;
            for (int64_t j = 0; j < G; ++j) {
                double s = oracle_bf16_to_double(scales[n * G + j]);
                double b = oracle_bf16_to_double(biases[n * G + j]);
                double sqx = 0.0, sx = 0.0;
                for (int64_t k = j * group; k < (j + 1) * group; ++k) {
                    double xv = oracle_bf16_to_double(xr[k]);
                    double q = (double)codes[n * K + k];
                    sqx += q * xv;
                    sx += xv;
                    amag += fabs(s * q + b) * fabs(xv);
                }
                acc += s * sqx + b * sx;
            }
            if (y_gs) y_gs[m * N + n] = acc;
            if (mag) mag[m * N + n] = amag;
        }
    }
    return 0;
}

int oracle_embed_rows(int bits, int group, int64_t N, int64_t K,
                      const uint8_t* codes, const uint16_t* scales,
                      const uint16_t* biases, const int32_t* ids, int64_t T,
                      int has_scale, uint16_t scale, uint16_t* out) {
    int rc = check_args(bits, group, N, K);
    if (rc) return rc;
    if (T < 0) return -3;
    const int64_t G = K / group;
    const uint32_t qmax = (1u << bits) - 1u;
    const double sc = oracle_bf16_to_double(scale);
    for (int64_t t = 0; t < T; ++t) {
        const int64_t n = ids[t];
        if (n < 0 || n >= N) return -6;
        for (int64_t k = 0; k < K; ++k) {
            uint32_t q = codes[n * K + k];
            if (q > qmax) return -4;
            int64_t j = k / group;
            uint16_t w = oracle_dequant_one(q, scales[n * G + j], biases[n * G + j]);
            /* Two bf16 values have 8 significant bits each, so their product is
             * exact in double and this is its single rounding. */
            out[t * K + k] = has_scale ? oracle_bf16_from_double(oracle_bf16_to_double(w) * sc) : w;
        }
    }
    return 0;
}

int oracle_qmm_groupsum_given(int bits, int group, int64_t M, int64_t N, int64_t K,
                              const uint16_t* x, const float* xsums, const uint8_t* codes,
                              const uint16_t* scales, const uint16_t* biases, double* y) {
    int rc = check_args(bits, group, N, K);
    if (rc) return rc;
    if (M < 0) return -3;
    const int64_t G = K / group;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* xr = x + m * K;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < G; ++j) {
                double s = oracle_bf16_to_double(scales[n * G + j]);
                double b = oracle_bf16_to_double(biases[n * G + j]);
                double sqx = 0.0;
                for (int64_t k = j * group; k < (j + 1) * group; ++k)
                    sqx += (double)codes[n * K + k] * oracle_bf16_to_double(xr[k]);
                acc += s * sqx + b * (double)xsums[m * G + j];
            }
            y[m * N + n] = acc;
        }
    }
    return 0;
}

/* bf16 of an exact real given as a double: the products of two bf16 values,
 * the cube of one and the sum of two are exact in double (at most 24
 * significant bits, or an exponent gap beyond which the smaller addend cannot
 * move the bf16 rounding of the larger), so one rounding here is the single
 * rounding of the exact result. */
static uint16_t bf_round(double v) { return oracle_bf16_from_double(v); }
static double bf(uint16_t h) { return oracle_bf16_to_double(h); }

/* The steps after tanh (t the bf16 tanh's value): e = bf16(1 + t),
 * p = bf16(0.5 g), r = bf16(p e), h = bf16(r up). */
static uint16_t geglu_tail(uint16_t g, double t, uint16_t up) {
    uint16_t e = bf_round(1.0 + t);
    uint16_t p = bf_round(0.5 * bf(g));
    uint16_t r = bf_round(bf(p) * bf(e));
    return bf_round(bf(r) * bf(up));
}

void oracle_geglu(int64_t n, const uint16_t* gate, const uint16_t* up, int tanh_ulps,
                  uint16_t* h_lo, uint16_t* h_hi) {
    const uint16_t c1 = bf_round(0.044715);
    const uint16_t c2 = bf_round(sqrt(2.0 / 3.14159265358979323846));
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t g = gate[i];
        const double gv = bf(g);
        uint16_t c3 = bf_round(gv * gv * gv);
        uint16_t a = bf_round(bf(c1) * bf(c3));
        uint16_t z = bf_round(gv + bf(a));
        uint16_t u = bf_round(bf(c2) * bf(z));
        const double tv = tanh(bf(u));
        /* the fp32 tanh of a GPU is tv within tanh_ulps fp32 ulps; its bf16
         * rounding is one of the roundings of the interval's ends */
        double d = 0.0;
        if (isfinite(tv) && tv != 0.0) {
            int e = 0;
            (void)frexp(tv, &e);
            d = ldexp((double)tanh_ulps, e - 24);
        }
        uint16_t t_lo = bf_round(tv - d), t_hi = bf_round(tv + d);
        if (isnan(tv)) t_lo = t_hi = bf_round(tv);
        h_lo[i] = geglu_tail(g, bf(t_lo), up[i]);
        h_hi[i] = geglu_tail(g, bf(t_hi), up[i]);
    }
}
