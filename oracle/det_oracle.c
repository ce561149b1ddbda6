/*
 * det_oracle.c -- the CPU oracle for the frozen FP32 numerical profile, v1.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the library. It is deliberately plain:
 * explicit loops in the order the profile defines, one rounding per written
 * operation, fmaf where the profile says fused multiply-add. There is no
 * blocking, fusion or reordering beyond the definitions.
 *
 * Build: cc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        (no -march flags: the same source must give the same bits on x86-64
 *        and on aarch64, as the "mojolearn" PyPI page, section "The evidence
 *        behind the claim", reports for CPUs of both kinds).
 *
 * Sources. "mojolearn" (PyPI project page), section "What bitwise identity
 * means, and why it is not the default": vendors differ in summation order, FMA
 * contraction, denormal handling, tie-breaking and the spelling of exp and log;
 * the frozen profile fixes each. Section "The exact scope of the claim" lists
 * the profile's knobs (reduction order, partitioning, FMA policy, flush-to-zero
 * seams, transcendental spellings, tie rules). "MojoLearn 162M: one model, two
 * hardware routes", tables "Compared with GPT-3 Small" and "Training", give
 * the operations' hyperparameters (RMSNorm eps 1e-6; AdamW beta (0.9, 0.95),
 * eps 1e-8, weight decay 0.1). The pages give no numeric spellings; the v1
 * readings implemented below are the plainest ones and are listed in the
 * repository's design notes.
 *
 * Separating arms. Blocks under #ifdef SABOTAGE_* plant one plausible mistake
 * each (a wrong chunk width, a reversed order, roundf for rintf, a contracted
 * multiply-add, ...). The shipped oracle defines none of them; the test suite
 * builds each arm into a scratch library and checks that a named pin fails,
 * so every such pin is shown to separate the rule it guards.
 *
 * Parity status of each function against something other than itself is kept
 * in the tests (closed forms, exact-rational brute force, double-precision
 * bounds). The bit patterns chosen by readings R14-R18 (exp/log polynomials,
 * AdamW operation order) are fixed by those readings, not by the pages:
 * parity unpinned by the pages for those exact bits; pinned by accuracy bounds
 * and closed forms.
 */
#define _GNU_SOURCE
#include "det_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif
#if defined(__FAST_MATH__)
#error "the oracle must not be built with fast-math"
#endif

/* ------------------------------------------------------------------------ */
/* bit helpers                                                               */
/* ------------------------------------------------------------------------ */
static inline uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
/* 2^e as a float, for -126 <= e <= 127 (a normal power of two). */
static inline float pow2f(int e) { return u2f((uint32_t)(e + 127) << 23); }

int detor_fp_env_ok(void) {
    /* Behavioural check (no inline assembly): with flush-to-zero or
     * denormals-are-zero set, these products of a subnormal are 0. */
    volatile float tiny = 0x1p-140f;        /* subnormal */
    volatile float one = 1.0f;
    volatile float half_min = FLT_MIN;
    float a = tiny * one;                   /* DAZ would read tiny as 0 */
    float b = half_min * 0.5f;              /* FTZ would flush the result */
    return (a != 0.0f) && (b != 0.0f) && (FLT_EVAL_METHOD == 0);
}

/* ------------------------------------------------------------------------ */
/* exp: Cody-Waite argument reduction and a Taylor polynomial               */
/* ------------------------------------------------------------------------ */
/* Constants, each the float nearest to its definition:
 *   LOG2E  = 1/ln 2;  LN2_HI = ln 2;  LN2_LO = ln 2 - LN2_HI (exact difference,
 *   rounded);  E_k = 1/k!  (k = 0..7). */
static const float LOG2E  = 0x1.715476p+0f;
#ifndef SABOTAGE_EXP_LN2_SPLIT
static const float LN2_HI = 0x1.62e430p-1f;
static const float LN2_LO = -0x1.05c610p-29f;
#else   /* separating arm: Cody and Waite's split with trailing zero bits */
static const float LN2_HI = 0x1.62e400p-1f;
static const float LN2_LO = 0x1.7f7d1cp-20f;
#endif
static const float E0 = 0x1p+0f, E1 = 0x1p+0f, E2 = 0x1p-1f;
static const float E3 = 0x1.555556p-3f, E4 = 0x1.555556p-5f;
static const float E5 = 0x1.111112p-7f, E6 = 0x1.6c16c2p-10f;
static const float E7 = 0x1.a01a02p-13f;
/* Largest float whose exp is finite in float: the float just below ln(FLT_MAX)
 * rounded up (0x42b17217). Below EXP_LO the result is below half the smallest
 * subnormal for every reduction, so it is +0. */
static const float EXP_HI = 0x1.62e42ep+6f;
static const float EXP_LO = -104.0f;

float detor_exp(float x) {
    if (x != x) return x + x;                 /* NaN in, NaN out */
    if (x > EXP_HI) return INFINITY;
    if (x < EXP_LO) return 0.0f;
    /* x = n ln2 + r with n = round-half-even(x / ln2): the tie rule of the
     * reduction is that of rintf in round-to-nearest mode. */
    float t = x * LOG2E;
#ifndef SABOTAGE_ROUNDF
    float n = rintf(t);
#else   /* separating arm: ties away from zero */
    float n = roundf(t);
#endif
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    /* e^r by Horner on the degree-7 Taylor polynomial, highest term first. */
    float p = E7;
#ifndef SABOTAGE_EXP_HORNER_UNFUSED
    p = fmaf(p, r, E6);
    p = fmaf(p, r, E5);
    p = fmaf(p, r, E4);
    p = fmaf(p, r, E3);
    p = fmaf(p, r, E2);
    p = fmaf(p, r, E1);
    p = fmaf(p, r, E0);
#else   /* separating arm: each Horner step a rounded product, then the add */
    p = p * r + E6;
    p = p * r + E5;
    p = p * r + E4;
    p = p * r + E3;
    p = p * r + E2;
    p = p * r + E1;
    p = p * r + E0;
#endif
    /* scale by 2^n with exactly one rounding */
    int ni = (int)n;                           /* |n| <= 150, exact */
    if (ni > 127) return (p + p) * pow2f(127);             /* ni == 128 */
    if (ni < -126) return (p * pow2f(ni + 64)) * pow2f(-64);
    return p * pow2f(ni);
}

/* ------------------------------------------------------------------------ */
/* log: exponent split, atanh series in s = (f-1)/(f+1)                      */
/* ------------------------------------------------------------------------ */
/* With x = 2^e f, f in (sqrt(1/2), sqrt 2), u = f - 1 and s = u / (2 + u):
 *   log f = 2 atanh s = 2s + s R,  R = 2(z/3 + z^2/5 + ... + z^5/11),  z = s^2,
 * and since 2s = u - s u = u - h + s h with h = u^2/2,
 *   log f = u - (h - s (h + R)).
 * The leading term u is exact, so the rounding errors sit in the small
 * correction (the arrangement used by the freely distributable fdlibm log;
 * here with the Taylor coefficients 2/k of atanh instead of fitted ones).
 * T_k = 2/k (k = 3, 5, 7, 9, 11). SQRT2_BITS: bits of the largest float below
 * sqrt 2. */
static const float T3 = 0x1.555556p-1f, T5 = 0x1.99999ap-2f, T7 = 0x1.24924ap-2f;
static const float T9 = 0x1.c71c72p-3f, T11 = 0x1.745d18p-3f;
static const uint32_t SQRT2_BITS = 0x3fb504f3u;

float detor_log(float x) {
    if (x != x) return x + x;
    if (x < 0.0f) return NAN;
    if (x == 0.0f) return -INFINITY;
    if (x == INFINITY) return x;
    int e = 0;
    if (x < FLT_MIN) { x = x * 0x1p23f; e = -23; }   /* subnormal: exact scaling */
    uint32_t b = f2u(x);
    e += (int)(b >> 23) - 127;
    uint32_t fb = (b & 0x007fffffu) | 0x3f800000u;    /* f in [1, 2) */
    if (fb > SQRT2_BITS) { fb -= 0x00800000u; e += 1; } /* f in (sqrt(1/2), sqrt 2) */
    float f = u2f(fb);
    float u = f - 1.0f;                               /* exact (Sterbenz) */
    float s = u / (2.0f + u);
    float z = s * s;
    float R = T11;
    R = fmaf(R, z, T9);
    R = fmaf(R, z, T7);
    R = fmaf(R, z, T5);
    R = fmaf(R, z, T3);
    R = R * z;
    float h = (0.5f * u) * u;
#ifndef SABOTAGE_CONTRACT_LOG
    float lf = u - (h - s * (h + R));
#else   /* separating arm: h - s (h + R) contracted into one fmaf */
    float lf = u - fmaf(-s, h + R, h);
#endif
    float ef = (float)e;
    return fmaf(ef, LN2_HI, fmaf(ef, LN2_LO, lf));
}

/* ------------------------------------------------------------------------ */
/* a tiny parallel-for over [0, n): contiguous ranges, one per thread.       */
/* Every output is produced by exactly one thread with the same operations, */
/* so results never depend on the thread count.                             */
/* ------------------------------------------------------------------------ */
#define MAX_THREADS 256
typedef void (*range_fn)(int64_t lo, int64_t hi, int t, void *ctx);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; int t; } range_job;

static void *range_trampoline(void *arg) {
    range_job *j = (range_job *)arg;
    j->fn(j->lo, j->hi, j->t, j->ctx);
    return NULL;
}

/* Runs fn over contiguous ranges; thread t gets the t-th range and may write
 * slot t of a per-thread array in ctx. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    if (nthreads == 1) { fn(0, n, 0, ctx); return; }
    pthread_t tid[MAX_THREADS];
    range_job jobs[MAX_THREADS];
    int started[MAX_THREADS];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].t = t;
        jobs[t].lo = n * t / nthreads; jobs[t].hi = n * (t + 1) / nthreads;
        started[t] = pthread_create(&tid[t], NULL, range_trampoline, &jobs[t]) == 0;
        if (!started[t]) range_trampoline(&jobs[t]);   /* run inline instead */
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* elementwise exp / log                                                     */
/* ------------------------------------------------------------------------ */
typedef struct { const float *x; float *y; } map_ctx;
static void exp_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    map_ctx *m = (map_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) m->y[i] = detor_exp(m->x[i]);
}
static void log_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    map_ctx *m = (map_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) m->y[i] = detor_log(m->x[i]);
}
void detor_exp_n(int64_t n, const float *x, float *y, int nthreads) {
    map_ctx c = {x, y};
    parallel_for(n, nthreads, exp_range, &c);
}
void detor_log_n(int64_t n, const float *x, float *y, int nthreads) {
    map_ctx c = {x, y};
    parallel_for(n, nthreads, log_range, &c);
}

static void sin_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    map_ctx *m = (map_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) m->y[i] = detor_sin(m->x[i]);
}
static void cos_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    map_ctx *m = (map_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) m->y[i] = detor_cos(m->x[i]);
}
void detor_sin_n(int64_t n, const float *x, float *y, int nthreads) {
    map_ctx c = {x, y};
    parallel_for(n, nthreads, sin_range, &c);
}
void detor_cos_n(int64_t n, const float *x, float *y, int nthreads) {
    map_ctx c = {x, y};
    parallel_for(n, nthreads, cos_range, &c);
}

/* ------------------------------------------------------------------------ */
/* fixed-order GEMM                                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    int transA, transB;
    int64_t M, N, K, lda, ldb, ldc, kc;
    const float *A, *B;
    float *C;
} gemm_ctx;

static void gemm_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    gemm_ctx *g = (gemm_ctx *)c;
#ifdef SABOTAGE_CHUNK_REVERSED
    float part[4096];
#endif
    for (int64_t i = lo; i < hi; ++i) {
        for (int64_t j = 0; j < g->N; ++j) {
            float total = 0.0f;                   /* K == 0: the empty sum, +0 */
            for (int64_t c0 = 0; c0 < g->K; c0 += g->kc) {
                int64_t c1 = c0 + g->kc < g->K ? c0 + g->kc : g->K;
                float acc = 0.0f;                 /* every chunk starts from +0 */
                for (int64_t k = c0; k < c1; ++k) {
                    float a = g->transA ? g->A[k * g->lda + i] : g->A[i * g->lda + k];
                    float b = g->transB ? g->B[j * g->ldb + k] : g->B[k * g->ldb + j];
#ifndef SABOTAGE_FIRST_PRODUCT_SEED
                    acc = fmaf(a, b, acc);        /* ascending k, one rounding each */
#else   /* separating arm: the chain seeded with the first product */
                    acc = (k == c0) ? a * b : fmaf(a, b, acc);
#endif
                }
#ifndef SABOTAGE_CHUNK_REVERSED
                if (c0 == 0) total = acc;         /* first partial taken as is */
                else total = total + acc;         /* then left to right */
#else   /* separating arm: partials kept, then added right to left */
                part[c0 / g->kc] = acc;
#endif
            }
#ifdef SABOTAGE_CHUNK_REVERSED
            {
                int64_t nc = (g->K + g->kc - 1) / g->kc;
                if (nc > 0) total = part[nc - 1];
                for (int64_t c = nc - 2; c >= 0; --c) total = total + part[c];
            }
#endif
            g->C[i * g->ldc + j] = total;
        }
    }
}

void detor_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
                const float *A, int64_t lda, const float *B, int64_t ldb,
                float *C, int64_t ldc, int64_t k_chunk, int nthreads) {
    gemm_ctx g = {transA, transB, M, N, K, lda, ldb, ldc, k_chunk, A, B, C};
    if (k_chunk <= 0) return;
#ifdef SABOTAGE_CHUNK128
    g.kc = 128;   /* separating arm: chunks half as wide */
#endif
    parallel_for(M, nthreads, gemm_rows, &g);
}

/* Gradient accumulation (beta = 1): the new product is formed exactly as
 * detor_gemm forms it, then added to the old C once, C on the left, so that
 * accumulating shard after shard gives the same bits as the left-to-right
 * shard sum below. */
void detor_gemm_acc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda, const float *B, int64_t ldb,
                    float *C, int64_t ldc, int64_t k_chunk, int nthreads) {
    if (k_chunk <= 0 || M <= 0 || N <= 0) return;
    float *R = (float *)malloc(sizeof(float) * (size_t)M * (size_t)N);
    if (!R) return;
    detor_gemm(transA, transB, M, N, K, A, lda, B, ldb, R, N, k_chunk, nthreads);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) C[i * ldc + j] = C[i * ldc + j] + R[i * N + j];
    free(R);
}

/* ------------------------------------------------------------------------ */
/* sin and cos (v1 spelling)                                                 */
/* ------------------------------------------------------------------------ */
/* The pages fix that the transcendental spellings are part of the profile and
 * print none; the model card's rotary positions ("MojoLearn 162M", table
 * "Compared with GPT-3 Small": rotary, theta = 10,000) need sin and cos.
 * Reading R31 of the design notes, Cody & Waite's reduction with Taylor
 * polynomials:
 *   k = rint(x * 2/pi) (ties to even); r = x - k pi/2 by three fmaf steps with
 *   pi/2 split in three floats; z = r * r;
 *   sin_r = fmaf(r, z * Ps(z), r), Ps = Horner of the Taylor terms 1/3! .. 1/9!
 *   cos_r = fmaf(Pc(z), z, 1),  Pc = Horner of the terms 1/2! .. 1/10!
 *   then the quadrant k mod 4 picks +-sin_r or +-cos_r.
 * Zero returns x for sin and 1 for cos; |x| > 2^20 and NaN give NaN. Every
 * constant is the float nearest to its definition. */
static const float TWO_OVER_PI = 0x1.45f306p-1f;
static const float PIO2_1 = 0x1.921fb6p+0f, PIO2_2 = -0x1.777a5cp-25f;
static const float PIO2_3 = -0x1.ee59dap-50f;
static const float S3F = -0x1.555556p-3f, S5F = 0x1.111112p-7f;
static const float S7F = -0x1.a01a02p-13f, S9F = 0x1.71de3ap-19f;
static const float C2F = -0x1p-1f, C4F = 0x1.555556p-5f, C6F = -0x1.6c16c2p-10f;
static const float C8F = 0x1.a01a02p-16f, C10F = -0x1.27e4fcp-22f;
static const float TRIG_MAX = 0x1p20f;

static void sincos_v1(float x, float *sn, float *cs) {
    if (x != x || fabsf(x) > TRIG_MAX) { *sn = NAN; *cs = NAN; return; }
    if (x == 0.0f) { *sn = x; *cs = 1.0f; return; }
    float k = rintf(x * TWO_OVER_PI);
    float r = fmaf(-k, PIO2_1, x);
    r = fmaf(-k, PIO2_2, r);
    r = fmaf(-k, PIO2_3, r);
    float z = r * r;
    float ps = S9F;
    ps = fmaf(ps, z, S7F);
    ps = fmaf(ps, z, S5F);
    ps = fmaf(ps, z, S3F);
    float s = fmaf(r, z * ps, r);
    float pc = C10F;
    pc = fmaf(pc, z, C8F);
    pc = fmaf(pc, z, C6F);
    pc = fmaf(pc, z, C4F);
    pc = fmaf(pc, z, C2F);
    float c = fmaf(pc, z, 1.0f);
    int q = (int)k & 3;
    *sn = q == 0 ? s : q == 1 ? c : q == 2 ? -s : -c;
    *cs = q == 0 ? c : q == 1 ? -s : q == 2 ? -c : s;
}

float detor_sin(float x) { float s, c; sincos_v1(x, &s, &c); return s; }
float detor_cos(float x) { float s, c; sincos_v1(x, &s, &c); return c; }

/* ------------------------------------------------------------------------ */
/* rotary position embedding                                                 */
/* ------------------------------------------------------------------------ */
/* Reading R30: pairs (x_2i, x_2i+1) of each head (the rotary paper's
 * pairing) turn by a = pos * w_i, w_i = exp((-(2i / d)) * log(theta)) with the
 * profile's exp and log, each step rounded once; then
 *   y_2i = x_2i * c - x_2i+1 * s,  y_2i+1 = x_2i * s + x_2i+1 * c
 * (each product rounded, then the subtraction or addition). */
typedef struct {
    int64_t heads, d, ldx, seq;
    float *x;
    float theta;
    int backward;
} rope_ctx;

static void rope_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    rope_ctx *q = (rope_ctx *)c;
    const float L = detor_log(q->theta);
    for (int64_t t = lo; t < hi; ++t) {
        const float pos = (float)(t % q->seq);
        for (int64_t i = 0; i < q->d / 2; ++i) {
            const float e = (float)(2 * i) / (float)q->d;
            const float w = detor_exp(-e * L);
            const float a = pos * w;
            float sn, cs;
            sincos_v1(a, &sn, &cs);
            for (int64_t h = 0; h < q->heads; ++h) {
                float *p = q->x + t * q->ldx + h * q->d + 2 * i;
                const float x0 = p[0], x1 = p[1];
                if (!q->backward) {
                    p[0] = x0 * cs - x1 * sn;
                    p[1] = x0 * sn + x1 * cs;
                } else {          /* the transpose: turn by -a (R35) */
                    p[0] = x0 * cs + x1 * sn;
                    p[1] = x1 * cs - x0 * sn;
                }
            }
        }
    }
}

void detor_rope(int64_t rows, int64_t heads, int64_t head_dim, float *x, int64_t ldx,
                int64_t seq_len, float theta, int nthreads) {
    if (head_dim < 2 || head_dim % 2 || seq_len < 1 || heads < 1) return;
    rope_ctx c = {heads, head_dim, ldx, seq_len, x, theta, 0};
    parallel_for(rows, nthreads, rope_rows, &c);
}

/* Rotary backward (design notes R35): the forward's angles; the gradient pair
 * turns by -a: dx0 = dy0 * c + dy1 * s, dx1 = dy1 * c - dy0 * s. */
void detor_rope_bwd(int64_t rows, int64_t heads, int64_t head_dim, float *x, int64_t ldx,
                    int64_t seq_len, float theta, int nthreads) {
    if (head_dim < 2 || head_dim % 2 || seq_len < 1 || heads < 1) return;
    rope_ctx c = {heads, head_dim, ldx, seq_len, x, theta, 1};
    parallel_for(rows, nthreads, rope_rows, &c);
}

/* Embedding backward (design notes R36): per id v and column j, the tokens'
 * gradients in ascending token order, the first as is, then left to right. */
typedef struct {
    int64_t ntok, dim;
    const int32_t *tok;
    const float *dx;
    float *de;
} embb_ctx;

static void embb_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    embb_ctx *q = (embb_ctx *)c;
    for (int64_t v = lo; v < hi; ++v) {
        for (int64_t j = 0; j < q->dim; ++j) {
            float t = 0.0f;
            int first = 1;
            for (int64_t k = 0; k < q->ntok; ++k) {
                if (q->tok[k] != v) continue;
                t = first ? q->dx[k * q->dim + j] : t + q->dx[k * q->dim + j];
                first = 0;
            }
            q->de[v * q->dim + j] = t;
        }
    }
}

void detor_embedding_bwd(int64_t ntok, int64_t dim, const int32_t *tokens, const float *dx,
                         int64_t vocab, float *de, int nthreads) {
    embb_ctx c = {ntok, dim, tokens, dx, de};
    parallel_for(vocab, nthreads, embb_range, &c);
}

/* ------------------------------------------------------------------------ */
/* element-wise block operations                                             */
/* ------------------------------------------------------------------------ */
/* "MojoLearn 162M" model card, table "Compared with GPT-3 Small": SwiGLU
 * feed-forward (2,048 wide), pre-norm residual blocks. Readings (design notes
 * R27, R28): silu(g) = g / (1 + exp(-g)) with the profile's exp, IEEE
 * division, then the product with the up projection; the residual add is one
 * rounded addition. */
typedef struct {
    const float *a, *b;
    float *out;
} ew_ctx;

static void swiglu_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    ew_ctx *q = (ew_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) {
        float g = q->a[i];
        float den = 1.0f + detor_exp(-g);
        float silu = g / den;
        q->out[i] = silu * q->b[i];
    }
}

static void add_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    ew_ctx *q = (ew_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) q->out[i] = q->a[i] + q->b[i];
}

void detor_swiglu(int64_t n, const float *gate, const float *up, float *out, int nthreads) {
    ew_ctx c = {gate, up, out};
    parallel_for(n, nthreads, swiglu_range, &c);
}

/* SwiGLU backward (design notes R33): with e = exp(-g), den = 1 + e,
 * silu = g / den (the forward's value) and sig = 1 / den,
 *   d_up   = dh * silu
 *   d_gate = (dh * u) * (sig * (1 + g * (1 - sig)))
 * every operation rounded once, in that order. */
typedef struct {
    const float *g, *u, *dh;
    float *dg, *du;
} swb_ctx;

static void swiglu_bwd_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    swb_ctx *q = (swb_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) {
        float g = q->g[i];
        float den = 1.0f + detor_exp(-g);
        float silu = g / den;
        float sig = 1.0f / den;
        float ds = sig * (1.0f + g * (1.0f - sig));
        q->du[i] = q->dh[i] * silu;
        q->dg[i] = (q->dh[i] * q->u[i]) * ds;
    }
}

void detor_swiglu_bwd(int64_t n, const float *gate, const float *up, const float *dh,
                      float *d_gate, float *d_up, int nthreads) {
    swb_ctx c = {gate, up, dh, d_gate, d_up};
    parallel_for(n, nthreads, swiglu_bwd_range, &c);
}

void detor_add(int64_t n, const float *a, const float *b, float *out, int nthreads) {
    ew_ctx c = {a, b, out};
    parallel_for(n, nthreads, add_range, &c);
}

/* ------------------------------------------------------------------------ */
/* fixed-order shard gradient sum                                            */
/* ------------------------------------------------------------------------ */
/* "MojoLearn 162M" model card, table "Training": 64 logical shards, each a
 * mean over 4 x 2,048 tokens; the shard gradients are summed in a fixed order.
 * Reading: left to right over the shard index, one rounding per addition, then
 * one multiply by the caller's scale (1/64 for the mean of 64 shards, exact). */
typedef struct {
    int64_t S, ld;
    const float *g;
    float scale;
    float *out;
} shard_ctx;

static void shard_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    shard_ctx *q = (shard_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) {
#ifndef SABOTAGE_SHARD_REVERSED
        float t = q->g[i];                        /* shard 0 as is */
        for (int64_t s = 1; s < q->S; ++s) t = t + q->g[s * q->ld + i];
#else   /* separating arm: right to left */
        float t = q->g[(q->S - 1) * q->ld + i];
        for (int64_t s = q->S - 2; s >= 0; --s) t = t + q->g[s * q->ld + i];
#endif
        q->out[i] = t * q->scale;
    }
}

void detor_shardsum(int64_t nshards, int64_t n, const float *shards, int64_t ld,
                    float scale, float *out, int nthreads) {
    if (nshards < 1 || n < 1) return;
    shard_ctx c = {nshards, ld, shards, scale, out};
    parallel_for(n, nthreads, shard_range, &c);
}

/* ------------------------------------------------------------------------ */
/* the profile's fixed reduction tree over `lanes` chain sums               */
/* ------------------------------------------------------------------------ */
/* Level offsets: 16, 8, 4, 2, 1 (within a group of 32 lanes), then 32, 64, ...
 * up to lanes/2. At each level every lane l becomes s[l] + s[l ^ off]. The
 * addition is commutative, so all lanes end with the same value: lane 0's. */
static float butterfly(float *s, int lanes) {
    float t[1024];
#ifndef SABOTAGE_BUTTERFLY_ORDER
    static const int low[5] = {16, 8, 4, 2, 1};
#else   /* separating arm: the levels in the opposite order */
    static const int low[5] = {1, 2, 4, 8, 16};
#endif
    for (int li = 0; li < 5; ++li) {
        int off = low[li];
        if (off >= lanes) continue;
        for (int l = 0; l < lanes; ++l) t[l] = s[l] + s[l ^ off];
        for (int l = 0; l < lanes; ++l) s[l] = t[l];
    }
    for (int off = 32; off < lanes; off *= 2) {
        for (int l = 0; l < lanes; ++l) t[l] = s[l] + s[l ^ off];
        for (int l = 0; l < lanes; ++l) s[l] = t[l];
    }
    return s[0];
}

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                   */
/* ------------------------------------------------------------------------ */
typedef struct {
    int64_t D, ldx, ldy;
    const float *x, *gain;
    float eps;
    float *y, *inv;
    int lanes, group;
} rms_ctx;

static void rms_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    rms_ctx *q = (rms_ctx *)c;
    float s[1024];
    for (int64_t r = lo; r < hi; ++r) {
        const float *x = q->x + r * q->ldx;
        for (int l = 0; l < q->lanes; ++l) s[l] = 0.0f;
        for (int64_t j = 0; j < q->D; ++j) {
#ifndef SABOTAGE_ELEMENT_OWNERSHIP
            int l = (int)((j / q->group) % q->lanes);
#else   /* separating arm: chains own single elements, not groups of 4 */
            int l = (int)(j % q->lanes);
#endif
            s[l] = fmaf(x[j], x[j], s[l]);        /* each lane: ascending j */
        }
        float ss = butterfly(s, q->lanes);
#ifndef SABOTAGE_RECIP_D
        float ms = ss / (float)q->D;
#else   /* separating arm: a multiply by 1/D for the division */
        float ms = ss * (1.0f / (float)q->D);
#endif
        float rr = 1.0f / sqrtf(ms + q->eps);
        float *y = q->y + r * q->ldy;
        for (int64_t j = 0; j < q->D; ++j) y[j] = (x[j] * rr) * q->gain[j];
        if (q->inv) q->inv[r] = rr;
    }
}

void detor_rmsnorm(int64_t rows, int64_t D, const float *x, int64_t ldx,
                   const float *gain, float eps, float *y, int64_t ldy,
                   float *inv_rms, int lanes, int group, int nthreads) {
    if (lanes < 1 || lanes > 1024 || group < 1 || D < 1) return;
    rms_ctx c = {D, ldx, ldy, x, gain, eps, y, inv_rms, lanes, group};
    parallel_for(rows, nthreads, rms_rows, &c);
}

/* ------------------------------------------------------------------------ */
/* RMSNorm backward                                                          */
/* ------------------------------------------------------------------------ */
/* The gradient of y_j = (x_j r) g_j with r = 1/sqrt(mean(x^2) + eps), in the
 * textbook form dx = r (h - xhat mean(h xhat)), h = dy g, xhat = x r, and
 * dgain_j = sum over rows of dy_j xhat_j. Per row, with r the forward's
 * inv_rms (readings R20-R24 of the design notes):
 *   xhat_j = x_j * r;  h_j = dy_j * g_j                (one rounding each)
 *   dot    = the lane sums of fmaf(h_j, xhat_j, .)    (lane l owning groups g
 *            with g mod lanes == l, ascending j, from +0) folded by the
 *            butterfly -- the forward's sum-of-squares arrangement
 *   q      = dot / D
 *   dx_j   = (h_j - xhat_j * q) * r                   (three roundings)
 * dgain_j is a contraction over the rows, so it takes the GEMM's spelling: for
 * each k_chunk-wide chunk of rows an fmaf chain of dy_ij * xhat_ij from +0 in
 * ascending i, the chunk partials added left to right (the first as is). It
 * is therefore the diagonal of the profile's GEMM xhat^T dy. */
typedef struct {
    int64_t rows, D, ldx, lddy, lddx, kc;
    const float *x, *gain, *inv, *dy;
    float *dx, *dgain;
    int lanes, group;
} rmsb_ctx;

static void rmsb_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    rmsb_ctx *q = (rmsb_ctx *)c;
    float s[1024];
    for (int64_t r = lo; r < hi; ++r) {
        const float *x = q->x + r * q->ldx;
        const float *dy = q->dy + r * q->lddy;
        const float rr = q->inv[r];
        for (int l = 0; l < q->lanes; ++l) s[l] = 0.0f;
        for (int64_t j = 0; j < q->D; ++j) {
            int l = (int)((j / q->group) % q->lanes);
            float xhat = x[j] * rr;
            float h = dy[j] * q->gain[j];
            s[l] = fmaf(h, xhat, s[l]);           /* each lane: ascending j */
        }
        float dot = butterfly(s, q->lanes);
        float qm = dot / (float)q->D;
        float *dx = q->dx + r * q->lddx;
        for (int64_t j = 0; j < q->D; ++j) {
            float xhat = x[j] * rr;
            float h = dy[j] * q->gain[j];
#ifndef SABOTAGE_CONTRACT_RMSBWD
            float p = xhat * qm;
            float d = h - p;
#else   /* separating arm: h - xhat q contracted into one fmaf */
            float d = fmaf(-xhat, qm, h);
#endif
            dx[j] = d * rr;
        }
    }
}

static void rmsb_cols(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    rmsb_ctx *q = (rmsb_ctx *)c;
    for (int64_t j = lo; j < hi; ++j) {
        float total = 0.0f;                       /* no rows: the empty sum, +0 */
#ifndef SABOTAGE_ONE_CHAIN_DGAIN
        const int64_t kc = q->kc;
#else   /* separating arm: one chain over all rows */
        const int64_t kc = q->rows > 0 ? q->rows : 1;
#endif
        for (int64_t c0 = 0; c0 < q->rows; c0 += kc) {
            int64_t c1 = c0 + kc < q->rows ? c0 + kc : q->rows;
            float acc = 0.0f;                     /* every chunk starts from +0 */
            for (int64_t i = c0; i < c1; ++i) {
                float xhat = q->x[i * q->ldx + j] * q->inv[i];
                acc = fmaf(q->dy[i * q->lddy + j], xhat, acc);
            }
            if (c0 == 0) total = acc;             /* first partial taken as is */
            else total = total + acc;             /* then left to right */
        }
        q->dgain[j] = total;
    }
}

void detor_rmsnorm_bwd(int64_t rows, int64_t D, const float *x, int64_t ldx,
                       const float *gain, const float *inv_rms, const float *dy,
                       int64_t lddy, float *dx, int64_t lddx, float *dgain,
                       int lanes, int group, int64_t k_chunk, int nthreads) {
    if (lanes < 1 || lanes > 1024 || group < 1 || D < 1 || k_chunk < 1) return;
    rmsb_ctx c = {rows, D, ldx, lddy, lddx, k_chunk, x, gain, inv_rms, dy, dx, dgain,
                  lanes, group};
    parallel_for(rows, nthreads, rmsb_rows, &c);
    if (dgain) parallel_for(D, nthreads, rmsb_cols, &c);
}

/* ------------------------------------------------------------------------ */
/* softmax cross-entropy                                                     */
/* ------------------------------------------------------------------------ */
/* Per row: m = max_j x_j; e_j = exp(x_j - m); S = the lane sums of e_j (plain
 * adds, lane l owning groups g with g mod lanes == l, ascending j) folded by the
 * butterfly; loss = log(S) - (x_y - m). With dlogits requested:
 * d_j = (e_j * (1/S) - [j == y]) * dscale, e_j recomputed. A label outside
 * [0, V) gives loss NaN and a NaN dlogits row. */
typedef struct {
    int64_t V, ld, ldd;
    const float *x;
    const int32_t *labels;
    float *loss, *dl;
    float dscale;
    int lanes, group;
    int64_t bad[MAX_THREADS];     /* per-thread count of out-of-range labels */
} xent_ctx;

static void xent_rows(int64_t lo, int64_t hi, int tix, void *c) {
    xent_ctx *q = (xent_ctx *)c;
    float s[1024];
    int64_t bad = 0;
    for (int64_t r = lo; r < hi; ++r) {
        const float *x = q->x + r * q->ld;
        int64_t y = q->labels[r];
        float *d = q->dl ? q->dl + r * q->ldd : NULL;
        if (y < 0 || y >= q->V) {
            ++bad;
            q->loss[r] = NAN;
            if (d) for (int64_t j = 0; j < q->V; ++j) d[j] = NAN;
            continue;
        }
        float m = x[0];
        /* max, NaN-propagating: a NaN anywhere in the row makes m NaN */
        for (int64_t j = 1; j < q->V; ++j) if (x[j] > m || x[j] != x[j]) m = x[j];
        for (int l = 0; l < q->lanes; ++l) s[l] = 0.0f;
        for (int64_t j = 0; j < q->V; ++j) {
            int l = (int)((j / q->group) % q->lanes);
            s[l] = s[l] + detor_exp(x[j] - m);
        }
        float S = butterfly(s, q->lanes);
        q->loss[r] = detor_log(S) - (x[y] - m);
        if (d) {
            float inv = 1.0f / S;
            for (int64_t j = 0; j < q->V; ++j) {
                float e = detor_exp(x[j] - m);
                float onehot = (j == y) ? 1.0f : 0.0f;
                d[j] = (e * inv - onehot) * q->dscale;
            }
        }
    }
    q->bad[tix] = bad;
}

/* ------------------------------------------------------------------------ */
/* causal softmax of attention scores                                        */
/* ------------------------------------------------------------------------ */
/* The cross-entropy's row spelling applied to attention probabilities
 * (design notes R29): row r keeps the columns j < n_r = min(cols, r + diag + 1);
 * x_j = s_j * scale (one rounding; 1/8 for 64-wide heads, exact);
 * m = max (NaN-propagating); e_j = exp(x_j - m); S = the lanes-chain sum of
 * e_j folded by the butterfly; p_j = e_j * (1 / S); masked columns p_j = +0.
 * A row with no column kept is +0 throughout. */
typedef struct {
    int64_t cols, lds, ldp, diag;
    const float *s;
    float scale;
    float *p;
    int lanes, group;
} smax_ctx;

static void smax_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    smax_ctx *q = (smax_ctx *)c;
    float acc[1024];
    for (int64_t r = lo; r < hi; ++r) {
        const float *s = q->s + r * q->lds;
        float *p = q->p + r * q->ldp;
        int64_t nr = r + q->diag + 1;
        if (nr > q->cols) nr = q->cols;
        if (nr < 0) nr = 0;
        for (int64_t j = nr; j < q->cols; ++j) p[j] = 0.0f;
        if (nr == 0) continue;
        float m = s[0] * q->scale;
        for (int64_t j = 1; j < nr; ++j) {
            float x = s[j] * q->scale;
            if (x > m || x != x) m = x;
        }
        for (int l = 0; l < q->lanes; ++l) acc[l] = 0.0f;
        for (int64_t j = 0; j < nr; ++j) {
            int l = (int)((j / q->group) % q->lanes);
            acc[l] = acc[l] + detor_exp(s[j] * q->scale - m);
        }
        float inv = 1.0f / butterfly(acc, q->lanes);
        for (int64_t j = 0; j < nr; ++j) p[j] = detor_exp(s[j] * q->scale - m) * inv;
    }
}

/* Causal softmax backward (design notes R34): per row, over the kept columns
 * j < n_r, dot = the lanes-chain sum of fmaf(dP_j, P_j, .) (lane l owning
 * groups g mod lanes == l, ascending, from +0) folded by the butterfly; then
 * dS_j = (P_j * (dP_j - dot)) * scale; masked columns +0. */
typedef struct {
    int64_t cols, ld, diag;
    const float *p, *dp;
    float scale;
    float *ds;
    int lanes, group;
} smaxb_ctx;

static void smaxb_rows(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    smaxb_ctx *q = (smaxb_ctx *)c;
    float acc[1024];
    for (int64_t r = lo; r < hi; ++r) {
        const float *p = q->p + r * q->ld, *dp = q->dp + r * q->ld;
        float *ds = q->ds + r * q->ld;
        int64_t nr = r + q->diag + 1;
        if (nr > q->cols) nr = q->cols;
        if (nr < 0) nr = 0;
        for (int64_t j = nr; j < q->cols; ++j) ds[j] = 0.0f;
        if (nr == 0) continue;
        for (int l = 0; l < q->lanes; ++l) acc[l] = 0.0f;
        for (int64_t j = 0; j < nr; ++j) {
            int l = (int)((j / q->group) % q->lanes);
            acc[l] = fmaf(dp[j], p[j], acc[l]);
        }
        float dot = butterfly(acc, q->lanes);
        for (int64_t j = 0; j < nr; ++j) ds[j] = (p[j] * (dp[j] - dot)) * q->scale;
    }
}

void detor_softmax_causal_bwd(int64_t rows, int64_t cols, const float *p, const float *dp,
                              int64_t ld, float scale, int64_t diag, float *ds, int lanes,
                              int group, int nthreads) {
    if (lanes < 1 || lanes > 1024 || group < 1 || cols < 1) return;
    smaxb_ctx c = {cols, ld, diag, p, dp, scale, ds, lanes, group};
    parallel_for(rows, nthreads, smaxb_rows, &c);
}

void detor_softmax_causal(int64_t rows, int64_t cols, const float *s, int64_t lds,
                          float scale, int64_t diag, float *p, int64_t ldp, int lanes,
                          int group, int nthreads) {
    if (lanes < 1 || lanes > 1024 || group < 1 || cols < 1) return;
    smax_ctx c = {cols, lds, ldp, diag, s, scale, p, lanes, group};
    parallel_for(rows, nthreads, smax_rows, &c);
}

int64_t detor_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                   const int32_t *labels, float *loss, float *dlogits,
                   int64_t ldd, float dscale, int lanes, int group, int nthreads) {
    if (lanes < 1 || lanes > 1024 || group < 1 || V < 1) return -1;
    xent_ctx *c = (xent_ctx *)calloc(1, sizeof(xent_ctx));
    if (!c) return -1;
    c->V = V; c->ld = ld; c->ldd = ldd; c->x = logits; c->labels = labels;
    c->loss = loss; c->dl = dlogits; c->dscale = dscale;
    c->lanes = lanes; c->group = group;
#ifdef SABOTAGE_XENT_LANES32
    c->lanes = 32;   /* separating arm: the RMSNorm's 32 chains */
#endif
    parallel_for(rows, nthreads, xent_rows, c);
    int64_t total = 0;
    for (int t = 0; t < MAX_THREADS; ++t) total += c->bad[t];
    free(c);
    return total;
}

/* ------------------------------------------------------------------------ */
/* mean of n floats                                                          */
/* ------------------------------------------------------------------------ */
float detor_mean(int64_t n, const float *x, int lanes, int group) {
    float s[1024];
    if (lanes < 1 || lanes > 1024 || group < 1 || n < 1) return NAN;
    for (int l = 0; l < lanes; ++l) s[l] = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        int l = (int)((i / group) % lanes);
        s[l] = s[l] + x[i];
    }
    float S = butterfly(s, lanes);
    return S / (float)n;
}

/* ------------------------------------------------------------------------ */
/* AdamW                                                                     */
/* ------------------------------------------------------------------------ */
void detor_adamw_bias_correction(int64_t step, float beta1, float beta2,
                                 float *bc1, float *bc2) {
    float p1 = beta1, p2 = beta2;
    for (int64_t t = 2; t <= step; ++t) { p1 = p1 * beta1; p2 = p2 * beta2; }
    *bc1 = 1.0f - p1;
    *bc2 = 1.0f - p2;
}

typedef struct {
    float *p, *m, *v;
    const float *g;
    float lr, b1, b2, eps, omb1, omb2, wdf, bc1, bc2;
} adamw_ctx;

static void adamw_range(int64_t lo, int64_t hi, int tix, void *c) {
    (void)tix;
    adamw_ctx *a = (adamw_ctx *)c;
    for (int64_t i = lo; i < hi; ++i) {
        float g = a->g[i];
        float m = fmaf(a->b1, a->m[i], a->omb1 * g);
        float v = fmaf(a->b2, a->v[i], a->omb2 * (g * g));
#ifndef SABOTAGE_ADAMW_RECIP_BC
        float mh = m / a->bc1;
        float vh = v / a->bc2;
#else   /* separating arm: multiplies by the reciprocal corrections */
        float mh = m * (1.0f / a->bc1);
        float vh = v * (1.0f / a->bc2);
#endif
        float u = mh / (sqrtf(vh) + a->eps);
        a->p[i] = fmaf(-a->lr, u, a->p[i] * a->wdf);
        a->m[i] = m;
        a->v[i] = v;
    }
}

void detor_adamw(int64_t n, float *p, const float *g, float *m, float *v,
                 float lr, float beta1, float beta2, float eps,
                 float weight_decay, int64_t step, int nthreads) {
    adamw_ctx a;
    a.p = p; a.m = m; a.v = v; a.g = g;
    a.lr = lr; a.b1 = beta1; a.b2 = beta2; a.eps = eps;
    a.omb1 = 1.0f - beta1;
    a.omb2 = 1.0f - beta2;
    a.wdf = 1.0f - lr * weight_decay;
    detor_adamw_bias_correction(step, beta1, beta2, &a.bc1, &a.bc2);
    parallel_for(n, nthreads, adamw_range, &a);
}

/* ------------------------------------------------------------------------ */
/* accuracy scans against the C library's double exp / log                   */
/* ------------------------------------------------------------------------ */
/* ulp of the float grid at the exact value r (r finite, in float range). */
static double float_ulp_at(double r) {
    double a = fabs(r);
    if (a < (double)FLT_MIN) return 0x1p-149;
    int e;
    frexp(a, &e);                 /* a = f 2^e, f in [0.5, 1) */
    return ldexp(1.0, e - 1 - 23);
}

typedef struct {
    uint32_t lo;
    int is_log;
    double worst[MAX_THREADS];
    uint32_t worst_bits[MAX_THREADS];
} scan_ctx;

static void scan_range(int64_t lo, int64_t hi, int tix, void *c) {
    scan_ctx *s = (scan_ctx *)c;
    double worst = 0.0;
    uint32_t wb = 0;
    for (int64_t i = lo; i < hi; ++i) {
        uint32_t bits = s->lo + (uint32_t)i;
        float x = u2f(bits);
        if (x != x) continue;
        double ref = s->is_log ? log((double)x) : exp((double)x);
        if (isinf(ref) || fabs(ref) > (double)FLT_MAX) continue;
        float y = s->is_log ? detor_log(x) : detor_exp(x);
        double err;
        if (isinf(y) || y != y) err = INFINITY;
        else err = fabs((double)y - ref) / float_ulp_at(ref);
        if (err > worst) { worst = err; wb = bits; }
    }
    s->worst[tix] = worst;
    s->worst_bits[tix] = wb;
}

static void ulp_scan(int is_log, uint32_t lo_bits, uint32_t hi_bits, int nthreads,
                     double *max_ulp, uint32_t *worst_bits) {
    *max_ulp = -1.0; *worst_bits = 0;
    if (hi_bits < lo_bits) return;
    scan_ctx *s = (scan_ctx *)calloc(1, sizeof(scan_ctx));
    if (!s) return;
    s->lo = lo_bits; s->is_log = is_log;
    for (int k = 0; k < MAX_THREADS; ++k) s->worst[k] = -1.0;
    parallel_for((int64_t)hi_bits - (int64_t)lo_bits + 1, nthreads, scan_range, s);
    for (int k = 0; k < MAX_THREADS; ++k) {
        if (s->worst[k] > *max_ulp) { *max_ulp = s->worst[k]; *worst_bits = s->worst_bits[k]; }
    }
    free(s);
}

/* sin / cos: which = 0 sin, 1 cos. The error is in ulps of the true value
 * where |true| >= 2^-6, and in ulps of 2^-6 (an absolute error of 2^-29)
 * nearer the zeros, where an ulp of the tiny true value measures nothing a
 * rotation cares about. Inputs step through the bit patterns [lo, hi). */
typedef struct {
    uint32_t lo, step;
    int which;
    double worst[MAX_THREADS];
    uint32_t worst_bits[MAX_THREADS];
} tscan_ctx;

static void tscan_range(int64_t lo, int64_t hi, int tix, void *c) {
    tscan_ctx *s = (tscan_ctx *)c;
    double worst = 0.0;
    uint32_t wb = 0;
    for (int64_t i = lo; i < hi; ++i) {
        uint32_t bits = s->lo + (uint32_t)(i * (int64_t)s->step);
        float x = u2f(bits);
        if (x != x || fabsf(x) > TRIG_MAX) continue;
        double ref = s->which ? cos((double)x) : sin((double)x);
        float y = s->which ? detor_cos(x) : detor_sin(x);
        double unit = fabs(ref) >= 0x1p-6 ? float_ulp_at(ref) : 0x1p-29;
        double err = (y != y) ? INFINITY : fabs((double)y - ref) / unit;
        if (err > worst) { worst = err; wb = bits; }
    }
    s->worst[tix] = worst;
    s->worst_bits[tix] = wb;
}

double detor_sincos_ulp_scan(int which, uint32_t lo, uint32_t hi, uint32_t step,
                             int nthreads, uint32_t *worst) {
    *worst = 0;
    if (hi <= lo || step == 0) return -1.0;
    tscan_ctx *s = (tscan_ctx *)calloc(1, sizeof(tscan_ctx));
    if (!s) return -1.0;
    s->lo = lo; s->step = step; s->which = which;
    for (int k = 0; k < MAX_THREADS; ++k) s->worst[k] = -1.0;
    parallel_for(((int64_t)hi - (int64_t)lo + step - 1) / step, nthreads, tscan_range, s);
    double m = -1.0;
    for (int k = 0; k < MAX_THREADS; ++k)
        if (s->worst[k] > m) { m = s->worst[k]; *worst = s->worst_bits[k]; }
    free(s);
    return m;
}

void detor_exp_ulp_scan(uint32_t lo_bits, uint32_t hi_bits, int nthreads,
                        double *max_ulp, uint32_t *worst_bits) {
    ulp_scan(0, lo_bits, hi_bits, nthreads, max_ulp, worst_bits);
}
void detor_log_ulp_scan(uint32_t lo_bits, uint32_t hi_bits, int nthreads,
                        double *max_ulp, uint32_t *worst_bits) {
    ulp_scan(1, lo_bits, hi_bits, nthreads, max_ulp, worst_bits);
}
