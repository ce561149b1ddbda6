/*
 * det_oracle.h -- the CPU oracle for the frozen FP32 numerical profile, v1.
 *
 * TEST INFRASTRUCTURE ONLY. This header and det_oracle.c are the plain, slow,
 * obviously-ordered restatement of what the GPU library computes. Only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or constant with the CUDA library: every
 * constant below is re-derived here from its mathematical definition.
 *
 * Sources ("mojolearn" PyPI page, section "What bitwise identity means, and why
 * it is not the default"; same text in "The exact scope of the claim"): the
 * profile fixes reduction order, partitioning, FMA policy, flush-to-zero seams,
 * the spellings of exp and log, and tie rules. The pages name these knobs but
 * print no values; the values implemented here are the v1 readings that the
 * repository's design notes list one by one.
 *
 * Floating-point environment: the oracle must be compiled with
 * -ffp-contract=off, no fast-math, FLT_EVAL_METHOD == 0, and must run with
 * subnormals enabled (detor_fp_env_ok() checks the last two at run time).
 */
#ifndef DET_ORACLE_H
#define DET_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1 when the host FP environment can run the profile (no FTZ/DAZ, float
 * expressions evaluated in float), else 0. */
int detor_fp_env_ok(void);

/* The profile's exp and log spellings for one float. */
float detor_exp(float x);
float detor_log(float x);

/* The profile's sin and cos spellings (det_oracle.c), defined for
 * |x| <= 2^20; NaN outside and for NaN. */
float detor_sin(float x);
float detor_cos(float x);

/* Elementwise maps over n floats. */
void detor_exp_n(int64_t n, const float *x, float *y, int nthreads);
void detor_log_n(int64_t n, const float *x, float *y, int nthreads);
void detor_sin_n(int64_t n, const float *x, float *y, int nthreads);
void detor_cos_n(int64_t n, const float *x, float *y, int nthreads);

/* Rotary position embedding in place (det_oracle.c): rows of `heads` heads of
 * head_dim floats, row t at position t mod seq_len; pairs (2i, 2i + 1) of a
 * head turn by the angle pos * theta^(-2i / head_dim). */
void detor_rope(int64_t rows, int64_t heads, int64_t head_dim, float *x, int64_t ldx,
                int64_t seq_len, float theta, int nthreads);

/* Fixed-order GEMM: C = op(A) * op(B), op = optional transpose of a row-major
 * operand. Each C[i,j] is a sequential fmaf chain from +0 over each k_chunk-wide
 * chunk of k in ascending k; the chunk partials are summed left to right with
 * the first taken as is. K == 0 gives +0. */
void detor_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
                const float *A, int64_t lda, const float *B, int64_t ldb,
                float *C, int64_t ldc, int64_t k_chunk, int nthreads);

/* RMSNorm over `rows` rows of D floats: lanes-way chain sums of x^2 by fmaf,
 * lane l owning the `group`-wide groups g with g mod lanes == l, then an xor
 * butterfly; y = (x * r) * gain with r = 1 / sqrt(ss / D + eps). inv_rms may be
 * NULL. */
void detor_rmsnorm(int64_t rows, int64_t D, const float *x, int64_t ldx,
                   const float *gain, float eps, float *y, int64_t ldy,
                   float *inv_rms, int lanes, int group, int nthreads);

/* C = C + op(A) op(B): the profile GEMM's result R (chunk partials left to
 * right) added to the old C by one rounded addition, C on the left. */
void detor_gemm_acc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda, const float *B, int64_t ldb,
                    float *C, int64_t ldc, int64_t k_chunk, int nthreads);

/* out[i] = scale * (((g_0[i] + g_1[i]) + g_2[i]) + ... + g_{S-1}[i]) over the
 * S shards g_s = shards + s * ld, left to right, one rounding each. */
void detor_shardsum(int64_t nshards, int64_t n, const float *shards, int64_t ld,
                    float scale, float *out, int nthreads);

/* Max ulp error of detor_sin (which = 0) or detor_cos (which = 1) against
 * the C library's double sin/cos over the floats [lo, hi) stepping by `step`
 * bit patterns; the worst input goes to *worst. */
double detor_sincos_ulp_scan(int which, uint32_t lo, uint32_t hi, uint32_t step,
                             int nthreads, uint32_t *worst);

/* SwiGLU's gate: out = (g / (1 + exp(-g))) * u element-wise (det_oracle.c). */
void detor_swiglu(int64_t n, const float *gate, const float *up, float *out, int nthreads);

/* SwiGLU backward (det_oracle.c): d_gate and d_up from gate, up and the
 * upstream gradient dh. */
void detor_swiglu_bwd(int64_t n, const float *gate, const float *up, const float *dh,
                      float *d_gate, float *d_up, int nthreads);

/* Causal softmax backward: dS from the probabilities P and dP, row r keeping
 * the columns j <= r + diag; masked columns +0. */
void detor_softmax_causal_bwd(int64_t rows, int64_t cols, const float *p, const float *dp,
                              int64_t ld, float scale, int64_t diag, float *ds, int lanes,
                              int group, int nthreads);

/* Rotary embedding backward in place: the pairs turned by -a. */
void detor_rope_bwd(int64_t rows, int64_t heads, int64_t head_dim, float *x, int64_t ldx,
                    int64_t seq_len, float theta, int nthreads);

/* Embedding backward: dE[v] = the left-to-right sum of dX[t] over the tokens
 * t (ascending) with tokens[t] == v; +0 for ids no token uses. */
void detor_embedding_bwd(int64_t ntok, int64_t dim, const int32_t *tokens, const float *dx,
                         int64_t vocab, float *de, int nthreads);

/* Residual add: out = a + b element-wise, one rounding. */
void detor_add(int64_t n, const float *a, const float *b, float *out, int nthreads);

/* Causal softmax of attention scores (det_oracle.c): row r keeps the columns
 * j <= r + diag of x = s * scale; p = exp(x - max) * (1 / S) with S the
 * lanes-chain sum; masked columns are +0. */
void detor_softmax_causal(int64_t rows, int64_t cols, const float *s, int64_t lds,
                          float scale, int64_t diag, float *p, int64_t ldp, int lanes,
                          int group, int nthreads);

/* RMSNorm backward (see det_oracle.c): dx (rows x D, row stride lddx) and
 * dgain (D) from x, gain, the forward's inv_rms and dy. */
void detor_rmsnorm_bwd(int64_t rows, int64_t D, const float *x, int64_t ldx,
                       const float *gain, const float *inv_rms, const float *dy,
                       int64_t lddy, float *dx, int64_t lddx, float *dgain,
                       int lanes, int group, int64_t k_chunk, int nthreads);

/* Softmax cross-entropy per row (see det_oracle.c). dlogits may be NULL.
 * Returns the number of rows whose label was out of range (their loss, and
 * their dlogits row if requested, are NaN). */
int64_t detor_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                   const int32_t *labels, float *loss, float *dlogits,
                   int64_t ldd, float dscale, int lanes, int group, int nthreads);

/* Mean of n floats: lanes-way chain sums (plain adds), xor butterfly, then a
 * division by (float)n. */
float detor_mean(int64_t n, const float *x, int lanes, int group);

/* 1 - beta^step with beta^step formed by step-1 sequential float products. */
void detor_adamw_bias_correction(int64_t step, float beta1, float beta2,
                                 float *bc1, float *bc2);

/* One decoupled-weight-decay Adam (AdamW) update of p, m, v in place. */
void detor_adamw(int64_t n, float *p, const float *g, float *m, float *v,
                 float lr, float beta1, float beta2, float eps,
                 float weight_decay, int64_t step, int nthreads);

/* Accuracy scans against the C library's double exp/log, over the float bit
 * patterns [lo_bits, hi_bits] (inclusive, sign-magnitude order irrelevant: all
 * patterns in the range are visited). Writes the largest error in units of the
 * float ulp of the exact result and the bit pattern where it occurred. Inputs
 * whose exact result overflows the float range are skipped. */
void detor_exp_ulp_scan(uint32_t lo_bits, uint32_t hi_bits, int nthreads,
                        double *max_ulp, uint32_t *worst_bits);
void detor_log_ulp_scan(uint32_t lo_bits, uint32_t hi_bits, int nthreads,
                        double *max_ulp, uint32_t *worst_bits);

#ifdef __cplusplus
}
#endif
#endif
