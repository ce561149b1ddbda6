/*
 * detfp32.h -- C ABI of the bit-exact fixed-order FP32 library for GB300
 * (sm_103a): libdetfp32.so.
 *
 * What it computes. Four operations of FP32 transformer training, under one
 * frozen numerical profile, so that the result bits depend only on the inputs,
 * the shapes and the profile version. They do not depend on the launch
 * configuration, the stream, the tiling or the run. The profile fixes
 * reduction order, partitioning, FMA policy, flush-to-zero behaviour, the
 * spellings of exp and log, and tie rules ("mojolearn" PyPI page, section
 * "What bitwise identity means, and why it is not the default"; the same list
 * in "The exact scope of the claim"). Profile v1's values are stated at each
 * entry point below.
 *
 * Conventions shared by every entry point.
 *  - Pointers named as device pointers must be device memory of the current
 *    CUDA device (cudaMalloc, or torch's caching allocator). The caller owns
 *    all memory. The library allocates nothing and keeps no state between
 *    calls, except a per-device watchdog word (det_watchdog_status).
 *  - Matrices are row-major float32 with an explicit row stride (ld*, in
 *    elements, >= the row length).
 *  - `stream` is a cudaStream_t; NULL means the legacy default stream. Every
 *    call is asynchronous on that stream: it validates its arguments on the
 *    host, launches, and returns without synchronising.
 *  - The return value is a det_status. Argument, profile and device checks
 *    are synchronous. A failed launch returns DET_ERR_CUDA. Nothing throws or
 *    exits across the ABI.
 *  - float32 only; there is no other precision and no fallback path. The
 *    pages' FP32-only claim is in "The exact scope of the claim".
 *  - Subnormals are kept everywhere: no flush-to-zero, no fast math.
 */
#ifndef DETFP32_H
#define DETFP32_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Identical to cudaStream_t. */
typedef struct CUstream_st *det_stream_t;

#define DET_PROFILE_VERSION 1u

/* The numerical profile the caller asks for. Version 1 is the only one
 * implemented; every field must hold its v1 value, or the call is refused
 * with DET_ERR_PROFILE. A change to any value would change result bits, so
 * the library never runs an unlisted profile. The pages require the same:
 * refusal by a named error, never a weaker result ("mojolearn" PyPI page,
 * "Which families offer which tiers"). */
typedef struct det_profile_v1 {
    uint32_t version;     /* 1 */
    uint32_t k_chunk;     /* 256: GEMM k-chunk width */
    uint32_t rms_lanes;   /* 32: chains per RMSNorm row (and per mean) */
    uint32_t xent_lanes;  /* 256: chains per cross-entropy row */
    uint32_t lane_group;  /* 4: consecutive elements a chain owns per sweep */
    uint32_t flags;       /* 0: no FTZ, no fast math (no other value exists) */
} det_profile_v1;

typedef enum det_status {
    DET_OK = 0,
    DET_ERR_INVALID_ARG = 1,        /* null pointer, negative size, ld too small */
    DET_ERR_PROFILE = 2,            /* profile version or field not implemented */
    DET_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    DET_ERR_ALIGNMENT = 4,          /* reserved */
    DET_ERR_WORKSPACE = 5,          /* workspace too small or misaligned */
    DET_ERR_TIMEOUT = 6,            /* a device-side bounded wait gave up */
    DET_ERR_CUDA = 7                /* a CUDA runtime call or launch failed */
} det_status;

/* Fills *p with profile v1. */
void det_profile_default(det_profile_v1 *p);

/* Static description of a status code (never NULL). */
const char *det_status_string(int status);

/* Fixed-order GEMM: C = op(A) * op(B), with op(X) = X or X^T.
 *
 * Profile v1 (a1-a3): for each C[i,j] and each 256-wide chunk c of k
 * ([256c, min(256c+256, K))), P_c is a sequential fmaf chain that starts at
 * +0.0f and runs over k in ascending order: acc = fmaf(opA[i,k], opB[k,j], acc).
 * Then C[i,j] = P_0 + P_1 + ... summed left to right (the first partial taken
 * as is). K == 0 gives C = +0. The bits depend only on (M, N, K, the operand
 * values, the profile), never on tiling or launch configuration.
 *
 * transA == 0: A is M x K row-major, row stride lda >= K.
 * transA != 0: A is stored K x M row-major (lda >= M), and op(A) = A^T; this
 *              is the weight-gradient form dW = X^T dY (contraction over the
 *              tokens).
 * transB == 0: B is K x N row-major, ldb >= N.
 * transB != 0: B is stored N x K row-major (ldb >= K), op(B) = B^T; this is
 *              the [out_features, in_features] Linear layout.
 * C: M x N row-major, ldc >= N, device pointer, must not overlap A or B.
 * workspace / workspace_bytes: optional device scratch (16-byte aligned, not
 *   overlapping A, B or C). With at least detgemm_workspace_bytes() bytes the
 *   library may cut K into groups of whole 256-wide chunks computed by
 *   different CTAs: each chunk partial P_c (the first group's running total
 *   as one) is written to the workspace and a second kernel adds them left
 *   to right. For a large product with transA ==
 *   0 it may instead copy A transposed (K x M) into the workspace and read
 *   that copy, which its FFMA loop consumes faster; likewise B (N x K, to
 *   K x N) for transB != 0. With NULL, or too few
 *   bytes, every output's chunks are computed by one thread from A in place.
 *   The result bits are the same either way; only the speed differs. Calls
 *   that share a workspace must be ordered (one stream).
 * Speed: the kernel stages A and B by TMA when each is 16-byte aligned with a
 *   row stride that is a multiple of 4 floats; otherwise it stages them with
 *   plain loads, about four times slower (same bits). A k-contiguous A read
 *   through its transposed copy needs only the copy aligned. Pad rows that
 *   would miss this (a 50,257-wide logits row to a stride of 50,260).
 *
 * Errors: DET_ERR_INVALID_ARG for negative sizes, a dimension >= 2^31, an ld
 * below its row length or null pointers with nonzero sizes. A TMA wait that
 * exceeds its bound makes the kernel skip its stores and record a code that
 * det_watchdog_status() returns. */
det_status detgemm_f32(const det_profile_v1 *prof, int transA, int transB,
                       int64_t M, int64_t N, int64_t K,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc,
                       void *workspace, size_t workspace_bytes,
                       det_stream_t stream);

/* One product of a group (detgemm_group_f32): the arguments of detgemm_f32,
 * with the same meaning, layout and rules. */
typedef struct det_gemm_problem {
    int transA, transB;
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
} det_gemm_problem;

/* Several independent products in one call, for example the weight gradients
 * of one layer (dW = X^T dY for each of its weights; "mojolearn" PyPI page,
 * section "Install": weight gradients contract over the token count). Every
 * C receives exactly the bits detgemm_f32 would give it: the profile fixes
 * each output's chains and chunk order, never the schedule.
 *
 * problems: count host structs, read during the call. The products are taken
 * in consecutive pairs (0, 1), (2, 3), ... (an odd last one alone); a pair
 * of the same transA/transB layout runs as one launch when the library's
 * model finds that faster -- its work units are dealt out together, which
 * fills the grid's last round from both products -- and otherwise the two
 * run one after the other. Each C must not overlap any A, B or other C.
 * workspace / workspace_bytes: as detgemm_f32's, at least
 * detgemm_group_workspace_bytes() for the same problems to take the faster
 * plans (less, or NULL, still gives the same bits). The calls of a group are
 * asynchronous on `stream`, in order.
 *
 * Errors: as detgemm_f32 for any problem (nothing is launched then);
 * DET_ERR_INVALID_ARG for count < 0 or a null array with count > 0. */
det_status detgemm_group_f32(const det_profile_v1 *prof, int64_t count,
                             const det_gemm_problem *problems, void *workspace,
                             size_t workspace_bytes, det_stream_t stream);

/* Workspace that detgemm_group_f32 can use for these problems on the current
 * device, written to *bytes (a pair that shares a launch needs the sum of its
 * split partials; otherwise the largest single need). */
det_status detgemm_group_workspace_bytes(const det_profile_v1 *prof, int64_t count,
                                         const det_gemm_problem *problems, size_t *bytes);

/* The number of kernels detgemm_group_f32 launches for these problems with a
 * workspace of workspace_bytes, written to *launches (for callers that count
 * or capture launches). Same argument rules; host-only apart from reading the
 * device's SM count. */
det_status detgemm_group_launches(const det_profile_v1 *prof, int64_t count,
                                  const det_gemm_problem *problems, size_t workspace_bytes,
                                  int64_t *launches);

/* Gradient accumulation (beta = 1): C = C + op(A) op(B). The product is formed
 * exactly as detgemm_f32 forms it (256-wide chunk chains from +0, partials
 * added left to right) and then added to the old C by one rounded addition,
 * so accumulating the shards of a batch one after another gives the same bits
 * as detshardsum_f32 over their separate products ("MojoLearn 162M" model
 * card, table "Training": shard gradients summed in a fixed order). The pages
 * print no spelling of the accumulation; this is profile v1's reading.
 *
 * Arguments, layout, workspace and errors as detgemm_f32; C is read and
 * written (K == 0 gives C + 0). */
det_status detgemm_acc_f32(const det_profile_v1 *prof, int transA, int transB,
                           int64_t M, int64_t N, int64_t K,
                           const float *A, int64_t lda,
                           const float *B, int64_t ldb,
                           float *C, int64_t ldc,
                           void *workspace, size_t workspace_bytes,
                           det_stream_t stream);

/* Fixed-order sum of gathered shard gradients ("MojoLearn 162M" model card,
 * table "Training": 64 logical shards, each a mean over 4 x 2,048 tokens,
 * summed in a fixed order). Profile v1 reads the order as left to right:
 *   out[i] = scale * (((g_0[i] + g_1[i]) + g_2[i]) + ... + g_{S-1}[i])
 * one rounding per addition and one multiply (scale = 1/64 gives the mean of
 * 64 shards exactly). A multi-device caller gathers the shard gradients
 * unreduced (an all-gather moves bytes only) and calls this; a collective's
 * own reduction must not be used, because its order is not the profile's.
 *
 * shards: nshards x n floats, shard s at shards + s * ld, ld >= n (device).
 * out: n floats (device); it may be shard 0 itself and must not overlap any
 * other shard. nshards >= 1; n may be 0 (no work).
 * Errors: DET_ERR_INVALID_ARG for nshards < 1, n < 0, ld < n, null pointers
 * with n > 0, or an overlap other than out == shards. */
det_status detshardsum_f32(const det_profile_v1 *prof, int64_t nshards, int64_t n,
                           const float *shards, int64_t ld, float scale, float *out,
                           det_stream_t stream);

/* Workspace that detgemm_f32 can use for this shape and layout on the
 * current device, written to *bytes: for a large product with transA == 0,
 * the transposed copy of A (K x M, rows padded to 4 floats) where it pays,
 * and the split-K chunk partials where splitting K helps (after the copy,
 * which is then rounded up to 256 bytes); 0 when neither helps. A smaller
 * workspace that holds the partials alone gives the split without the copy.
 * Same argument rules as detgemm_f32; a host-only query apart from reading
 * the device's SM count. */
det_status detgemm_workspace_bytes(const det_profile_v1 *prof, int transA, int transB,
                                   int64_t M, int64_t N, int64_t K, size_t *bytes);

/* The number of kernels detgemm_f32 launches for this shape and layout with a
 * workspace of workspace_bytes (1 to 5: the transposed copies of B and of A;
 * the GEMM, or the GEMM of the first rows unsplit and then of the rest; the
 * split-K second pass), written to *launches, for callers that count or
 * capture launches. Same argument rules; host-only apart from reading the
 * device's SM count. */
det_status detgemm_launches(const det_profile_v1 *prof, int transA, int transB, int64_t M,
                            int64_t N, int64_t K, size_t workspace_bytes, int64_t *launches);

/* detgemm_f32 for callers that cannot allocate device memory when they
 * multiply: code that runs inside another framework's memory pool, where
 * every allocation must go through that pool, or a latency-critical loop
 * where cudaMalloc's implicit device synchronisation is not acceptable. The
 * pages have no counterpart to this entry point; it only changes where the
 * split-K scratch lives.
 *
 * Same arguments, arithmetic and result bits as detgemm_f32. Where
 * detgemm_f32 would use a workspace, this call uses a scratch array built into
 * the library instead: 64 MiB of device memory that every device which loads
 * the library holds until the process exits. The call itself allocates
 * nothing (no cudaMalloc, no allocating library routine).
 *
 * Limits and sharing:
 *  - A shape whose split plan needs more than 64 MiB (a split-K workspace
 *    above 67,108,864 bytes) is refused with DET_ERR_WORKSPACE; nothing is
 *    launched. A transposed copy of A that needs more than 64 MiB is skipped
 *    (A is read in place). Shapes that need no scratch always run.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents. A call writes every scratch element it reads, so no
 *    clearing is needed, but calls whose kernels overlap on the GPU (two
 *    streams, or concurrent host threads) race on the array: order them.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current). Make that first call before any
 *    stream capture begins. A device reset (cudaDeviceReset) unloads the
 *    library's device code with the context; the first call after it, in
 *    the new context, looks the address up again, so it too belongs before
 *    any capture. */
det_status detgemm_f32_noalloc(const det_profile_v1 *prof, int transA, int transB,
                               int64_t M, int64_t N, int64_t K,
                               const float *A, int64_t lda,
                               const float *B, int64_t ldb,
                               float *C, int64_t ldc, det_stream_t stream);

/* RMSNorm over `rows` rows of D floats: y = (x * r) * gain, with
 * r = 1.0f / sqrtf(ss / (float)D + eps). "MojoLearn 162M" model card, table
 * "Compared with GPT-3 Small": RMSNorm, eps 1e-6, pre-norm.
 *
 * Profile v1 (a4): ss is the sum of squares over 32 chains. Chain l owns the
 * 4-element groups g of the row with g mod 32 == l and accumulates
 * s_l = fmaf(x_j, x_j, s_l) from +0 in ascending j. The chains are then folded
 * by an xor butterfly with offsets 16, 8, 4, 2, 1 (s_l = s_l + s_{l^off}). The
 * divisions and the square root are IEEE round-to-nearest; there is no rsqrt.
 *
 * x: rows x D, row stride ldx >= D (device). gain: D floats (device).
 * y: rows x D, ldy >= D (device; may equal x when ldy == ldx, in place).
 * inv_rms: rows floats receiving r (device) or NULL. D must be >= 1; rows may
 * be 0 (no work). */
det_status detrmsnorm_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                          const float *x, int64_t ldx, const float *gain,
                          float eps, float *y, int64_t ldy, float *inv_rms,
                          det_stream_t stream);

/* RMSNorm backward: the gradients of y = (x * r) * gain with respect to x and
 * gain, given the upstream gradient dy and the forward's r (inv_rms). The
 * pages define the forward ("MojoLearn 162M" model card, table "Compared with
 * GPT-3 Small") and fix, for every operation of training, the reduction order
 * and partitioning ("mojolearn" PyPI page, section "What bitwise identity
 * means, and why it is not the default"); they print no backward spelling.
 *
 * Profile v1, per row (r = inv_rms[row]):
 *   xhat_j = x_j * r,  h_j = dy_j * gain_j         (each rounded once)
 *   dot    = sum of h_j * xhat_j by the forward's arrangement: 32 chains of
 *            fmaf over the 4-element groups g with g mod 32 == l, from +0 in
 *            ascending j, folded by the xor butterfly 16, 8, 4, 2, 1
 *   q      = dot / (float)D                         (IEEE division)
 *   dx_j   = (h_j - xhat_j * q) * r                 (three roundings)
 * and dgain_j, a contraction over the rows, in the GEMM's spelling: for each
 * 256-row chunk an fmaf chain of dy_ij * xhat_ij from +0 in ascending row,
 * the chunk partials added left to right (the first as is). dgain is thus the
 * diagonal of detgemm_f32's xhat^T dy. rows == 0 writes dgain = +0.
 *
 * x, dy: rows x D, row strides ldx, lddy >= D (device). gain: D floats,
 * inv_rms: rows floats (device). dx: rows x D, lddx >= D (device); it may
 * equal dy when lddx == lddy (in place) and must not overlap x, gain or
 * inv_rms otherwise. dgain: D floats (device), written.
 * workspace / workspace_bytes: device scratch, 16-byte aligned, of at least
 * detrmsnorm_bwd_workspace_bytes() bytes (0 when rows <= 256), not
 * overlapping any other argument: the chunk partials of dgain. Calls that
 * share a workspace must be ordered (one stream).
 *
 * Errors: DET_ERR_INVALID_ARG for negative rows, D < 1, a dimension >= 2^31,
 * a stride below D or a null pointer that the shape needs; DET_ERR_WORKSPACE
 * when the workspace is needed and missing, too small or misaligned. A TMA
 * wait that exceeds its bound makes the kernel skip its stores and record
 * bit 2 of det_watchdog_status(). */
det_status detrmsnorm_bwd_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                              const float *x, int64_t ldx, const float *gain,
                              const float *inv_rms, const float *dy, int64_t lddy,
                              float *dx, int64_t lddx, float *dgain,
                              void *workspace, size_t workspace_bytes,
                              det_stream_t stream);

/* Workspace detrmsnorm_bwd_f32 needs for rows x D, written to *bytes:
 * ceil(rows / 256) * D floats when rows > 256, else 0. Host-only. */
det_status detrmsnorm_bwd_workspace_bytes(const det_profile_v1 *prof, int64_t rows,
                                          int64_t D, size_t *bytes);

/* Softmax cross-entropy per row of V logits, with an optional gradient and an
 * optional mean. Cross entropy is on the verified path in "mojolearn"
 * (andrewhendel.com), "Handing training off between vendors".
 *
 * Profile v1 (a5): m = max_j x_j (order-free; bit-inert for finite inputs).
 * e_j = exp(x_j - m), with the profile's exp (detexp_f32). S is the sum of the
 * e_j over 256 chains (chain l owns the 4-element groups g with
 * g mod 256 == l, plain adds from +0 in ascending j), folded by the xor
 * butterfly 16, 8, 4, 2, 1, 32, 64, 128. loss = log(S) - (x_y - m), with the
 * profile's log (detlog_f32).
 * dlogits (optional): d_j = (e_j * (1.0f / S) - [j == y]) * dscale.
 * loss_mean (optional): the 32-chain tree (groups of 4, plain adds) over the
 * rows' losses, divided by (float)rows.
 *
 * logits: rows x V, row stride ld >= V (device; the rows need not be 16-byte
 *         aligned).
 * labels: rows int32 (device).
 * loss:   rows floats (device).
 * loss_mean: 1 float (device) or NULL.
 * dlogits: rows x V, stride ldd >= V (device) or NULL. It may be exactly
 *          logits (same pointer and ldd == ld: computed in place); any other
 *          overlap with logits is not allowed.
 * dev_status: one int32 (device) or NULL. A label outside [0, V) sets bit 0
 *          (atomic OR; the library never clears it), and that row's loss and
 *          dlogits row are NaN.
 * V >= 1; rows may be 0. */
det_status detxent_f32(const det_profile_v1 *prof, int64_t rows, int64_t V,
                       const float *logits, int64_t ld, const int32_t *labels,
                       float *loss, float *loss_mean, float *dlogits,
                       int64_t ldd, float dscale, int32_t *dev_status,
                       det_stream_t stream);

/* AdamW hyperparameters for one update (host struct, read during the call).
 * "MojoLearn 162M" model card, table "Training": AdamW, beta (0.9, 0.95),
 * eps 1e-8, weight decay 0.1, no gradient clipping; lr from the schedule. */
typedef struct det_adamw_hp {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    int64_t step;         /* 1-based step number t (>= 1) */
} det_adamw_hp;

/* AdamW's bias corrections for step t: *bc1 = 1 - beta1^t and
 * *bc2 = 1 - beta2^t, where beta^t is the product of t-1 sequential float
 * multiplications (beta * beta * ... * beta, each product rounded once), and
 * the difference is rounded once. "MojoLearn 162M" model card, table
 * "Training": AdamW, beta (0.9, 0.95); the pages print no spelling of the
 * correction, and this is profile v1's reading. detadamw_f32 divides by these
 * two values, so a caller can read, check or log exactly the corrections an
 * update uses.
 *
 * A host-only call (no device, no stream); bc1 and bc2 are host pointers.
 * Errors: DET_ERR_INVALID_ARG for step < 1, a beta outside [0, 1] (or NaN) or
 * a null pointer; nothing is written then. */
det_status det_adamw_bias_correction(int64_t step, float beta1, float beta2,
                                     float *bc1, float *bc2);

/* One AdamW update of n parameters, in place on p, m, v (device arrays of n
 * floats; g read-only). Decoupled decay applied to every element.
 *
 * Profile v1 (a6): bc1 and bc2 are det_adamw_bias_correction(hp->step,
 * hp->beta1, hp->beta2), formed on the host at the call; then per element
 *   m' = fmaf(beta1, m, (1 - beta1) * g)
 *   v' = fmaf(beta2, v, (1 - beta2) * (g * g))
 *   u  = (m' / bc1) / (sqrtf(v' / bc2) + eps)
 *   p' = fmaf(-lr, u, p * (1 - lr * weight_decay))
 * where (1 - beta1), (1 - beta2) and (1 - lr * weight_decay) are rounded to
 * float once each. n may be 0.
 * Errors: DET_ERR_INVALID_ARG for n < 0, a null hp, hp->step < 1, a beta
 * outside [0, 1] (or NaN), or null arrays with n > 0. */
det_status detadamw_f32(const det_profile_v1 *prof, int64_t n, float *p,
                        const float *g, float *m, float *v,
                        const det_adamw_hp *hp, det_stream_t stream);

/* Elementwise profile exp / log over n floats (device x -> device y; y may
 * equal x). These are the spellings the cross-entropy uses
 * ("mojolearn" PyPI page, section "What bitwise identity means...": the
 * spellings of exp and log are part of the profile).
 *
 * exp (v1): NaN -> NaN; x > 0x1.62e42ep+6 -> +Inf; x < -104 -> +0; otherwise
 * n = rintf(x * log2(e)) (ties to even), r = x - n ln2 in two fmaf steps
 * (ln2 split in two floats), a degree-7 Taylor polynomial in r by fmaf
 * Horner, then scaling by 2^n with a single rounding.
 * log (v1): x < 0 or NaN -> NaN, 0 -> -Inf, +Inf -> +Inf; otherwise
 * x = 2^e f with f in (sqrt(1/2), sqrt 2), u = f - 1, s = u / (2 + u),
 * log f = u - (h - s (h + R)) with h = u^2/2 and R the atanh series to z^5
 * in z = s^2, and log x = e ln2 + log f by two fmaf steps. */
det_status detexp_f32(const det_profile_v1 *prof, int64_t n, const float *x,
                      float *y, det_stream_t stream);
det_status detlog_f32(const det_profile_v1 *prof, int64_t n, const float *x,
                      float *y, det_stream_t stream);

/* ------------------------------------------------------------------ block forward
 * The rest of a decoder block's forward ("MojoLearn 162M" model card, table
 * "Compared with GPT-3 Small": 12 heads of 64, rotary positions with
 * theta = 10,000, SwiGLU 2,048 wide, pre-norm residual blocks). The pages fix
 * the profile's reduction order and transcendental spellings but print none
 * of these; the v1 readings are stated with each call. All pointers are
 * device pointers; calls are asynchronous on `stream`. */

/* SwiGLU's gate: out[i] = (g[i] / (1 + exp(-g[i]))) * up[i], with the
 * profile's exp, IEEE division, each operation rounded once. n floats each;
 * out may equal gate or up and must not otherwise overlap them. */
det_status detswiglu_f32(const det_profile_v1 *prof, int64_t n, const float *gate,
                         const float *up, float *out, det_stream_t stream);

/* Residual add: out[i] = a[i] + b[i], one rounding. out may equal a or b. */
det_status detadd_f32(const det_profile_v1 *prof, int64_t n, const float *a,
                      const float *b, float *out, det_stream_t stream);

/* The residual add and the RMSNorm that follows it, in one kernel where the
 * rows allow: x = a + b (detadd_f32's bits, rows x D, all three dense with row
 * stride D), then y = detrmsnorm_f32(x) with gain, eps, y's row stride ldy
 * and inv_rms (nullable) as there: the same bits as the two calls. x must
 * not overlap a, b or y. With 16-byte aligned rows and D a multiple of 4 it
 * is one launch (the streamed RMSNorm reads a's and b's rows by bulk copy
 * and writes x once); otherwise the two operations run apart. */
det_status detadd_rmsnorm_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                              const float *a, const float *b, float *x, const float *gain,
                              float eps, float *y, int64_t ldy, float *inv_rms,
                              det_stream_t stream);

/* Causal softmax of attention scores, row by row: row r keeps the columns
 * j <= (r mod period) + diag of x = scores * scale (one rounding); then the
 * cross-entropy's spelling: m = the row max (NaN-propagating), e = exp(x - m),
 * S = the 256-chain sum (chain l owns the 4-element groups g mod 256 == l, in
 * ascending order) folded by the xor butterfly, p = e * (1 / S). Masked
 * columns are +0; a row that keeps no column is +0 throughout.
 * scores: rows x cols, lds >= cols; p: rows x cols, ldp >= cols; p may equal
 * scores when ldp == lds (in place) and must not otherwise overlap it.
 * period >= 1 (the rows of one square score matrix: its query index is
 * r mod period). With 16-byte aligned scores, lds and cols multiples of 4 and
 * cols <= 2048, each row comes into shared memory by one bulk copy; a wait for
 * a copy that gives up after 2 s sets bit 4 of det_watchdog_status() and
 * leaves the remaining rows unwritten. */
det_status detsoftmax_causal_f32(const det_profile_v1 *prof, int64_t rows, int64_t cols,
                                 const float *scores, int64_t lds, float scale, int64_t diag,
                                 int64_t period, float *p, int64_t ldp, det_stream_t stream);

/* Rotary position embedding, in place: row t of x holds `heads` heads of
 * head_dim floats (row stride ldx >= heads * head_dim) at position
 * pos = t mod seq_len. Pair (2i, 2i+1) of every head turns by
 * a = pos * w_i, w_i = exp(-((float)(2i) / (float)head_dim) * log(theta)) with
 * the profile's exp and log: y0 = x0 cos a - x1 sin a, y1 = x0 sin a +
 * x1 cos a (products rounded, then the difference or sum). head_dim even. */
det_status detrope_f32(const det_profile_v1 *prof, int64_t rows, int64_t heads,
                       int64_t head_dim, float *x, int64_t ldx, int64_t seq_len, float theta,
                       det_stream_t stream);

/* Token embedding: out[t] = table[tokens[t]] for t < ntok (rows of dim
 * floats; table is vocab x dim with row stride ldt, out has row stride ldo).
 * A copy, so exact. A token outside [0, vocab) writes a NaN row and ORs 1
 * into *dev_status (device int32, may be NULL). */
det_status detembedding_f32(const det_profile_v1 *prof, int64_t ntok, int64_t dim,
                            const float *table, int64_t ldt, int64_t vocab,
                            const int32_t *tokens, float *out, int64_t ldo,
                            int32_t *dev_status, det_stream_t stream);

/* The profile's sin and cos over n floats (v1): k = rint(x 2/pi) (ties to
 * even); r = x - k pi/2 by three fmaf steps with pi/2 split in three floats;
 * z = r^2; sin_r = fmaf(r, z Ps(z), r) and cos_r = fmaf(Pc(z), z, 1) with the
 * Taylor terms to degree 9 and 10 by fmaf Horner; the quadrant k mod 4 picks
 * the signs. sin(+-0) = +-0, cos(+-0) = 1; |x| > 2^20 and NaN give NaN. */
det_status detsin_f32(const det_profile_v1 *prof, int64_t n, const float *x, float *y,
                      det_stream_t stream);
det_status detcos_f32(const det_profile_v1 *prof, int64_t n, const float *x, float *y,
                      det_stream_t stream);

/* Causal self-attention over a packed QKV activation: qkv holds batch
 * sequences of seq rows; a row is [Q | K | V], each heads x head_dim, row stride
 * ldqkv >= 3 heads head_dim. For every sequence and head:
 * S = Q K^T (detgemm_f32's arithmetic), P = detsoftmax_causal_f32(S, scale,
 * diag 0), O = P V (detgemm_f32's arithmetic), written to out (batch seq rows
 * of heads x head_dim, row stride ldout >= heads head_dim). The heads run in
 * groups whose seq x seq score buffers share the workspace (at least
 * detattention_workspace_bytes for the same batch, seq, heads and head_dim,
 * 256-byte aligned: about 1 GiB at most, plus 256 bytes, plus, for seq >= 512,
 * a transposed copy of the Q and K blocks, 2 heads head_dim x batch seq
 * floats, from which the score product reads Q and K): each step is one
 * launch over a group, and
 * the score tiles wholly above the diagonal, which the softmax masks, are not
 * computed. P is +0 above the diagonal, so in
 * O = P V the 256-wide k-chunks past a row block's last row add +0 partials;
 * they are skipped when the group's V is finite (counted on the device
 * first), which leaves every bit unchanged. Each head's bits are those of
 * its separate products. out must not overlap qkv or the workspace. batch may be 0.
 * Errors: DET_ERR_INVALID_ARG for seq or heads or head_dim outside 1..65536,
 * batch * seq >= 2^31, strides below their row lengths or null pointers;
 * DET_ERR_WORKSPACE for a missing, short or misaligned workspace. */
det_status detattention_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                            int64_t heads, int64_t head_dim, const float *qkv, int64_t ldqkv,
                            float scale, float *out, int64_t ldout, void *workspace,
                            size_t workspace_bytes, det_stream_t stream);
det_status detattention_workspace_bytes(const det_profile_v1 *prof, int64_t batch,
                                        int64_t seq, int64_t heads, int64_t head_dim,
                                        size_t *bytes);
/* The number of kernels detattention_f32 (backward 0), detattention_bwd_f32
 * (backward 1) or detattention_bwd_saved_f32 (backward 2) launches for these
 * sizes, written to *launches (for callers that count or capture launches).
 * Same argument rules; host-only. */
det_status detattention_launches(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                 int64_t heads, int64_t head_dim, int backward,
                                 int64_t *launches);

/* ------------------------------------------------------------------ block backward
 * The backward of the block operations, for the byte-level LM's training step
 * (the pages train "embedding, transformer forward and backward, cross entropy,
 * and AdamW" bit-identically; "mojolearn" PyPI page, section "Handing training
 * off between vendors"; they print no backward spelling). */

/* SwiGLU backward: with den = 1 + exp(-g), silu = g / den, sig = 1 / den:
 * d_up = dh * silu, d_gate = (dh * up) * (sig * (1 + g * (1 - sig))), each
 * operation rounded once in that order. n floats each; d_gate and d_up must
 * not overlap each other, gate or up (either may be dh itself). */
det_status detswiglu_bwd_f32(const det_profile_v1 *prof, int64_t n, const float *gate,
                             const float *up, const float *dh, float *d_gate, float *d_up,
                             det_stream_t stream);

/* Causal softmax backward: over row r's kept columns (j <= (r mod period) +
 * diag), dot = the 256-chain sum of fmaf(dP_j, P_j, .) (the forward's
 * arrangement) folded by the butterfly; dS_j = (P_j * (dP_j - dot)) * scale;
 * masked columns +0. p, dp: rows x cols with row stride ld; ds: row stride
 * ldd; ds may equal dp or p when ldd == ld. */
det_status detsoftmax_causal_bwd_f32(const det_profile_v1 *prof, int64_t rows, int64_t cols,
                                     const float *p, const float *dp, int64_t ld, float scale,
                                     int64_t diag, int64_t period, float *ds, int64_t ldd,
                                     det_stream_t stream);

/* Rotary backward, in place on a gradient laid out as detrope_f32's input:
 * with the forward's angle a, dx0 = dy0 cos a + dy1 sin a,
 * dx1 = dy1 cos a - dy0 sin a. */
det_status detrope_bwd_f32(const det_profile_v1 *prof, int64_t rows, int64_t heads,
                           int64_t head_dim, float *dx, int64_t ldx, int64_t seq_len,
                           float theta, det_stream_t stream);

/* Embedding backward: de[v] (vocab x dim, row stride ldde) = the gradient rows
 * dx[t] (row stride lddx) of the tokens t with tokens[t] == v, added in
 * ascending t, the first as is; +0 for an id no token uses. Every row of de
 * is written. */
det_status detembedding_bwd_f32(const det_profile_v1 *prof, int64_t ntok, int64_t dim,
                                const int32_t *tokens, const float *dx, int64_t lddx,
                                int64_t vocab, float *de, int64_t ldde, det_stream_t stream);

/* Backward of detattention_f32: given the packed qkv the forward read and the
 * gradient of its output (dout, batch seq rows of heads x head_dim), writes the
 * gradients of Q, K and V into dqkv (same packed layout). Per sequence and
 * head, P is recomputed by the forward's spelling; dP = dO V^T, dV = P^T dO,
 * dS = detsoftmax_causal_bwd_f32(P, dP, scale), dQ = dS K, dK = dS^T Q, every
 * product with detgemm_f32's arithmetic, each step one launch over a group of
 * heads as in detattention_f32; dV, dQ and dK skip the +0 chunks of P and dS
 * when dO, K and Q are finite. The workspace (at least
 * detattention_bwd_workspace_bytes, 256-byte aligned) holds two score
 * buffers of a group and, for seq >= 512, transposed copies of the Q block,
 * of dout and of the V block (heads head_dim x batch seq floats each), from
 * which S = Q K^T reads Q and dP = dO V^T reads dO and V. dqkv must not
 * overlap qkv, dout or the workspace. Errors as detattention_f32. */
det_status detattention_bwd_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                int64_t heads, int64_t head_dim, const float *qkv,
                                int64_t ldqkv, const float *dout, int64_t lddout, float scale,
                                float *dqkv, int64_t lddqkv, void *workspace,
                                size_t workspace_bytes, det_stream_t stream);
det_status detattention_bwd_workspace_bytes(const det_profile_v1 *prof, int64_t batch,
                                            int64_t seq, int64_t heads, int64_t head_dim,
                                            size_t *bytes);

/* detattention_bwd_f32, reading P from the forward instead of recomputing it.
 * fwd_workspace / fwd_workspace_bytes: the workspace of the detattention_f32
 * call that read the same qkv with the same batch, seq, heads, head_dim and
 * scale, with nothing written to it since. When that call ran every head as
 * one group (its score buffers fit the 1 GiB cap; detattention_launches then
 * reports 4 or 5), the workspace still holds P for every head, and the
 * backward skips S = Q K^T and the softmax; otherwise it recomputes them as
 * detattention_bwd_f32 does. The results are the same bits either way (P is
 * the same function of the same inputs). The forward wrote P's +0 columns up
 * to the end of each row's 256-row block when its V was finite; when dout is
 * not finite, the backward first fills the rest of those rows with +0 in
 * fwd_workspace, which it may therefore write. workspace: at least
 * detattention_bwd_workspace_bytes. Errors as detattention_bwd_f32, and
 * DET_ERR_WORKSPACE for a null, misaligned or short fwd_workspace. */
det_status detattention_bwd_saved_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                      int64_t heads, int64_t head_dim, const float *qkv,
                                      int64_t ldqkv, const float *dout, int64_t lddout,
                                      float scale, void *fwd_workspace,
                                      size_t fwd_workspace_bytes, float *dqkv, int64_t lddqkv,
                                      void *workspace, size_t workspace_bytes,
                                      det_stream_t stream);

/* Reads, and optionally clears, the current device's watchdog word.
 * *code == 0 means no bounded device wait has ever given up; otherwise bit k
 * identifies the kernel family that gave up (bit 0: GEMM operand staging,
 * bit 1: cross-entropy row staging, bit 2: RMSNorm-backward tile staging,
 * bit 3: RMSNorm row staging, bit 4: causal-softmax row staging).
 * This call synchronises the device (it copies from device memory). */
det_status det_watchdog_status(int32_t *code, int clear);

#ifdef __cplusplus
}
#endif
#endif /* DETFP32_H */
