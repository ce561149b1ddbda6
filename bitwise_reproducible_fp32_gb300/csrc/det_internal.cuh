// det_internal.cuh -- internal declarations and device helpers of libdetfp32.
// Not installed; the public ABI is include/detfp32.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "detfp32.h"

#define DET_API extern "C" __attribute__((visibility("default")))

namespace det {

// ---------------------------------------------------------------- profile v1
constexpr int kKChunk = 256;     // GEMM k-chunk width
constexpr int kRmsLanes = 32;    // chains per RMSNorm row / per mean
constexpr int kXentLanes = 256;  // chains per cross-entropy row
constexpr int kGroup = 4;        // consecutive elements per chain per sweep

// A bounded device wait gives up after this long (the longest legitimate wait
// in the library is one TMA tile, microseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Watchdog bits (det_watchdog_status).
constexpr unsigned int kWatchdogGemm = 1u;   // GEMM operand staging
// bit 1 (2u): cross-entropy row staging, defined in rowops.cu; bit 2 (4u):
// RMSNorm-backward staging (rmsbwd.cu); bit 3 (8u): RMSNorm row staging
// (rowops.cu); bit 4 (16u): causal-softmax row staging (block.cu)

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error; arguments are validated by
// the C-ABI layer before these run.
struct GemmArgs {
    int64_t M, N, K, lda, ldb, ldc;
    const float *A, *B;
    float *C;
    int transA, transB;
    int accumulate = 0;    // C = C + op(A) op(B) (beta = 1)
};
struct GemmPlan {
    int split;             // 1: chunk partials through the workspace
    int units_per_tile;    // chunk groups a tile is cut into
    int kt_per_unit;       // k-tiles a unit computes
    int nchunks;
    int transpose_a;       // 1: op(A) is read from a K x M copy in the workspace
    size_t copy_bytes;     // the copy's share of the workspace (first)
    size_t split_bytes;    // the split partials' share (after the copy)
    size_t workspace_bytes;
    int64_t head_rows;     // > 0: rows [0, head_rows) as an unsplit launch of their
                           // own, the rest as a product with its own plan
    int transpose_b;       // 1: op(B) is read from a K x N copy of B (N x K), first
                           // in the workspace; the rest of the plan follows it
    size_t copy_b_bytes;   // that copy's share of the workspace
};
// a_kmajor: op(A) is k-contiguous (transA == 0), the layout a copy can help;
// b_kmajor: op(B) is k-contiguous (transB != 0), or -1 for a plan that never
// pairs a split with a copy (the two-product plans).
GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sms, bool a_kmajor, int b_kmajor = -1);
// Kernels launch_gemm launches for a with a caller workspace of this size.
int64_t gemm_launches(const GemmArgs &a, size_t workspace_bytes);
cudaError_t launch_gemm(const GemmArgs &a, void *workspace, size_t workspace_bytes,
                        cudaStream_t s);
// Two independent products in one launch where that is faster (else one
// after the other); each product's bits are launch_gemm's.
struct PairPlan {
    int pair;              // 1: one launch for both
    int split;             // both split K (each under its own plan)
    int shared_transpose;  // both read one transposed copy of their common A
    int ctas0, grid;       // the grid's CTAs, the first ctas0 on product 0
    GemmPlan p0, p1;       // each product's plan (the pair's when pair == 1)
    size_t ws0_bytes;      // product 1's partials start here in the workspace
    size_t workspace_bytes;   // the pair's workspace
    size_t separate_bytes;    // the workspace of the two run one after the other
};
PairPlan gemm_pair_plan(const GemmArgs &a0, const GemmArgs &a1, int sms);
cudaError_t launch_gemm_pair(const GemmArgs &a0, const GemmArgs &a1, void *workspace,
                             size_t workspace_bytes, cudaStream_t s);
// A batch of products of one shape. Product z = zb * inner + zh (z < count)
// reads op(A) at A + zb * a_zb + zh * a_zh, op(B) likewise, and writes C at
// C + zb * c_zb + zh * c_zh. The A and B buffers are a_rows x a_cols and
// b_rows x b_cols as stored (row strides lda, ldb), and every product's
// operand lies inside them. causal: only the tiles holding an output with
// j <= i are computed (the rest of C is left unwritten). Never split; the
// bits of each product are detgemm_f32's.
struct GemmBatch {
    int64_t count = 1, inner = 1;
    int64_t a_zb = 0, a_zh = 0, b_zb = 0, b_zh = 0, c_zb = 0, c_zh = 0;
    int64_t a_rows = 0, a_cols = 0, b_rows = 0, b_cols = 0;
    int causal = 0;
    // op(A) triangular with exact +0 outside (1: above the diagonal, 2: below;
    // square products only): whole chunks of those zeros are skipped when
    // *tri_bad == 0 at run time, i.e. when every op(B) value is finite.
    int tri = 0;
    const int *tri_bad = nullptr;
};
// Counts into *bad (atomically) the non-finite values of a rows x cols block
// at base (row stride ld). *bad must be zeroed before.
// +0 in each row's columns from the end of its 256-row block of queries on
// (what launch_softmax_causal with chunk_zeros left unwritten), only when
// *flag (device) is not 0.
cudaError_t launch_zero_past_chunks(int64_t rows, int64_t cols, int64_t period, float *p,
                                   int64_t ld, const int *flag, cudaStream_t s);
cudaError_t launch_count_nonfinite(int64_t rows, int64_t cols, const float *base, int64_t ld,
                                   int *bad, cudaStream_t s);
cudaError_t launch_gemm_batched(const GemmArgs &a, const GemmBatch &bt, cudaStream_t s);
cudaError_t gemm_watchdog(unsigned int *code, int clear);
// T (K x M, row stride ldt) = A^T for A (M x K, row stride lda): data movement
// only, the copy the GEMM takes of a k-contiguous A.
cudaError_t launch_transpose_copy(const float *A, int64_t lda, int64_t M, int64_t K, float *T,
                                  int64_t ldt, cudaStream_t s);
// The same batched products with 64-wide CTA tiles (gemm_n64.cu): for N <= 64
// (a head's width) every warp works on live columns. Same bits.
namespace n64 {
cudaError_t launch_gemm_batched(const GemmArgs &a, const GemmBatch &bt, cudaStream_t s);
cudaError_t gemm_watchdog(unsigned int *code, int clear);
}  // namespace n64
// The same batched products with 128 x 64 CTA tiles (gemm_m128.cu): the
// triangular products of N <= 64 (causal attention's P V, dV, dQ, dK), whose
// row blocks differ in work, in units half as long. Same bits.
namespace m128 {
cudaError_t launch_gemm_batched(const GemmArgs &a, const GemmBatch &bt, cudaStream_t s);
cudaError_t gemm_watchdog(unsigned int *code, int clear);
}  // namespace m128
cudaError_t launch_gemm_noalloc(const GemmArgs &a, bool *too_big, cudaStream_t s);

cudaError_t rowops_watchdog(unsigned int *code, int clear);
cudaError_t rmsbwd_watchdog(unsigned int *code, int clear);
cudaError_t block_watchdog(unsigned int *code, int clear);

// 2-D fp32 TMA descriptor over a row-major matrix: inner = contiguous extent,
// outer = rows, ld = row stride (elements); out-of-range boxes read zeros.
bool make_tensor_map_2d(CUtensorMap *map, const float *base, int64_t inner, int64_t outer,
                        int64_t ld, uint32_t box_inner, uint32_t box_outer, bool swizzle128);
// Whether TMA can describe a matrix at base with row stride ld (16-byte rules).
bool tma_operand_ok(const float *base, int64_t ld);
// x = a + b (dense rows of D), then the RMSNorm of x into y, in one kernel
// (the streamed RMSNorm with a second input); cudaErrorNotSupported when the
// rows do not meet its alignment, and the caller runs the two apart.
cudaError_t launch_add_rmsnorm(int64_t rows, int64_t D, const float *a, const float *b,
                               float *x, int64_t ldx, const float *gain, float eps, float *y,
                               int64_t ldy, float *inv_rms, cudaStream_t s);
cudaError_t launch_rmsnorm(int64_t rows, int64_t D, const float *x, int64_t ldx,
                           const float *gain, float eps, float *y, int64_t ldy,
                           float *inv_rms, cudaStream_t s);
cudaError_t launch_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                        const int32_t *labels, float *loss, float *loss_mean,
                        float *dlogits, int64_t ldd, float dscale,
                        int32_t *dev_status, cudaStream_t s);
size_t rmsnorm_bwd_workspace_bytes(int64_t rows, int64_t D);
cudaError_t launch_rmsnorm_bwd(int64_t rows, int64_t D, const float *x, int64_t ldx,
                               const float *gain, const float *inv_rms, const float *dy,
                               int64_t lddy, float *dx, int64_t lddx, float *dgain,
                               float *workspace, cudaStream_t s);
cudaError_t launch_swiglu(int64_t n, const float *g, const float *u, float *out,
                          cudaStream_t s);
cudaError_t launch_add(int64_t n, const float *a, const float *b, float *out, cudaStream_t s);
// chunk_zeros (device, nullable): when it holds 0, masked columns are zeroed
// only up to the end of each row's 256-row block of queries (the reach of a
// P V that skips the +0 chunks); otherwise, and when null, all of them.
cudaError_t launch_softmax_causal(int64_t rows, int64_t cols, const float *sc, int64_t lds,
                                  float scale, int64_t diag, int64_t period, float *p,
                                  int64_t ldp, cudaStream_t s,
                                  const int *chunk_zeros = nullptr);
cudaError_t launch_rope(int64_t rows, int heads, int head_dim, float *x, int64_t ldx,
                        int64_t seq_len, float theta, int backward, cudaStream_t s);
cudaError_t launch_swiglu_bwd(int64_t n, const float *g, const float *u, const float *dh,
                              float *dg, float *du, cudaStream_t s);
cudaError_t launch_softmax_causal_bwd(int64_t rows, int64_t cols, const float *p,
                                      const float *dp, int64_t ld, float scale, int64_t diag,
                                      int64_t period, float *ds, int64_t ldd, cudaStream_t s);
cudaError_t launch_embedding_bwd(int64_t ntok, int64_t dim, const int32_t *tokens,
                                 const float *dx, int64_t lddx, int64_t vocab, float *de,
                                 int64_t ldde, cudaStream_t s);
cudaError_t launch_embedding(int64_t ntok, int64_t dim, const float *table, int64_t ldt,
                             int64_t vocab, const int32_t *tokens, float *out, int64_t ldo,
                             int32_t *status, cudaStream_t s);
cudaError_t launch_sincos_map(int64_t n, const float *x, float *y, int want_cos,
                              cudaStream_t s);
cudaError_t launch_shardsum(int64_t nshards, int64_t n, const float *shards, int64_t ld,
                            float scale, float *out, cudaStream_t s);
cudaError_t launch_exp_map(int64_t n, const float *x, float *y, int is_log,
                           cudaStream_t s);
cudaError_t launch_adamw(int64_t n, float *p, const float *g, float *m, float *v,
                         const det_adamw_hp &hp, cudaStream_t s);
// Host: bc = 1 - beta^t for both betas (beta^t by t-1 sequential products).
void adamw_bias_correction(int64_t step, float beta1, float beta2, float *bc1, float *bc2);

int sm_count_current_device();

// Launches kern as a programmatic dependent of the work before it on stream s:
// its launch overlaps the tail of the previous kernel, and the kernel must
// call grid_dependency_wait() before it touches global memory.
template <class... KParams, class... Args>
cudaError_t launch_dependent(void (*kern)(KParams...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, KParams(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------- device helpers
// Waits until the grid this kernel was launched as a programmatic dependent of
// has completed and its memory operations are visible; returns at once for a
// plain launch.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next programmatic dependent grid on the stream be launched now:
// its CTAs are placed as resources free up and wait in grid_dependency_wait()
// until this grid has completed. Called after this grid's own wait, so a
// dependent that reads its inputs before waiting (the RMSNorm backward's dx
// kernel) still starts after everything before this grid.
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- Tensor Memory (tcgen05) as per-thread scratch: a warp reaches the 32
// TMEM lanes of its quarter (warp % 4), a thread its own lane; an address
// holds the lane in its high 16 bits and the column in its low 16 bits.
// One warp allocates ncols columns (a power of two, 32..512) for the CTA and
// writes their base address to shared memory at smem_dst. The caller keeps
// the columns that the CTAs resident on an SM ask for within the SM's 512,
// so the allocation never waits.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_dst), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// The allocating warp frees them, after a CTA barrier between the two fences
// below has ordered every access before it (each access returns complete).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive 32-bit columns of the thread's lane, from / to registers
// (warp-wide: every lane of the warp takes part). Each returns once the copy
// is complete: the wait sits in the same asm statement, so the compiler can
// neither read the loaded registers nor reuse the stored ones earlier.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%0, %1, %2, %3, %4, %5, %6, %7,"
                 "%8, %9, %10, %11, %12, %13, %14, %15,"
                 "%16, %17, %18, %19, %20, %21, %22, %23,"
                 "%24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
                   "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
                   "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
                   "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
                 "%1, %2, %3, %4, %5, %6, %7, %8,"
                 "%9, %10, %11, %12, %13, %14, %15, %16,"
                 "%17, %18, %19, %20, %21, %22, %23, %24,"
                 "%25, %26, %27, %28, %29, %30, %31, %32};\n\t"
                 "tcgen05.wait::st.sync.aligned;"
                 :: "r"(taddr),
                   "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                   "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
                   "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
                   "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                   "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
                   "r"(v[30]), "r"(v[31])
                 : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same phase (test_wait never suspends the thread;
// try_wait may, for a system-dependent time).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete, giving up after
// kWaitLimitNs. Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// As mbar_wait_bounded, but also gives up as soon as *abort is set, and sets
// *abort itself when the time limit passes, so every waiter of the CTA stops.
// A limit of 0 gives up whenever the phase is not complete at the first,
// non-blocking look.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int *abort,
                                                   unsigned long long limit_ns = kWaitLimitNs) {
    if (limit_ns == 0) {
        if (mbar_test_wait(bar, parity)) return true;
        *abort = 1;
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}

// 2-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Packed FP32 pairs (sm_100+ add/sub/mul/fma .rn.f32x2): each half is rounded
// exactly as the scalar operation (round to nearest even, no flush), so two
// independent scalar chains can share one instruction without changing a bit
// -- except that a packed multiply must not feed a packed add or subtract: that
// pair was measured to round as if fused.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 splat2(float v) { return pack2(v, v); }

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

}  // namespace det
