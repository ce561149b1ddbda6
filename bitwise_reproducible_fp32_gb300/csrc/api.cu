// api.cu -- the C ABI of libdetfp32 (declared in include/detfp32.h).
//
// Every entry point checks the profile, the device and its arguments on the
// host, then launches on the caller's stream and returns without
// synchronising. A profile the library does not implement is refused by name
// (DET_ERR_PROFILE), never run as something close: the "mojolearn" PyPI page,
// section "Which families offer which tiers", asks for a named error rather
// than a weaker result.
#include <algorithm>
#include <atomic>
#include <vector>

#include "det_internal.cuh"

namespace det {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];       // 0: unknown
std::atomic<int> g_device_ok[kMaxDevices];      // 0 unknown, 1 ok, 2 refused

det_status check_profile(const det_profile_v1 *p) {
    if (!p) return DET_ERR_INVALID_ARG;
    if (p->version != DET_PROFILE_VERSION || p->k_chunk != uint32_t(kKChunk) ||
        p->rms_lanes != uint32_t(kRmsLanes) || p->xent_lanes != uint32_t(kXentLanes) ||
        p->lane_group != uint32_t(kGroup) || p->flags != 0)
        return DET_ERR_PROFILE;
    return DET_OK;
}

det_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DET_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DET_ERR_UNSUPPORTED_DEVICE;
    int st = g_device_ok[dev].load(std::memory_order_relaxed);
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DET_ERR_CUDA;
        g_sm_count[dev].store(sms, std::memory_order_relaxed);
        st = (major == 10 && minor == 3) ? 1 : 2;
        g_device_ok[dev].store(st, std::memory_order_relaxed);
    }
    return st == 1 ? DET_OK : DET_ERR_UNSUPPORTED_DEVICE;
}

det_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DET_OK : DET_ERR_CUDA; }

constexpr int64_t kDimMax = 0x7fffffff;   // dimensions below 2^31

// An AdamW decay rate in [0, 1] (NaN fails).
bool beta_ok(float b) { return b >= 0.0f && b <= 1.0f; }
}  // namespace

int sm_count_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        const int n = g_sm_count[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            sms > 0) {
            g_sm_count[dev].store(sms, std::memory_order_relaxed);
            return sms;
        }
    }
    return 152;
}

}  // namespace det

using namespace det;

DET_API void det_profile_default(det_profile_v1 *p) {
    if (!p) return;
    p->version = DET_PROFILE_VERSION;
    p->k_chunk = kKChunk;
    p->rms_lanes = kRmsLanes;
    p->xent_lanes = kXentLanes;
    p->lane_group = kGroup;
    p->flags = 0;
}

DET_API const char *det_status_string(int status) {
    switch (status) {
        case DET_OK: return "DET_OK";
        case DET_ERR_INVALID_ARG: return "DET_ERR_INVALID_ARG: invalid argument";
        case DET_ERR_PROFILE: return "DET_ERR_PROFILE: numerical profile not implemented";
        case DET_ERR_UNSUPPORTED_DEVICE:
            return "DET_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
        case DET_ERR_ALIGNMENT: return "DET_ERR_ALIGNMENT: misaligned buffer";
        case DET_ERR_WORKSPACE: return "DET_ERR_WORKSPACE: workspace too small";
        case DET_ERR_TIMEOUT: return "DET_ERR_TIMEOUT: a bounded device wait gave up";
        case DET_ERR_CUDA: return "DET_ERR_CUDA: CUDA runtime error";
        default: return "unknown det_status";
    }
}

DET_API det_status detgemm_workspace_bytes(const det_profile_v1 *prof, int transA,
                                           int transB, int64_t M, int64_t N, int64_t K,
                                           size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || M < 0 || N < 0 || K < 0 || M > kDimMax || N > kDimMax || K > kDimMax)
        return DET_ERR_INVALID_ARG;
    *bytes = 0;
    if (M == 0 || N == 0 || K == 0) return DET_OK;
    if ((st = check_device()) != DET_OK) return st;
    *bytes = gemm_plan(M, N, K, sm_count_current_device(), transA == 0, transB != 0 ? 1 : 0)
                 .workspace_bytes;
    return DET_OK;
}

DET_API det_status detgemm_launches(const det_profile_v1 *prof, int transA, int transB,
                                    int64_t M, int64_t N, int64_t K, size_t workspace_bytes,
                                    int64_t *launches) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!launches || M < 0 || N < 0 || K < 0 || M > kDimMax || N > kDimMax || K > kDimMax)
        return DET_ERR_INVALID_ARG;
    *launches = 0;
    if (M == 0 || N == 0) return DET_OK;
    if ((st = check_device()) != DET_OK) return st;
    GemmArgs a;
    a.M = M; a.N = N; a.K = K;
    a.transA = transA != 0; a.transB = transB != 0;
    *launches = gemm_launches(a, workspace_bytes);
    return DET_OK;
}

namespace {
det_status gemm_entry(const det_profile_v1 *prof, int transA, int transB, int64_t M,
                      int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                      int64_t ldb, float *C, int64_t ldc, void *workspace,
                      size_t workspace_bytes, det_stream_t stream, int accumulate) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (M < 0 || N < 0 || K < 0 || M > kDimMax || N > kDimMax || K > kDimMax)
        return DET_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DET_OK;
    const int64_t a_row = transA ? M : K, b_row = transB ? K : N;
    if (ldc < N || lda < std::max<int64_t>(a_row, 1) || ldb < std::max<int64_t>(b_row, 1))
        return DET_ERR_INVALID_ARG;
    if (!C || (K > 0 && (!A || !B))) return DET_ERR_INVALID_ARG;
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    if (tiles > kDimMax) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    GemmArgs a;
    a.M = M; a.N = N; a.K = K; a.lda = lda; a.ldb = ldb; a.ldc = ldc;
    a.A = A; a.B = B; a.C = C; a.transA = transA != 0; a.transB = transB != 0;
    a.accumulate = accumulate;
    return from_cuda(launch_gemm(a, workspace, workspace_bytes,
                                 reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

DET_API det_status detgemm_f32(const det_profile_v1 *prof, int transA, int transB,
                               int64_t M, int64_t N, int64_t K, const float *A,
                               int64_t lda, const float *B, int64_t ldb, float *C,
                               int64_t ldc, void *workspace, size_t workspace_bytes,
                               det_stream_t stream) {
    return gemm_entry(prof, transA, transB, M, N, K, A, lda, B, ldb, C, ldc, workspace,
                      workspace_bytes, stream, 0);
}

DET_API det_status detgemm_acc_f32(const det_profile_v1 *prof, int transA, int transB,
                                   int64_t M, int64_t N, int64_t K, const float *A,
                                   int64_t lda, const float *B, int64_t ldb, float *C,
                                   int64_t ldc, void *workspace, size_t workspace_bytes,
                                   det_stream_t stream) {
    return gemm_entry(prof, transA, transB, M, N, K, A, lda, B, ldb, C, ldc, workspace,
                      workspace_bytes, stream, 1);
}

// ---------------------------------------------------------------- groups of products
namespace {
// A problem's arguments as GemmArgs, after detgemm_f32's checks. Returns
// DET_OK with *empty set when the product has no outputs.
det_status check_problem(const det_gemm_problem &q, GemmArgs *a, bool *empty) {
    *empty = false;
    if (q.M < 0 || q.N < 0 || q.K < 0 || q.M > kDimMax || q.N > kDimMax || q.K > kDimMax)
        return DET_ERR_INVALID_ARG;
    if (q.M == 0 || q.N == 0) {
        *empty = true;
        return DET_OK;
    }
    const int64_t a_row = q.transA ? q.M : q.K, b_row = q.transB ? q.K : q.N;
    if (q.ldc < q.N || q.lda < std::max<int64_t>(a_row, 1) ||
        q.ldb < std::max<int64_t>(b_row, 1))
        return DET_ERR_INVALID_ARG;
    if (!q.C || (q.K > 0 && (!q.A || !q.B))) return DET_ERR_INVALID_ARG;
    const int64_t tiles = ((q.M + 127) / 128) * ((q.N + 127) / 128);
    if (tiles > kDimMax) return DET_ERR_INVALID_ARG;
    a->M = q.M; a->N = q.N; a->K = q.K; a->lda = q.lda; a->ldb = q.ldb; a->ldc = q.ldc;
    a->A = q.A; a->B = q.B; a->C = q.C;
    a->transA = q.transA != 0; a->transB = q.transB != 0;
    a->accumulate = 0;
    return DET_OK;
}

// Runs fn(first, second-or-null) over the problems in pairs (0, 1), (2, 3), ...
// after checking every problem; empty products are dropped from the pairing.
template <class Fn>
det_status for_pairs(const det_profile_v1 *prof, int64_t count,
                     const det_gemm_problem *probs, Fn fn) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (count < 0 || (count > 0 && !probs)) return DET_ERR_INVALID_ARG;
    std::vector<GemmArgs> live;
    for (int64_t i = 0; i < count; ++i) {
        GemmArgs a;
        bool empty = false;
        if ((st = check_problem(probs[i], &a, &empty)) != DET_OK) return st;
        if (!empty) live.push_back(a);
    }
    if (live.empty()) return DET_OK;
    if ((st = check_device()) != DET_OK) return st;
    for (size_t i = 0; i < live.size(); i += 2) {
        const GemmArgs *second = i + 1 < live.size() ? &live[i + 1] : nullptr;
        if ((st = fn(live[i], second)) != DET_OK) return st;
    }
    return DET_OK;
}
}  // namespace

DET_API det_status detgemm_group_workspace_bytes(const det_profile_v1 *prof, int64_t count,
                                                 const det_gemm_problem *problems,
                                                 size_t *bytes) {
    if (!bytes) return DET_ERR_INVALID_ARG;
    size_t need = 0;
    const det_status st = for_pairs(prof, count, problems,
                                    [&](const GemmArgs &a, const GemmArgs *b) {
        const int sms = sm_count_current_device();
        if (!b) {
            need = std::max(need, gemm_plan(a.M, a.N, a.K, sms, !a.transA, a.transB ? 1 : 0)
                                      .workspace_bytes);
        } else {
            const PairPlan pp = gemm_pair_plan(a, *b, sms);
            need = std::max(need, pp.pair ? pp.workspace_bytes : pp.separate_bytes);
        }
        return DET_OK;
    });
    if (st == DET_OK) *bytes = need;
    return st;
}

DET_API det_status detgemm_group_launches(const det_profile_v1 *prof, int64_t count,
                                          const det_gemm_problem *problems,
                                          size_t workspace_bytes, int64_t *launches) {
    if (!launches) return DET_ERR_INVALID_ARG;
    int64_t n = 0;
    const int sms = sm_count_current_device();
    // kernels one product issues alone with this much workspace
    auto alone = [&](const GemmArgs &a) -> int64_t { return gemm_launches(a, workspace_bytes); };
    const det_status st = for_pairs(prof, count, problems,
                                    [&](const GemmArgs &a, const GemmArgs *b) {
        if (!b) {
            n += alone(a);
            return DET_OK;
        }
        const PairPlan pp = gemm_pair_plan(a, *b, sms);
        if (pp.pair && workspace_bytes >= pp.workspace_bytes)
            n += pp.shared_transpose ? 2 : pp.split ? 3 : 1;
        else
            n += alone(a) + alone(*b);
        return DET_OK;
    });
    if (st == DET_OK) *launches = n;
    return st;
}

DET_API det_status detgemm_group_f32(const det_profile_v1 *prof, int64_t count,
                                     const det_gemm_problem *problems, void *workspace,
                                     size_t workspace_bytes, det_stream_t stream) {
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return for_pairs(prof, count, problems, [&](const GemmArgs &a, const GemmArgs *b) {
        return from_cuda(b ? launch_gemm_pair(a, *b, workspace, workspace_bytes, s)
                           : launch_gemm(a, workspace, workspace_bytes, s));
    });
}

// ---------------------------------------------------------------- block forward
namespace {
bool overlaps(const float *a, int64_t na, const float *b, int64_t nb) {
    return a < b + nb && b < a + na;
}
}  // namespace

DET_API det_status detswiglu_f32(const det_profile_v1 *prof, int64_t n, const float *gate,
                                 const float *up, float *out, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!gate || !up || !out) return DET_ERR_INVALID_ARG;
    if ((out != gate && overlaps(out, n, gate, n)) || (out != up && overlaps(out, n, up, n)))
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_swiglu(n, gate, up, out, reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detadd_f32(const det_profile_v1 *prof, int64_t n, const float *a,
                              const float *b, float *out, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!a || !b || !out) return DET_ERR_INVALID_ARG;
    if ((out != a && overlaps(out, n, a, n)) || (out != b && overlaps(out, n, b, n)))
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_add(n, a, b, out, reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detsoftmax_causal_f32(const det_profile_v1 *prof, int64_t rows,
                                         int64_t cols, const float *scores, int64_t lds,
                                         float scale, int64_t diag, int64_t period, float *p,
                                         int64_t ldp, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || cols < 1 || cols > kDimMax || period < 1) return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (lds < cols || ldp < cols || !scores || !p) return DET_ERR_INVALID_ARG;
    if (p == scores && ldp != lds) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_softmax_causal(rows, cols, scores, lds, scale, diag, period, p, ldp,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detrope_f32(const det_profile_v1 *prof, int64_t rows, int64_t heads,
                               int64_t head_dim, float *x, int64_t ldx, int64_t seq_len,
                               float theta, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || heads < 1 || head_dim < 2 || head_dim % 2 || head_dim > 65536 ||
        heads > 65536 || seq_len < 1)
        return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (!x || ldx < heads * head_dim) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_rope(rows, int(heads), int(head_dim), x, ldx, seq_len, theta, 0,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detrope_bwd_f32(const det_profile_v1 *prof, int64_t rows, int64_t heads,
                                   int64_t head_dim, float *dx, int64_t ldx, int64_t seq_len,
                                   float theta, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || heads < 1 || head_dim < 2 || head_dim % 2 || head_dim > 65536 ||
        heads > 65536 || seq_len < 1)
        return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (!dx || ldx < heads * head_dim) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_rope(rows, int(heads), int(head_dim), dx, ldx, seq_len, theta, 1,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detswiglu_bwd_f32(const det_profile_v1 *prof, int64_t n, const float *gate,
                                     const float *up, const float *dh, float *d_gate,
                                     float *d_up, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!gate || !up || !dh || !d_gate || !d_up) return DET_ERR_INVALID_ARG;
    // the outputs may overwrite dh, element for element, but nothing else
    for (const float *in : {gate, up})
        for (const float *o : {static_cast<const float *>(d_gate), static_cast<const float *>(d_up)})
            if (overlaps(o, n, in, n)) return DET_ERR_INVALID_ARG;
    if (overlaps(d_gate, n, d_up, n)) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_swiglu_bwd(n, gate, up, dh, d_gate, d_up,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detsoftmax_causal_bwd_f32(const det_profile_v1 *prof, int64_t rows,
                                             int64_t cols, const float *p, const float *dp,
                                             int64_t ld, float scale, int64_t diag,
                                             int64_t period, float *ds, int64_t ldd,
                                             det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || cols < 1 || cols > kDimMax || period < 1) return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (ld < cols || ldd < cols || !p || !dp || !ds) return DET_ERR_INVALID_ARG;
    if ((ds == dp || ds == p) && ldd != ld) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_softmax_causal_bwd(rows, cols, p, dp, ld, scale, diag, period, ds,
                                               ldd, reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detembedding_bwd_f32(const det_profile_v1 *prof, int64_t ntok, int64_t dim,
                                        const int32_t *tokens, const float *dx, int64_t lddx,
                                        int64_t vocab, float *de, int64_t ldde,
                                        det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (ntok < 0 || dim < 1 || dim > kDimMax || vocab < 1 || vocab > kDimMax)
        return DET_ERR_INVALID_ARG;
    if (!de || ldde < dim || (ntok > 0 && (!tokens || !dx || lddx < dim)))
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_embedding_bwd(ntok, dim, tokens, dx, lddx, vocab, de, ldde,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detembedding_f32(const det_profile_v1 *prof, int64_t ntok, int64_t dim,
                                    const float *table, int64_t ldt, int64_t vocab,
                                    const int32_t *tokens, float *out, int64_t ldo,
                                    int32_t *dev_status, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (ntok < 0 || dim < 1 || dim > kDimMax || vocab < 1 || vocab > kDimMax)
        return DET_ERR_INVALID_ARG;
    if (ntok == 0) return DET_OK;
    if (!table || !tokens || !out || ldt < dim || ldo < dim) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_embedding(ntok, dim, table, ldt, vocab, tokens, out, ldo, dev_status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detsin_f32(const det_profile_v1 *prof, int64_t n, const float *x, float *y,
                              det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!x || !y) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_sincos_map(n, x, y, 0, reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detcos_f32(const det_profile_v1 *prof, int64_t n, const float *x, float *y,
                              det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!x || !y) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_sincos_map(n, x, y, 1, reinterpret_cast<cudaStream_t>(stream)));
}

// Causal attention over one packed QKV activation, a group of heads at a time:
// S = Q_z K_z^T (profile GEMM) for every head z of the group in one batched
// launch, skipping the score tiles above the diagonal that the softmax masks;
// P = the causal softmax of S * scale over all the group's rows in one launch;
// O_z = P_z V_z (profile GEMM) in one batched launch. Each head's bits are
// those of its separate products.
namespace {
// Heads go in groups whose score buffers together stay within 1 GiB: whole
// sequences (all heads of gb sequences) when one sequence fits, else gh heads
// of one sequence; groups are balanced in size.
constexpr size_t kAttnScoreCap = size_t(1) << 30;
constexpr size_t kAttnFlagBytes = 256;   // the non-finite counts, after the score buffers
struct AttnGroups {
    int64_t gb, gh;       // sequences and heads a group spans (gb > 1 only when gh == heads)
    size_t score_bytes;   // one score buffer of the largest group, 256-byte rounded
};
AttnGroups attention_groups(int64_t batch, int64_t seq, int64_t heads) {
    const size_t per_head = size_t(seq) * size_t(seq) * 4;
    AttnGroups g{};
    if (size_t(heads) * per_head <= kAttnScoreCap) {
        // (at most 2^20 products a group, so the launch's unit count fits an int)
        const int64_t fit = std::max<int64_t>(
            1, std::min<int64_t>(int64_t(kAttnScoreCap / (size_t(heads) * per_head)),
                                 (int64_t(1) << 20) / heads));
        const int64_t ngroups = (std::max<int64_t>(batch, 1) + fit - 1) / fit;
        g.gb = (std::max<int64_t>(batch, 1) + ngroups - 1) / ngroups;
        g.gh = heads;
    } else {
        const int64_t fit = std::max<int64_t>(1, int64_t(kAttnScoreCap / per_head));
        const int64_t ngroups = (heads + fit - 1) / fit;
        g.gb = 1;
        g.gh = (heads + ngroups - 1) / ngroups;
    }
    g.score_bytes = (size_t(g.gb * g.gh) * per_head + 255) / 256 * 256;
    return g;
}

// Walks the groups: f(b0, nb, h0, nh) for sequences b0 .. b0+nb-1 and heads
// h0 .. h0+nh-1; stops at the first error.
template <typename F>
cudaError_t for_each_group(int64_t batch, int64_t heads, const AttnGroups &g, F f) {
    for (int64_t b0 = 0; b0 < batch; b0 += g.gb)
        for (int64_t h0 = 0; h0 < heads; h0 += g.gh) {
            const cudaError_t e = f(b0, std::min(g.gb, batch - b0), h0, std::min(g.gh, heads - h0));
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

// One operand of the heads of a group inside a packed [batch * seq, ld]
// buffer: the group's first head at column col0, sequence stride seq * ld,
// head stride head_dim; the map spans the rest of the buffer.
struct HeadOperand {
    const float *base;
    int64_t ld, rows, cols, zb, zh;
};
HeadOperand head_operand(const float *buf, int64_t ld, int64_t width, int64_t batch,
                         int64_t seq, int64_t b0, int64_t col0, int64_t head_dim) {
    HeadOperand o;
    o.base = buf + b0 * seq * ld + col0;
    o.ld = ld;
    o.rows = (batch - b0) * seq;
    o.cols = width - col0;
    o.zb = seq * ld;
    o.zh = head_dim;
    return o;
}

// One batched profile GEMM over the products of a group: op(A) from a, op(B)
// from b, C at c (base pointer, ldc, per-product strides).
cudaError_t group_gemm(int64_t M, int64_t N, int64_t K, const HeadOperand &a, int tA,
                       const HeadOperand &b, int tB, float *c, int64_t ldc, int64_t c_zb,
                       int64_t c_zh, int64_t count, int64_t inner, int causal,
                       cudaStream_t s, int tri = 0, const int *tri_bad = nullptr) {
    GemmArgs g;
    g.M = M; g.N = N; g.K = K;
    g.A = a.base; g.lda = a.ld; g.B = b.base; g.ldb = b.ld; g.C = c; g.ldc = ldc;
    g.transA = tA; g.transB = tB;
    GemmBatch bt;
    bt.count = count; bt.inner = inner;
    bt.a_zb = a.zb; bt.a_zh = a.zh; bt.b_zb = b.zb; bt.b_zh = b.zh;
    bt.c_zb = c_zb; bt.c_zh = c_zh;
    bt.a_rows = a.rows; bt.a_cols = a.cols; bt.b_rows = b.rows; bt.b_cols = b.cols;
    bt.causal = causal;
    bt.tri = tri;
    bt.tri_bad = tri_bad;
    // a head-wide N (P V, dV, dQ, dK) fills the 64-wide tiles; the triangular
    // ones take 128-row tiles, whose shorter units balance the CTAs' loads
    if (N <= 64 && tri) return m128::launch_gemm_batched(g, bt, s);
    if (N <= 64) return n64::launch_gemm_batched(g, bt, s);
    return launch_gemm_batched(g, bt, s);
}

// The group's stacked seq x seq buffers (product z at rows z * seq) as an
// operand.
HeadOperand stacked(const float *buf, int64_t seq, int64_t nh, int64_t count) {
    HeadOperand o;
    o.base = buf;
    o.ld = seq;
    o.rows = count * seq;
    o.cols = seq;
    o.zb = nh * seq * seq;
    o.zh = seq * seq;
    return o;
}

// Zeroes the n flag words, then counts each listed operand's non-finite
// values into its word (the triangular skips of the products that read it
// are taken only when the count is 0).
cudaError_t count_nonfinite_heads(int *flags, const HeadOperand *ops, int n, int64_t rows,
                                  int64_t cols, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(int) * n, s);
    for (int i = 0; i < n && e == cudaSuccess; ++i)
        e = launch_count_nonfinite(rows, cols, ops[i].base, ops[i].ld, flags + i, s);
    return e;
}

// The score products (S = Q K^T, and the backward's dP = dO V^T) read both
// operands k-contiguous, where the GEMM runs its scalar FFMA loop. Reading the
// left one from a transposed copy of its whole block (heads * head_dim rows of
// batch * seq tokens, m-contiguous) and the right one from a copy of its own
// (n-contiguous) the GEMM runs the row-pair loop with direct 16-byte stores,
// with the same bits. A copy (one launch for the forward's Q and K, one a
// block in the backward; 8 bytes an element) pays for itself once the
// sequences are long.
constexpr int64_t kAttnQCopyMinSeq = 512;
int64_t attn_qt_ld(int64_t batch, int64_t seq) { return (batch * seq + 3) / 4 * 4; }
// one block's copy
size_t attn_qt_bytes(int64_t batch, int64_t seq, int64_t heads, int64_t head_dim) {
    if (seq < kAttnQCopyMinSeq) return 0;
    return (size_t(heads * head_dim) * size_t(attn_qt_ld(batch, seq)) * 4 + 255) / 256 * 256;
}
// the forward's copy of the Q and K blocks (2 heads * head_dim rows)
size_t attn_qkt_bytes(int64_t batch, int64_t seq, int64_t heads, int64_t head_dim) {
    if (seq < kAttnQCopyMinSeq) return 0;
    return (size_t(2 * heads * head_dim) * size_t(attn_qt_ld(batch, seq)) * 4 + 255) / 256 *
           256;
}
// The heads h0.. of sequences b0.. of a block copied transposed into QT (row =
// head_dim index, column = token): op(A) of a score product (m-contiguous), or
// its op(B) (n-contiguous)
HeadOperand q_from_copy(const float *QT, int64_t ldt, int64_t batch, int64_t seq, int64_t hd,
                        int64_t b0, int64_t h0, int64_t head_dim) {
    HeadOperand o;
    o.base = QT + h0 * head_dim * ldt + b0 * seq;
    o.ld = ldt;
    o.rows = hd - h0 * head_dim;
    o.cols = (batch - b0) * seq;
    o.zb = seq;
    o.zh = head_dim * ldt;
    return o;
}

bool attention_args_ok(int64_t batch, int64_t seq, int64_t heads, int64_t head_dim) {
    return batch >= 0 && seq >= 1 && seq <= 65536 && heads >= 1 && heads <= 65536 &&
           head_dim >= 1 && head_dim <= 65536 && batch <= kDimMax / seq &&
           heads * head_dim <= kDimMax / 3;
}
}  // namespace

DET_API det_status detattention_workspace_bytes(const det_profile_v1 *prof, int64_t batch,
                                                int64_t seq, int64_t heads, int64_t head_dim,
                                                size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || !attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    *bytes = attention_groups(batch, seq, heads).score_bytes + kAttnFlagBytes +
             attn_qkt_bytes(batch, seq, heads, head_dim);
    return DET_OK;
}

DET_API det_status detattention_launches(const det_profile_v1 *prof, int64_t batch,
                                         int64_t seq, int64_t heads, int64_t head_dim,
                                         int backward, int64_t *launches) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!launches || !attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    if (batch == 0) {
        *launches = 0;
        return DET_OK;
    }
    const AttnGroups g = attention_groups(batch, seq, heads);
    const int64_t groups = ((batch + g.gb - 1) / g.gb) * ((heads + g.gh - 1) / g.gh);
    // forward: the Q and K copy (long sequences), then a group's score
    // product, the count of V's non-finite values, the softmax and P V;
    // backward: the Q, dO and V copies (long sequences), then S, the softmax,
    // dP, the counts of dO's, K's and Q's non-finite values, dV, the softmax
    // backward, dQ and dK
    const int64_t copies = attn_qt_bytes(batch, seq, heads, head_dim) ? 1 : 0;
    if (backward == 2 && groups == 1) {
        // detattention_bwd_saved_f32 with the forward's P: the dO and V
        // copies, the counts, the +0 fill past the chunks (when dO is not
        // finite), dP, dV, the softmax backward, dQ and dK
        *launches = 9 + 2 * copies;
        return DET_OK;
    }
    *launches = backward ? 10 * groups + 3 * copies : 4 * groups + copies;
    return DET_OK;
}

DET_API det_status detattention_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                    int64_t heads, int64_t head_dim, const float *qkv,
                                    int64_t ldqkv, float scale, float *out, int64_t ldout,
                                    void *workspace, size_t workspace_bytes,
                                    det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    if (batch == 0) return DET_OK;
    const int64_t hd = heads * head_dim;
    if (!qkv || !out || ldqkv < 3 * hd || ldout < hd) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    const AttnGroups g = attention_groups(batch, seq, heads);
    const size_t qt_bytes = attn_qkt_bytes(batch, seq, heads, head_dim);
    if (!workspace || workspace_bytes < g.score_bytes + kAttnFlagBytes + qt_bytes ||
        reinterpret_cast<uintptr_t>(workspace) % 256)
        return DET_ERR_WORKSPACE;
    float *S = static_cast<float *>(workspace);
    int *flags = reinterpret_cast<int *>(static_cast<char *>(workspace) + g.score_bytes);
    float *QT = qt_bytes ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                     g.score_bytes + kAttnFlagBytes)
                         : nullptr;
    const int64_t ldt = attn_qt_ld(batch, seq);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto group = [&](int64_t b0, int64_t nb, int64_t h0, int64_t nh) {
        const int64_t count = nb * nh;
        // Q and K from the copy (rows 0.. and hd..), or in place
        const HeadOperand Q =
            QT ? q_from_copy(QT, ldt, batch, seq, hd, b0, h0, head_dim)
               : head_operand(qkv, ldqkv, 3 * hd, batch, seq, b0, h0 * head_dim, head_dim);
        const HeadOperand K =
            QT ? q_from_copy(QT + hd * ldt, ldt, batch, seq, hd, b0, h0, head_dim)
               : head_operand(qkv, ldqkv, 3 * hd, batch, seq, b0, hd + h0 * head_dim, head_dim);
        const HeadOperand V = head_operand(qkv, ldqkv, 3 * hd, batch, seq, b0, 2 * hd + h0 * head_dim, head_dim);
        const HeadOperand P = stacked(S, seq, nh, count);
        cudaError_t r = group_gemm(seq, seq, head_dim, Q, QT ? 1 : 0, K, QT ? 0 : 1, S, seq, P.zb,
                                   P.zh, count, nh, 1, s);
        // P is +0 above the diagonal: with a finite V (counted first) P V
        // skips the chunks past each row block, so the softmax writes P's +0
        // columns only up to that block's end
        if (r == cudaSuccess) r = count_nonfinite_heads(flags, &V, 1, nb * seq, nh * head_dim, s);
        if (r == cudaSuccess)
            r = launch_softmax_causal(count * seq, seq, S, seq, scale, 0, seq, S, seq, s, flags);
        if (r == cudaSuccess)
            r = group_gemm(seq, head_dim, seq, P, 0, V, 0, out + b0 * seq * ldout + h0 * head_dim,
                           ldout, seq * ldout, head_dim, count, nh, 0, s, 1, flags);
        return r;
    };
    cudaError_t e = QT ? launch_transpose_copy(qkv, ldqkv, batch * seq, 2 * hd, QT, ldt, s)
                       : cudaSuccess;
    if (e == cudaSuccess) e = for_each_group(batch, heads, g, group);
    return from_cuda(e);
}

// Backward of detattention_f32, a group of heads at a time: P is recomputed
// by the forward's spelling (S = Q K^T, the causal softmax), then
//   dP = dO V^T, dV = P^T dO, dS = the softmax backward of (P, dP),
//   dQ = dS K, dK = dS^T Q
// each one batched launch over the group, with detgemm_f32's arithmetic for
// every product (the score products skip the tiles the softmax masks). The
// gradients are those of the Q, K and V that the forward read (after any
// rotary embedding).
DET_API det_status detattention_bwd_workspace_bytes(const det_profile_v1 *prof, int64_t batch,
                                                    int64_t seq, int64_t heads,
                                                    int64_t head_dim, size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || !attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    *bytes = 2 * attention_groups(batch, seq, heads).score_bytes + kAttnFlagBytes +
             3 * attn_qt_bytes(batch, seq, heads, head_dim);
    return DET_OK;
}

namespace {
// The backward of detattention_f32 (detattention_bwd_f32's operation); with
// Psaved (the forward's workspace, all heads in one group) P is read from it
// instead of recomputed.
det_status attention_bwd(const det_profile_v1 *prof, int64_t batch, int64_t seq, int64_t heads,
                         int64_t head_dim, const float *qkv, int64_t ldqkv, const float *dout,
                         int64_t lddout, float scale, float *Psaved, float *dqkv,
                         int64_t lddqkv, void *workspace, size_t workspace_bytes,
                         det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    if (batch == 0) return DET_OK;
    const int64_t hd = heads * head_dim;
    if (!qkv || !dout || !dqkv || ldqkv < 3 * hd || lddout < hd || lddqkv < 3 * hd)
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    const AttnGroups g = attention_groups(batch, seq, heads);
    const size_t qt_bytes = attn_qt_bytes(batch, seq, heads, head_dim);
    if (!workspace ||
        workspace_bytes < 2 * g.score_bytes + kAttnFlagBytes + 3 * qt_bytes ||
        reinterpret_cast<uintptr_t>(workspace) % 256)
        return DET_ERR_WORKSPACE;
    // the forward's P covers every head only when they ran as one group
    const bool saved = Psaved != nullptr && g.gb >= batch && g.gh >= heads;
    float *Pb = saved ? Psaved : static_cast<float *>(workspace);
    float *dPb = reinterpret_cast<float *>(static_cast<char *>(workspace) + g.score_bytes);
    int *flags = reinterpret_cast<int *>(static_cast<char *>(workspace) + 2 * g.score_bytes);
    // long sequences: the score products read Q and dO from transposed copies
    // (the row-pair loop, as in the forward), with the same bits
    float *QT = qt_bytes ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                     2 * g.score_bytes + kAttnFlagBytes)
                         : nullptr;
    float *dOT = qt_bytes ? reinterpret_cast<float *>(reinterpret_cast<char *>(QT) + qt_bytes)
                          : nullptr;
    float *VT = qt_bytes ? reinterpret_cast<float *>(reinterpret_cast<char *>(dOT) + qt_bytes)
                         : nullptr;
    const int64_t ldt = attn_qt_ld(batch, seq);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (QT) {
        if (!saved) e = launch_transpose_copy(qkv, ldqkv, batch * seq, hd, QT, ldt, s);
        if (e == cudaSuccess) e = launch_transpose_copy(dout, lddout, batch * seq, hd, dOT, ldt, s);
        if (e == cudaSuccess)
            e = launch_transpose_copy(qkv + 2 * hd, ldqkv, batch * seq, hd, VT, ldt, s);
    }
    if (e == cudaSuccess) e = for_each_group(batch, heads, g, [&](int64_t b0, int64_t nb,
                                                                  int64_t h0, int64_t nh) {
        const int64_t count = nb * nh;
        auto in = [&](const float *buf, int64_t ld, int64_t width, int64_t col) {
            return head_operand(buf, ld, width, batch, seq, b0, col + h0 * head_dim, head_dim);
        };
        const HeadOperand Q = in(qkv, ldqkv, 3 * hd, 0), K = in(qkv, ldqkv, 3 * hd, hd);
        const HeadOperand V = in(qkv, ldqkv, 3 * hd, 2 * hd), dO = in(dout, lddout, hd, 0);
        const HeadOperand P = stacked(Pb, seq, nh, count), dP = stacked(dPb, seq, nh, count);
        const HeadOperand Qs = QT ? q_from_copy(QT, ldt, batch, seq, hd, b0, h0, head_dim) : Q;
        const HeadOperand dOs =
            dOT ? q_from_copy(dOT, ldt, batch, seq, hd, b0, h0, head_dim) : dO;
        const HeadOperand Vs = VT ? q_from_copy(VT, ldt, batch, seq, hd, b0, h0, head_dim) : V;
        float *dbase = dqkv + b0 * seq * lddqkv + h0 * head_dim;
        const int64_t dzb = seq * lddqkv;
        // P and dS are +0 above the diagonal, so P^T and dS^T below it: with
        // finite dO, K and Q (flags 0, 1, 2) the chunks there are skipped
        const HeadOperand finite[3] = {dO, K, Q};
        cudaError_t r = cudaSuccess;
        if (saved) {
            // the forward wrote P's +0 columns up to the end of each row's
            // 256-row block (when its V was finite); dV reads past that only
            // when dO is not finite, and then this fills the rest with +0
            r = count_nonfinite_heads(flags, finite, 3, nb * seq, nh * head_dim, s);
            if (r == cudaSuccess)
                r = launch_zero_past_chunks(count * seq, seq, seq, Pb, seq, flags, s);
        } else {
            r = group_gemm(seq, seq, head_dim, Qs, QT ? 1 : 0, K, 1, Pb, seq, P.zb, P.zh, count,
                           nh, 1, s);
            if (r == cudaSuccess)
                r = launch_softmax_causal(count * seq, seq, Pb, seq, scale, 0, seq, Pb, seq, s);
        }
        if (r == cudaSuccess)
            r = group_gemm(seq, seq, head_dim, dOs, dOT ? 1 : 0, Vs, VT ? 0 : 1, dPb, seq, dP.zb,
                           dP.zh, count, nh, 1, s);
        if (r == cudaSuccess && !saved)
            r = count_nonfinite_heads(flags, finite, 3, nb * seq, nh * head_dim, s);
        if (r == cudaSuccess)   // dV = P^T dO
            r = group_gemm(seq, head_dim, seq, P, 1, dO, 0, dbase + 2 * hd, lddqkv, dzb,
                           head_dim, count, nh, 0, s, 2, flags);
        if (r == cudaSuccess)   // dS in place of dP
            r = launch_softmax_causal_bwd(count * seq, seq, Pb, dPb, seq, scale, 0, seq, dPb, seq,
                                          s);
        if (r == cudaSuccess)   // dQ = dS K
            r = group_gemm(seq, head_dim, seq, dP, 0, K, 0, dbase, lddqkv, dzb, head_dim, count,
                           nh, 0, s, 1, flags + 1);
        if (r == cudaSuccess)   // dK = dS^T Q
            r = group_gemm(seq, head_dim, seq, dP, 1, Q, 0, dbase + hd, lddqkv, dzb,
                           head_dim, count, nh, 0, s, 2, flags + 2);
        return r;
    });
    return from_cuda(e);
}
}  // namespace

DET_API det_status detattention_bwd_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                        int64_t heads, int64_t head_dim, const float *qkv,
                                        int64_t ldqkv, const float *dout, int64_t lddout,
                                        float scale, float *dqkv, int64_t lddqkv,
                                        void *workspace, size_t workspace_bytes,
                                        det_stream_t stream) {
    return attention_bwd(prof, batch, seq, heads, head_dim, qkv, ldqkv, dout, lddout, scale,
                         nullptr, dqkv, lddqkv, workspace, workspace_bytes, stream);
}

DET_API det_status detattention_bwd_saved_f32(const det_profile_v1 *prof, int64_t batch,
                                              int64_t seq, int64_t heads, int64_t head_dim,
                                              const float *qkv, int64_t ldqkv, const float *dout,
                                              int64_t lddout, float scale, void *fwd_workspace,
                                              size_t fwd_workspace_bytes, float *dqkv,
                                              int64_t lddqkv, void *workspace,
                                              size_t workspace_bytes, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!attention_args_ok(batch, seq, heads, head_dim)) return DET_ERR_INVALID_ARG;
    if (batch == 0) return DET_OK;
    // the forward's workspace as detattention_f32 lays it out: the group's
    // P first
    const AttnGroups g = attention_groups(batch, seq, heads);
    if (!fwd_workspace || reinterpret_cast<uintptr_t>(fwd_workspace) % 256 ||
        fwd_workspace_bytes < g.score_bytes + kAttnFlagBytes +
                                  attn_qkt_bytes(batch, seq, heads, head_dim))
        return DET_ERR_WORKSPACE;
    return attention_bwd(prof, batch, seq, heads, head_dim, qkv, ldqkv, dout, lddout, scale,
                         static_cast<float *>(fwd_workspace), dqkv, lddqkv, workspace,
                         workspace_bytes, stream);
}

DET_API det_status detshardsum_f32(const det_profile_v1 *prof, int64_t nshards, int64_t n,
                                   const float *shards, int64_t ld, float scale, float *out,
                                   det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (nshards < 1 || nshards > kDimMax || n < 0 || n > (int64_t(1) << 40))
        return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (ld < n || !shards || !out) return DET_ERR_INVALID_ARG;
    // out may be shard 0 itself; it must not overlap any other shard
    const float *end = shards + (nshards - 1) * ld + n;
    if (out != shards && out + n > shards && out < end) return DET_ERR_INVALID_ARG;
    if (out == shards && nshards > 1 && ld < n) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_shardsum(nshards, n, shards, ld, scale, out,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detgemm_f32_noalloc(const det_profile_v1 *prof, int transA, int transB,
                                       int64_t M, int64_t N, int64_t K, const float *A,
                                       int64_t lda, const float *B, int64_t ldb, float *C,
                                       int64_t ldc, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (M < 0 || N < 0 || K < 0 || M > kDimMax || N > kDimMax || K > kDimMax)
        return DET_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DET_OK;
    const int64_t a_row = transA ? M : K, b_row = transB ? K : N;
    if (ldc < N || lda < std::max<int64_t>(a_row, 1) || ldb < std::max<int64_t>(b_row, 1))
        return DET_ERR_INVALID_ARG;
    if (!C || (K > 0 && (!A || !B))) return DET_ERR_INVALID_ARG;
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    if (tiles > kDimMax) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    GemmArgs a;
    a.M = M; a.N = N; a.K = K; a.lda = lda; a.ldb = ldb; a.ldc = ldc;
    a.A = A; a.B = B; a.C = C; a.transA = transA != 0; a.transB = transB != 0;
    bool too_big = false;
    const cudaError_t e =
        launch_gemm_noalloc(a, &too_big, reinterpret_cast<cudaStream_t>(stream));
    if (too_big) return DET_ERR_WORKSPACE;
    return from_cuda(e);
}

DET_API det_status detrmsnorm_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                                  const float *x, int64_t ldx, const float *gain,
                                  float eps, float *y, int64_t ldy, float *inv_rms,
                                  det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || D < 1 || D > kDimMax) return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (ldx < D || ldy < D || !x || !gain || !y) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_rmsnorm(rows, D, x, ldx, gain, eps, y, ldy, inv_rms,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detadd_rmsnorm_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                                      const float *a, const float *b, float *x,
                                      const float *gain, float eps, float *y, int64_t ldy,
                                      float *inv_rms, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || D < 1 || D > kDimMax || rows > kDimMax) return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (ldy < D || !a || !b || !x || !gain || !y) return DET_ERR_INVALID_ARG;
    // x must not overlap a, b or y (it is written while they are read)
    const int64_t n = rows * D;
    auto overlap = [n](const float *p, const float *q) { return p < q + n && q < p + n; };
    if (overlap(x, a) || overlap(x, b) || (y < x + n && x < y + (rows - 1) * ldy + D))
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_add_rmsnorm(rows, D, a, b, x, D, gain, eps, y, ldy, inv_rms, s);
    if (e == cudaErrorNotSupported) {
        (void)cudaGetLastError();
        e = launch_add(n, a, b, x, s);
        if (e == cudaSuccess) e = launch_rmsnorm(rows, D, x, D, gain, eps, y, ldy, inv_rms, s);
    }
    return from_cuda(e);
}

DET_API det_status detrmsnorm_bwd_workspace_bytes(const det_profile_v1 *prof, int64_t rows,
                                                  int64_t D, size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || rows < 0 || rows > kDimMax || D < 1 || D > kDimMax) return DET_ERR_INVALID_ARG;
    *bytes = rmsnorm_bwd_workspace_bytes(rows, D);
    return DET_OK;
}

DET_API det_status detrmsnorm_bwd_f32(const det_profile_v1 *prof, int64_t rows, int64_t D,
                                      const float *x, int64_t ldx, const float *gain,
                                      const float *inv_rms, const float *dy, int64_t lddy,
                                      float *dx, int64_t lddx, float *dgain, void *workspace,
                                      size_t workspace_bytes, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || rows > kDimMax || D < 1 || D > kDimMax || !dgain) return DET_ERR_INVALID_ARG;
    if (rows > 0) {
        if (ldx < D || lddy < D || lddx < D || !x || !gain || !inv_rms || !dy || !dx)
            return DET_ERR_INVALID_ARG;
        if (dx == dy && lddx != lddy) return DET_ERR_INVALID_ARG;
        const size_t need = rmsnorm_bwd_workspace_bytes(rows, D);
        if (need > 0 && (!workspace || workspace_bytes < need ||
                         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
            return DET_ERR_WORKSPACE;
    }
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_rmsnorm_bwd(rows, D, x, ldx, gain, inv_rms, dy, lddy, dx, lddx,
                                        dgain, static_cast<float *>(workspace),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detxent_f32(const det_profile_v1 *prof, int64_t rows, int64_t V,
                               const float *logits, int64_t ld, const int32_t *labels,
                               float *loss, float *loss_mean, float *dlogits, int64_t ldd,
                               float dscale, int32_t *dev_status, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (rows < 0 || V < 1 || V > kDimMax) return DET_ERR_INVALID_ARG;
    if (rows == 0) return DET_OK;
    if (ld < V || !logits || !labels || !loss) return DET_ERR_INVALID_ARG;
    if (dlogits && ldd < V) return DET_ERR_INVALID_ARG;
    if (dlogits && dlogits == logits && ldd != ld) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_xent(rows, V, logits, ld, labels, loss, loss_mean, dlogits,
                                 ldd, dscale, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status det_adamw_bias_correction(int64_t step, float beta1, float beta2,
                                             float *bc1, float *bc2) {
    if (step < 1 || !beta_ok(beta1) || !beta_ok(beta2) || !bc1 || !bc2)
        return DET_ERR_INVALID_ARG;
    adamw_bias_correction(step, beta1, beta2, bc1, bc2);
    return DET_OK;
}

DET_API det_status detadamw_f32(const det_profile_v1 *prof, int64_t n, float *p,
                                const float *g, float *m, float *v,
                                const det_adamw_hp *hp, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0 || !hp || hp->step < 1 || !beta_ok(hp->beta1) || !beta_ok(hp->beta2))
        return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!p || !g || !m || !v) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_adamw(n, p, g, m, v, *hp, reinterpret_cast<cudaStream_t>(stream)));
}

static det_status exp_log(const det_profile_v1 *prof, int64_t n, const float *x, float *y,
                          det_stream_t stream, int is_log) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0) return DET_ERR_INVALID_ARG;
    if (n == 0) return DET_OK;
    if (!x || !y) return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    return from_cuda(launch_exp_map(n, x, y, is_log, reinterpret_cast<cudaStream_t>(stream)));
}

DET_API det_status detexp_f32(const det_profile_v1 *prof, int64_t n, const float *x,
                              float *y, det_stream_t stream) {
    return exp_log(prof, n, x, y, stream, 0);
}

DET_API det_status detlog_f32(const det_profile_v1 *prof, int64_t n, const float *x,
                              float *y, det_stream_t stream) {
    return exp_log(prof, n, x, y, stream, 1);
}

DET_API det_status det_watchdog_status(int32_t *code, int clear) {
    if (!code) return DET_ERR_INVALID_ARG;
    unsigned int c = 0, c2 = 0;
    cudaError_t e = gemm_watchdog(&c, clear);
    unsigned int c3 = 0, c4 = 0;
    if (e == cudaSuccess) e = n64::gemm_watchdog(&c4, clear);
    c |= c4;
    if (e == cudaSuccess) e = m128::gemm_watchdog(&c4, clear);
    c |= c4;
    if (e == cudaSuccess) e = rowops_watchdog(&c2, clear);
    if (e == cudaSuccess) e = rmsbwd_watchdog(&c3, clear);
    unsigned int c5 = 0;
    if (e == cudaSuccess) e = block_watchdog(&c5, clear);
    *code = int32_t(c | c2 | c3 | c5);
    return from_cuda(e);
}
