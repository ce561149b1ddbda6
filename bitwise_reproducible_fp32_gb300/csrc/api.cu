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
    (void)transB;
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || M < 0 || N < 0 || K < 0 || M > kDimMax || N > kDimMax || K > kDimMax)
        return DET_ERR_INVALID_ARG;
    *bytes = 0;
    if (M == 0 || N == 0 || K == 0) return DET_OK;
    if ((st = check_device()) != DET_OK) return st;
    *bytes = gemm_plan(M, N, K, sm_count_current_device(), transA == 0).workspace_bytes;
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

// Causal attention over one packed QKV activation: for every sequence b and
// head h, S = Q_bh K_bh^T (profile GEMM), P = the causal softmax of S * scale,
// O_bh = P V_bh (profile GEMM), each head one after the other through one
// seq x seq score buffer in the workspace.
namespace {
size_t attention_ws(int64_t seq, int64_t head_dim, size_t *gemm_ws) {
    *gemm_ws = gemm_plan(seq, head_dim, seq, sm_count_current_device(), true).workspace_bytes;
    return (size_t(seq) * size_t(seq) * 4 + 255) / 256 * 256 + *gemm_ws;
}
}  // namespace

DET_API det_status detattention_workspace_bytes(const det_profile_v1 *prof, int64_t seq,
                                                int64_t head_dim, size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || seq < 1 || seq > 65536 || head_dim < 1 || head_dim > 65536)
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    size_t g = 0;
    *bytes = attention_ws(seq, head_dim, &g);
    return DET_OK;
}

DET_API det_status detattention_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                    int64_t heads, int64_t head_dim, const float *qkv,
                                    int64_t ldqkv, float scale, float *out, int64_t ldout,
                                    void *workspace, size_t workspace_bytes,
                                    det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (batch < 0 || seq < 1 || seq > 65536 || heads < 1 || head_dim < 1 || head_dim > 65536 ||
        heads > 65536)
        return DET_ERR_INVALID_ARG;
    if (batch == 0) return DET_OK;
    if (!qkv || !out || ldqkv < 3 * heads * head_dim || ldout < heads * head_dim)
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    size_t gws = 0;
    const size_t need = attention_ws(seq, head_dim, &gws);
    if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
        return DET_ERR_WORKSPACE;
    float *scores = static_cast<float *>(workspace);
    void *pv_ws = gws ? static_cast<char *>(workspace) + (need - gws) : nullptr;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t hd = heads * head_dim;
    for (int64_t b = 0; b < batch; ++b) {
        const float *base = qkv + b * seq * ldqkv;
        for (int64_t h = 0; h < heads; ++h) {
            GemmArgs qk;
            qk.M = seq; qk.N = seq; qk.K = head_dim;
            qk.A = base + h * head_dim; qk.lda = ldqkv;
            qk.B = base + hd + h * head_dim; qk.ldb = ldqkv;
            qk.C = scores; qk.ldc = seq;
            qk.transA = 0; qk.transB = 1;
            cudaError_t e = launch_gemm(qk, nullptr, 0, s);
            if (e == cudaSuccess)
                e = launch_softmax_causal(seq, seq, scores, seq, scale, 0, seq, scores, seq, s);
            if (e != cudaSuccess) return DET_ERR_CUDA;
            GemmArgs pv;
            pv.M = seq; pv.N = head_dim; pv.K = seq;
            pv.A = scores; pv.lda = seq;
            pv.B = base + 2 * hd + h * head_dim; pv.ldb = ldqkv;
            pv.C = out + b * seq * ldout + h * head_dim; pv.ldc = ldout;
            pv.transA = 0; pv.transB = 0;
            if (launch_gemm(pv, pv_ws, gws, s) != cudaSuccess) return DET_ERR_CUDA;
        }
    }
    return DET_OK;
}

// Backward of detattention_f32, head after head: P is recomputed by the
// forward's spelling (S = Q K^T, the causal softmax), then
//   dP = dO V^T, dV = P^T dO, dS = the softmax backward of (P, dP),
//   dQ = dS K, dK = dS^T Q
// with detgemm_f32's arithmetic for every product. The gradients are those of
// the Q, K and V that the forward read (after any rotary embedding).
namespace {
size_t attention_bwd_ws(int64_t seq, int64_t head_dim, size_t *gemm_ws) {
    *gemm_ws = gemm_plan(seq, head_dim, seq, sm_count_current_device(), true).workspace_bytes;
    return 2 * ((size_t(seq) * size_t(seq) * 4 + 255) / 256 * 256) + *gemm_ws;
}
}  // namespace

DET_API det_status detattention_bwd_workspace_bytes(const det_profile_v1 *prof, int64_t seq,
                                                    int64_t head_dim, size_t *bytes) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (!bytes || seq < 1 || seq > 65536 || head_dim < 1 || head_dim > 65536)
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    size_t g = 0;
    *bytes = attention_bwd_ws(seq, head_dim, &g);
    return DET_OK;
}

DET_API det_status detattention_bwd_f32(const det_profile_v1 *prof, int64_t batch, int64_t seq,
                                        int64_t heads, int64_t head_dim, const float *qkv,
                                        int64_t ldqkv, const float *dout, int64_t lddout,
                                        float scale, float *dqkv, int64_t lddqkv,
                                        void *workspace, size_t workspace_bytes,
                                        det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (batch < 0 || seq < 1 || seq > 65536 || heads < 1 || head_dim < 1 || head_dim > 65536 ||
        heads > 65536)
        return DET_ERR_INVALID_ARG;
    if (batch == 0) return DET_OK;
    const int64_t hd = heads * head_dim;
    if (!qkv || !dout || !dqkv || ldqkv < 3 * hd || lddout < hd || lddqkv < 3 * hd)
        return DET_ERR_INVALID_ARG;
    if ((st = check_device()) != DET_OK) return st;
    size_t gws = 0;
    const size_t need = attention_bwd_ws(seq, head_dim, &gws);
    if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
        return DET_ERR_WORKSPACE;
    const size_t tt = (size_t(seq) * size_t(seq) * 4 + 255) / 256 * 256;
    float *P = static_cast<float *>(workspace);
    float *dP = reinterpret_cast<float *>(static_cast<char *>(workspace) + tt);
    void *gw = gws ? static_cast<char *>(workspace) + 2 * tt : nullptr;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto gemm = [&](int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, int tA,
                    const float *B, int64_t ldb, int tB, float *C, int64_t ldc, bool ws) {
        GemmArgs a;
        a.M = M; a.N = N; a.K = K; a.A = A; a.lda = lda; a.B = B; a.ldb = ldb;
        a.C = C; a.ldc = ldc; a.transA = tA; a.transB = tB;
        return launch_gemm(a, ws ? gw : nullptr, ws ? gws : 0, s);
    };
    for (int64_t b = 0; b < batch; ++b) {
        const float *base = qkv + b * seq * ldqkv;
        const float *dob = dout + b * seq * lddout;
        float *dbase = dqkv + b * seq * lddqkv;
        for (int64_t h = 0; h < heads; ++h) {
            const float *Q = base + h * head_dim, *K = base + hd + h * head_dim;
            const float *V = base + 2 * hd + h * head_dim, *dO = dob + h * head_dim;
            float *dQ = dbase + h * head_dim, *dK = dbase + hd + h * head_dim;
            float *dV = dbase + 2 * hd + h * head_dim;
            cudaError_t e = gemm(seq, seq, head_dim, Q, ldqkv, 0, K, ldqkv, 1, P, seq, false);
            if (e == cudaSuccess)
                e = launch_softmax_causal(seq, seq, P, seq, scale, 0, seq, P, seq, s);
            if (e == cudaSuccess)
                e = gemm(seq, seq, head_dim, dO, lddout, 0, V, ldqkv, 1, dP, seq, false);
            if (e == cudaSuccess)
                e = gemm(seq, head_dim, seq, P, seq, 1, dO, lddout, 0, dV, lddqkv, true);
            if (e == cudaSuccess)
                e = launch_softmax_causal_bwd(seq, seq, P, dP, seq, scale, 0, seq, dP, seq, s);
            if (e == cudaSuccess)
                e = gemm(seq, head_dim, seq, dP, seq, 0, K, ldqkv, 0, dQ, lddqkv, true);
            if (e == cudaSuccess)
                e = gemm(seq, head_dim, seq, dP, seq, 1, Q, ldqkv, 0, dK, lddqkv, true);
            if (e != cudaSuccess) return DET_ERR_CUDA;
        }
    }
    return DET_OK;
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

DET_API det_status detadamw_f32(const det_profile_v1 *prof, int64_t n, float *p,
                                const float *g, float *m, float *v,
                                const det_adamw_hp *hp, det_stream_t stream) {
    det_status st = check_profile(prof);
    if (st != DET_OK) return st;
    if (n < 0 || !hp || hp->step < 1) return DET_ERR_INVALID_ARG;
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
    unsigned int c3 = 0;
    if (e == cudaSuccess) e = rowops_watchdog(&c2, clear);
    if (e == cudaSuccess) e = rmsbwd_watchdog(&c3, clear);
    *code = int32_t(c | c2 | c3);
    return from_cuda(e);
}
