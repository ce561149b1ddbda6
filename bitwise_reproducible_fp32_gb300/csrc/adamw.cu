// adamw.cu -- the profile's AdamW update for sm_103a.
//
// "MojoLearn 162M" model card, table "Training": AdamW with beta (0.9, 0.95),
// eps 1e-8, weight decay 0.1 and no gradient clipping; the card's text adds
// that the untied input table puts 38.6M more parameters through every update.
// The update is the decoupled-decay form, elementwise, one rounding per
// written operation:
//   m' = fmaf(b1, m, (1-b1) g);  v' = fmaf(b2, v, (1-b2)(g g))
//   u  = (m'/bc1) / (sqrt(v'/bc2) + eps);  p' = fmaf(-lr, u, p (1 - lr wd))
// with bc = 1 - b^t and b^t formed by t-1 sequential float products.
// bc1 and bc2 are formed once on the host by adamw_bias_correction (exported
// as det_adamw_bias_correction) and passed to the kernel, so the bias
// corrections a caller can read through the C ABI are the ones every update
// uses. Host float arithmetic is IEEE binary32 on both build targets
// (x86-64 SSE, aarch64), and the library's host code is compiled without
// contraction, so each product and the difference are rounded once.
//
// The kernel is HBM-bound (16 bytes read and 12 written a parameter): a
// persistent grid of a few CTAs an SM walks the arrays as float4 with two
// vectors in flight a thread; the tail and unaligned arrays go scalar.
#include <algorithm>

#include "det_internal.cuh"

namespace det {
namespace {

constexpr int kThreads = 256;

struct Coef {
    float lr, b1, b2, eps, omb1, omb2, wdf, bc1, bc2;
};

__device__ __forceinline__ void adamw_one(const Coef &c, float &p, float g, float &m,
                                          float &v) {
    const float mn = __fmaf_rn(c.b1, m, __fmul_rn(c.omb1, g));
    const float vn = __fmaf_rn(c.b2, v, __fmul_rn(c.omb2, __fmul_rn(g, g)));
    const float mh = __fdiv_rn(mn, c.bc1);
    const float vh = __fdiv_rn(vn, c.bc2);
    const float u = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), c.eps));
    p = __fmaf_rn(-c.lr, u, __fmul_rn(p, c.wdf));
    m = mn;
    v = vn;
}

__global__ void __launch_bounds__(kThreads)
    adamw_kernel(int64_t n, float *__restrict__ P, const float *__restrict__ G,
                 float *__restrict__ M, float *__restrict__ Vv, float lr, float b1,
                 float b2, float eps, float wd, float bc1, float bc2, int vec) {
    Coef c;
    c.lr = lr; c.b1 = b1; c.b2 = b2; c.eps = eps;
    c.omb1 = __fsub_rn(1.0f, b1);
    c.omb2 = __fsub_rn(1.0f, b2);
    c.wdf = __fsub_rn(1.0f, __fmul_rn(lr, wd));
    c.bc1 = bc1;
    c.bc2 = bc2;

    const int64_t tid = blockIdx.x * int64_t(kThreads) + threadIdx.x;
    const int64_t nth = int64_t(gridDim.x) * kThreads;
    int64_t done = 0;
    if (vec) {
        const int64_t n4 = n / 4;
        float4 *P4 = reinterpret_cast<float4 *>(P);
        const float4 *G4 = reinterpret_cast<const float4 *>(G);
        float4 *M4 = reinterpret_cast<float4 *>(M);
        float4 *V4 = reinterpret_cast<float4 *>(Vv);
        int64_t i = tid;
        for (; i + nth < n4; i += 2 * nth) {
            float4 p[2], g[2], m[2], v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t k = i + u * nth;
                p[u] = P4[k]; g[u] = __ldcs(G4 + k); m[u] = M4[k]; v[u] = V4[k];
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                adamw_one(c, p[u].x, g[u].x, m[u].x, v[u].x);
                adamw_one(c, p[u].y, g[u].y, m[u].y, v[u].y);
                adamw_one(c, p[u].z, g[u].z, m[u].z, v[u].z);
                adamw_one(c, p[u].w, g[u].w, m[u].w, v[u].w);
                const int64_t k = i + u * nth;
                __stcs(P4 + k, p[u]); __stcs(M4 + k, m[u]); __stcs(V4 + k, v[u]);
            }
        }
        for (; i < n4; i += nth) {
            float4 p = P4[i], g = __ldcs(G4 + i), m = M4[i], v = V4[i];
            adamw_one(c, p.x, g.x, m.x, v.x);
            adamw_one(c, p.y, g.y, m.y, v.y);
            adamw_one(c, p.z, g.z, m.z, v.z);
            adamw_one(c, p.w, g.w, m.w, v.w);
            __stcs(P4 + i, p); __stcs(M4 + i, m); __stcs(V4 + i, v);
        }
        done = n4 * 4;
    }
    for (int64_t i = done + tid; i < n; i += nth) {
        float p = P[i], m = M[i], v = Vv[i];
        adamw_one(c, p, G[i], m, v);
        P[i] = p; M[i] = m; Vv[i] = v;
    }
}

}  // namespace

// beta^t by t-1 sequential float products, then 1 - beta^t, for both betas.
// Once a product stops changing (0, 1, or a subnormal that beta maps to
// itself) every later product is the same, so the loop may stop there: the
// result is that of all t-1 products.
void adamw_bias_correction(int64_t step, float beta1, float beta2, float *bc1, float *bc2) {
    volatile float p1 = beta1, p2 = beta2;   // each product stored, so rounded once
    for (int64_t t = 2; t <= step; ++t) {
        const float n1 = p1 * beta1, n2 = p2 * beta2;
        if (n1 == p1 && n2 == p2) break;
        p1 = n1;
        p2 = n2;
    }
    const float one = 1.0f;
    *bc1 = one - p1;
    *bc2 = one - p2;
}

cudaError_t launch_adamw(int64_t n, float *p, const float *g, float *m, float *v,
                         const det_adamw_hp &hp, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    auto al16 = [](const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    const int vec = al16(p) && al16(g) && al16(m) && al16(v);
    const int64_t want = (n / 4 + kThreads - 1) / kThreads;
    const int64_t blocks =
        std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sm_count_current_device()) * 4));
    float bc1 = 0.0f, bc2 = 0.0f;
    adamw_bias_correction(hp.step, hp.beta1, hp.beta2, &bc1, &bc2);
    adamw_kernel<<<unsigned(blocks), kThreads, 0, s>>>(n, p, g, m, v, hp.lr, hp.beta1,
                                                      hp.beta2, hp.eps, hp.weight_decay,
                                                      bc1, bc2, vec);
    return cudaGetLastError();
}

}  // namespace det
