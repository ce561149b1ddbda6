// rowops.cu -- fixed-tree row reductions for sm_103a: RMSNorm, softmax
// cross-entropy (+ dlogits, + mean) and the profile's exp / log.
//
// Profile v1 reduction ("mojolearn" PyPI page, section "What bitwise identity
// means, and why it is not the default": the reduction order and partitioning
// are fixed): a row is summed by L chains; chain l owns the 4-element groups
// g of the row with g mod L == l and adds them in ascending index; the L chain
// values are folded by an xor butterfly with offsets 16, 8, 4, 2, 1, then 32,
// 64, ... The GPU mapping is the natural one: chain l is thread l, a group is
// one float4-wide step of a coalesced sweep, the first five butterfly levels
// are __shfl_xor_sync inside a warp and the rest go through shared memory.
//
// The exp and log spellings are the profile's own (same page and section:
// the spellings of exp and log are fixed): Cody-Waite reduction with a
// degree-7 Taylor polynomial for exp, and the atanh series arranged as in
// fdlibm for log. Every operation is an explicitly rounded intrinsic; the
// library is built with -fmad=false -ftz=false -prec-div=true
// -prec-sqrt=true, so nothing is contracted or flushed.
#include <algorithm>

#include "det_internal.cuh"

namespace det {
namespace {

// ---------------------------------------------------------------- exp / log
// exp constants: each the float nearest to its definition. LOG2E = 1/ln 2,
// LN2_HI = ln 2, LN2_LO = ln 2 - LN2_HI, C_k = 1/k!.
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e430p-1f;
constexpr float kLn2Lo = -0x1.05c610p-29f;
constexpr float kC2 = 0x1p-1f, kC3 = 0x1.555556p-3f, kC4 = 0x1.555556p-5f;
constexpr float kC5 = 0x1.111112p-7f, kC6 = 0x1.6c16c2p-10f, kC7 = 0x1.a01a02p-13f;
constexpr float kExpHi = 0x1.62e42ep+6f;   // largest float with a finite exp
constexpr float kExpLo = -104.0f;          // below: +0
// log constants: A_k = 2/k (k = 3..11 odd); the largest float below sqrt 2.
constexpr float kA3 = 0x1.555556p-1f, kA5 = 0x1.99999ap-2f, kA7 = 0x1.24924ap-2f;
constexpr float kA9 = 0x1.c71c72p-3f, kA11 = 0x1.745d18p-3f;
constexpr unsigned kSqrt2Bits = 0x3fb504f3u;

__device__ __forceinline__ float pow2i(int e) {   // 2^e, -126 <= e <= 127
    return __uint_as_float(unsigned(e + 127) << 23);
}

__device__ __forceinline__ float det_exp(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x > kExpHi) return __uint_as_float(0x7f800000u);
    if (x < kExpLo) return 0.0f;
    const float t = __fmul_rn(x, kLog2e);
    const float n = rintf(t);                 // round half to even
    float r = __fmaf_rn(-n, kLn2Hi, x);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = kC7;
    p = __fmaf_rn(p, r, kC6);
    p = __fmaf_rn(p, r, kC5);
    p = __fmaf_rn(p, r, kC4);
    p = __fmaf_rn(p, r, kC3);
    p = __fmaf_rn(p, r, kC2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ni = __float2int_rn(n);         // |n| <= 150, exact
    if (ni > 127) return __fmul_rn(__fadd_rn(p, p), pow2i(127));
    if (ni < -126) return __fmul_rn(__fmul_rn(p, pow2i(ni + 64)), pow2i(-64));
    return __fmul_rn(p, pow2i(ni));
}

__device__ __forceinline__ float det_log(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x < 0.0f) return __uint_as_float(0x7fc00000u);
    if (x == 0.0f) return __uint_as_float(0xff800000u);
    if (x == __uint_as_float(0x7f800000u)) return x;
    int e = 0;
    if (x < 0x1p-126f) { x = __fmul_rn(x, 0x1p23f); e = -23; }
    const unsigned b = __float_as_uint(x);
    e += int(b >> 23) - 127;
    unsigned fb = (b & 0x007fffffu) | 0x3f800000u;
    if (fb > kSqrt2Bits) { fb -= 0x00800000u; e += 1; }
    const float f = __uint_as_float(fb);
    const float u = __fsub_rn(f, 1.0f);
    const float s = __fdiv_rn(u, __fadd_rn(2.0f, u));
    const float z = __fmul_rn(s, s);
    float R = kA11;
    R = __fmaf_rn(R, z, kA9);
    R = __fmaf_rn(R, z, kA7);
    R = __fmaf_rn(R, z, kA5);
    R = __fmaf_rn(R, z, kA3);
    R = __fmul_rn(R, z);
    const float h = __fmul_rn(__fmul_rn(0.5f, u), u);
    const float lf = __fsub_rn(u, __fsub_rn(h, __fmul_rn(s, __fadd_rn(h, R))));
    const float ef = __int2float_rn(e);
    return __fmaf_rn(ef, kLn2Hi, __fmaf_rn(ef, kLn2Lo, lf));
}

// NaN-propagating max (the profile's max: any NaN in a row makes m NaN).
__device__ __forceinline__ float nan_max(float a, float b) {
    return (a != a || a > b) ? a : b;
}

__device__ __forceinline__ float warp_butterfly_sum(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// ---------------------------------------------------------------- RMSNorm
// One warp per row; lane l owns groups l, l + 32, ... Rows whose start and
// length allow it are read as float4 and kept in registers (up to CACHE
// groups a lane), then written from registers.
constexpr int kRmsWarps = 8;
constexpr int kRmsCache = 8;

__global__ void __launch_bounds__(kRmsWarps * 32)
    rmsnorm_kernel(int64_t rows, int64_t D, const float *__restrict__ x, int64_t ldx,
                   const float *__restrict__ gain, float eps, float *__restrict__ y,
                   int64_t ldy, float *__restrict__ inv_rms, int vec) {
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kRmsWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float *xr = x + row * ldx;
    float *yr = y + row * ldy;
    const int64_t ngroups = (D + 3) / 4;
    float s = 0.0f;
    const float Df = __ll2float_rn(D);
    if (vec && ngroups <= int64_t(kRmsCache) * 32) {
        float4 v[kRmsCache];
#pragma unroll
        for (int t = 0; t < kRmsCache; ++t) {
            const int64_t g = lane + 32 * t;
            if (g < ngroups) v[t] = __ldg(reinterpret_cast<const float4 *>(xr) + g);
        }
#pragma unroll
        for (int t = 0; t < kRmsCache; ++t) {
            const int64_t g = lane + 32 * t;
            if (g < ngroups) {
                s = __fmaf_rn(v[t].x, v[t].x, s);
                s = __fmaf_rn(v[t].y, v[t].y, s);
                s = __fmaf_rn(v[t].z, v[t].z, s);
                s = __fmaf_rn(v[t].w, v[t].w, s);
            }
        }
        const float ss = warp_butterfly_sum(s);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Df), eps)));
#pragma unroll
        for (int t = 0; t < kRmsCache; ++t) {
            const int64_t g = lane + 32 * t;
            if (g < ngroups) {
                const float4 gg = __ldg(reinterpret_cast<const float4 *>(gain) + g);
                float4 o;
                o.x = __fmul_rn(__fmul_rn(v[t].x, r), gg.x);
                o.y = __fmul_rn(__fmul_rn(v[t].y, r), gg.y);
                o.z = __fmul_rn(__fmul_rn(v[t].z, r), gg.z);
                o.w = __fmul_rn(__fmul_rn(v[t].w, r), gg.w);
                reinterpret_cast<float4 *>(yr)[g] = o;
            }
        }
        if (inv_rms && lane == 0) inv_rms[row] = r;
        return;
    }
    // general rows: scalar loads, chain order by logical index
    for (int64_t g = lane; g < ngroups; g += 32) {
        const int64_t j0 = 4 * g;
        const int64_t jn = j0 + 4 < D ? j0 + 4 : D;
        for (int64_t j = j0; j < jn; ++j) {
            const float xv = xr[j];
            s = __fmaf_rn(xv, xv, s);
        }
    }
    const float ss = warp_butterfly_sum(s);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Df), eps)));
    for (int64_t j = lane; j < D; j += 32) yr[j] = __fmul_rn(__fmul_rn(xr[j], r), gain[j]);
    if (inv_rms && lane == 0) inv_rms[row] = r;
}

// ---------------------------------------------------------------- cross-entropy
// One 256-thread CTA per row (thread l = chain l of the 256-chain profile).
constexpr int kXentThreads = 256;
static_assert(kXentThreads == kXentLanes, "one thread per chain");

__global__ void __launch_bounds__(kXentThreads)
    xent_kernel(int64_t rows, int64_t V, const float *__restrict__ logits, int64_t ld,
                const int32_t *__restrict__ labels, float *__restrict__ loss,
                float *dlogits, int64_t ldd, float dscale, int32_t *dev_status) {
    __shared__ float red[kXentThreads / 32];
    __shared__ float bcast;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float *x = logits + row * ld;
        const int64_t y = labels[row];
        const bool bad = (y < 0 || y >= V);
        if (bad) {
            if (tid == 0) {
                loss[row] = __uint_as_float(0x7fc00000u);
                if (dev_status) atomicOr(reinterpret_cast<int *>(dev_status), 1);
            }
            if (dlogits) {
                float *d = dlogits + row * ldd;
                for (int64_t j = tid; j < V; j += kXentThreads)
                    d[j] = __uint_as_float(0x7fc00000u);
            }
            continue;   // uniform across the CTA
        }
        // 1. m = max (order-free)
        float m = x[0];
        for (int64_t j = tid; j < V; j += kXentThreads) m = nan_max(__ldg(x + j), m);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            m = nan_max(__shfl_xor_sync(0xffffffffu, m, off), m);
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (tid == 0) {
            float mm = red[0];
            for (int w = 1; w < kXentThreads / 32; ++w) mm = nan_max(red[w], mm);
            bcast = mm;
        }
        __syncthreads();
        m = bcast;
        // 2. chain sums of e_j = exp(x_j - m), groups g = tid, tid + 256, ...
        float s = 0.0f;
        const int64_t ngroups = (V + 3) / 4;
        for (int64_t g = tid; g < ngroups; g += kXentThreads) {
            const int64_t j0 = 4 * g;
            if (j0 + 3 < V) {
                const float x0 = __ldg(x + j0), x1 = __ldg(x + j0 + 1);
                const float x2 = __ldg(x + j0 + 2), x3 = __ldg(x + j0 + 3);
                s = __fadd_rn(s, det_exp(__fsub_rn(x0, m)));
                s = __fadd_rn(s, det_exp(__fsub_rn(x1, m)));
                s = __fadd_rn(s, det_exp(__fsub_rn(x2, m)));
                s = __fadd_rn(s, det_exp(__fsub_rn(x3, m)));
            } else {
                for (int64_t j = j0; j < V; ++j)
                    s = __fadd_rn(s, det_exp(__fsub_rn(__ldg(x + j), m)));
            }
        }
        // 3. butterfly: 16..1 in the warp, then 32, 64, 128 across warps
        s = warp_butterfly_sum(s);
        __syncthreads();    // red[] reuse
        if (lane == 0) red[warp] = s;
        __syncthreads();
        if (tid == 0) {
            const float a01 = __fadd_rn(red[0], red[1]), a23 = __fadd_rn(red[2], red[3]);
            const float a45 = __fadd_rn(red[4], red[5]), a67 = __fadd_rn(red[6], red[7]);
            const float S = __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67));
            bcast = S;
            loss[row] = __fsub_rn(det_log(S), __fsub_rn(x[y], m));
        }
        __syncthreads();
        // 4. dlogits
        if (dlogits) {
            const float S = bcast;
            const float inv = __fdiv_rn(1.0f, S);
            float *d = dlogits + row * ldd;
            for (int64_t j = tid; j < V; j += kXentThreads) {
                const float e = det_exp(__fsub_rn(__ldg(x + j), m));
                const float onehot = (j == y) ? 1.0f : 0.0f;
                d[j] = __fmul_rn(__fsub_rn(__fmul_rn(e, inv), onehot), dscale);
            }
        }
        __syncthreads();    // bcast / red reuse by the next row
    }
}

// Mean of n floats: 32 chains (groups of 4, plain adds), butterfly, / n.
__global__ void mean_kernel(int64_t n, const float *__restrict__ v, float *out) {
    const int lane = threadIdx.x;
    float s = 0.0f;
    const int64_t ngroups = (n + 3) / 4;
    for (int64_t g = lane; g < ngroups; g += 32) {
        const int64_t j0 = 4 * g;
        const int64_t jn = j0 + 4 < n ? j0 + 4 : n;
        for (int64_t j = j0; j < jn; ++j) s = __fadd_rn(s, v[j]);
    }
    s = warp_butterfly_sum(s);
    if (lane == 0) *out = __fdiv_rn(s, __ll2float_rn(n));
}

__global__ void exp_map_kernel(int64_t n, const float *x, float *y, int is_log) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        y[i] = is_log ? det_log(x[i]) : det_exp(x[i]);
}

}  // namespace

cudaError_t launch_rmsnorm(int64_t rows, int64_t D, const float *x, int64_t ldx,
                           const float *gain, float eps, float *y, int64_t ldy,
                           float *inv_rms, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    auto al16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    const int vec = (D % 4 == 0) && (ldx % 4 == 0) && (ldy % 4 == 0) && al16(x) &&
                    al16(y) && al16(gain);
    const int64_t blocks = (rows + kRmsWarps - 1) / kRmsWarps;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    rmsnorm_kernel<<<unsigned(blocks), kRmsWarps * 32, 0, s>>>(rows, D, x, ldx, gain, eps,
                                                              y, ldy, inv_rms, vec);
    return cudaGetLastError();
}

cudaError_t launch_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                        const int32_t *labels, float *loss, float *loss_mean,
                        float *dlogits, int64_t ldd, float dscale, int32_t *dev_status,
                        cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>(rows, int64_t(sm_count_current_device()) * 8);
    xent_kernel<<<unsigned(grid), kXentThreads, 0, s>>>(rows, V, logits, ld, labels, loss,
                                                        dlogits, ldd, dscale, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !loss_mean) return e;
    mean_kernel<<<1, 32, 0, s>>>(rows, loss, loss_mean);
    return cudaGetLastError();
}

cudaError_t launch_exp_map(int64_t n, const float *x, float *y, int is_log,
                           cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int64_t blocks =
        std::min<int64_t>((n + 255) / 256, int64_t(sm_count_current_device()) * 16);
    exp_map_kernel<<<unsigned(blocks), 256, 0, s>>>(n, x, y, is_log);
    return cudaGetLastError();
}

}  // namespace det
