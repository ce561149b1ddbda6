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
// One warp per row; lane l owns groups l, l + 32, ... Rows whose start, stride
// and length allow it are read as float4 and held in registers (NG float4 a
// lane, NG = ceil(D / 128) up to 8), then written from registers; the register
// budget is kept small so every row of a typical batch is resident at once
// (8192 rows x 768 fit in one wave). Other rows take scalar loads in the same
// chain order.
constexpr int kRmsWarps = 8;
constexpr int kRmsMaxNG = 8;

template <int NG>
__global__ void __launch_bounds__(kRmsWarps * 32, (NG <= 4 ? 7 : NG <= 6 ? 6 : 4))
    rmsnorm_vec_kernel(int64_t rows, int64_t D, const float *__restrict__ x, int64_t ldx,
                       const float *__restrict__ gain, float eps, float *__restrict__ y,
                       int64_t ldy, float *__restrict__ inv_rms) {
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kRmsWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + row * ldx);
    const int ngroups = int(D >> 2);
    float4 v[NG];
#pragma unroll
    for (int t = 0; t < NG; ++t) {
        const int g = lane + 32 * t;
        if (g < ngroups) v[t] = __ldcs(xr + g);
    }
    float s = 0.0f;
#pragma unroll
    for (int t = 0; t < NG; ++t) {
        if (lane + 32 * t < ngroups) {
            s = __fmaf_rn(v[t].x, v[t].x, s);
            s = __fmaf_rn(v[t].y, v[t].y, s);
            s = __fmaf_rn(v[t].z, v[t].z, s);
            s = __fmaf_rn(v[t].w, v[t].w, s);
        }
    }
    const float ss = warp_butterfly_sum(s);
    const float r =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, __ll2float_rn(D)), eps)));
    float4 *yr = reinterpret_cast<float4 *>(y + row * ldy);
    const float4 *g4 = reinterpret_cast<const float4 *>(gain);
#pragma unroll
    for (int t = 0; t < NG; ++t) {
        const int g = lane + 32 * t;
        if (g < ngroups) {
            const float4 gg = __ldg(g4 + g);
            float4 o;
            o.x = __fmul_rn(__fmul_rn(v[t].x, r), gg.x);
            o.y = __fmul_rn(__fmul_rn(v[t].y, r), gg.y);
            o.z = __fmul_rn(__fmul_rn(v[t].z, r), gg.z);
            o.w = __fmul_rn(__fmul_rn(v[t].w, r), gg.w);
            __stcs(yr + g, o);
        }
    }
    if (inv_rms && lane == 0) inv_rms[row] = r;
}

__global__ void __launch_bounds__(kRmsWarps * 32)
    rmsnorm_kernel(int64_t rows, int64_t D, const float *__restrict__ x, int64_t ldx,
                   const float *__restrict__ gain, float eps, float *__restrict__ y,
                   int64_t ldy, float *__restrict__ inv_rms) {
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kRmsWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float *xr = x + row * ldx;
    float *yr = y + row * ldy;
    const int64_t ngroups = (D + 3) / 4;
    float s = 0.0f;
    for (int64_t g = lane; g < ngroups; g += 32) {
        const int64_t j0 = 4 * g;
        const int64_t jn = j0 + 4 < D ? j0 + 4 : D;
        for (int64_t j = j0; j < jn; ++j) {
            const float xv = xr[j];
            s = __fmaf_rn(xv, xv, s);
        }
    }
    const float ss = warp_butterfly_sum(s);
    const float r =
        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, __ll2float_rn(D)), eps)));
    for (int64_t j = lane; j < D; j += 32) yr[j] = __fmul_rn(__fmul_rn(xr[j], r), gain[j]);
    if (inv_rms && lane == 0) inv_rms[row] = r;
}

// ---------------------------------------------------------------- cross-entropy
// exp for arguments d <= 0 (or -inf), never NaN: the same bits as det_exp(d).
// n = rint(t) is formed as (t + 1.5 2^23) - 1.5 2^23, which rounds t to an
// integer with ties to even for |t| < 2^22; it can differ from rintf only in
// the sign of a zero n, which reaches the result only through r = d - n ln2
// and the polynomial's products with r, where it is inert. When n >= -125 the
// scaling p 2^n is exact and is done on the exponent bits; otherwise (deep
// underflow, -inf) the general routine runs.
constexpr float kRoundMagic = 0x1.8p23f;

__device__ __forceinline__ float det_exp_le0(float d) {
    const float t = __fmul_rn(d, kLog2e);
    const float tm = __fadd_rn(t, kRoundMagic);
    const int ni = __float_as_int(tm) - __float_as_int(kRoundMagic);
    if (ni < -125) return det_exp(d);
    const float n = __fsub_rn(tm, kRoundMagic);
    float r = __fmaf_rn(-n, kLn2Hi, d);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = kC7;
    p = __fmaf_rn(p, r, kC6);
    p = __fmaf_rn(p, r, kC5);
    p = __fmaf_rn(p, r, kC4);
    p = __fmaf_rn(p, r, kC3);
    p = __fmaf_rn(p, r, kC2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __int_as_float(__float_as_int(p) + int(unsigned(ni) << 23));
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float4 ld4_policy(const float *p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_policy(float *p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol)
                 : "memory");
}

// One 256-thread CTA per row at a time (thread l = chain l of the 256-chain
// profile), a persistent grid of two CTAs an SM. Per row:
//  1. m = max over the row: 16-byte loads of the row's 16-byte-aligned
//     granules (elements outside the row masked), kept in L2 (evict_last);
//  2. chain sums: chain l reads its logical groups 4g..4g+3 (g = l, l+256, ...)
//     from the aligned granule g and, through a lane shuffle, granule g+1;
//     e_j = exp(x_j - m) is added in ascending j and, when dlogits is
//     requested (and does not alias the logits), written to dlogits[j];
//  3. the butterfly 16..1 by shuffles, 32/64/128 through shared memory; thread
//     0 forms loss = log(S) - (x_y - m);
//  4. dlogits: d_j = (e_j * (1/S) - [j == y]) * dscale over the dlogits row's
//     granules, reading back e_j (or recomputing it in place).
// Rows with a non-finite max or a bad label take the general element-wise
// code, which performs the same operations.
constexpr int kXentThreads = 256;
constexpr int kU = 8;    // independent 16-byte loads a thread keeps in flight
constexpr int kU2 = 4;   // sweeps of the chain pass loaded ahead
static_assert(kXentThreads == kXentLanes, "one thread per chain");

__device__ __forceinline__ float4 pick_group(float4 c0, float4 c1, int h) {
    switch (h) {
        case 0: return c0;
        case 1: return make_float4(c0.y, c0.z, c0.w, c1.x);
        case 2: return make_float4(c0.z, c0.w, c1.x, c1.y);
        default: return make_float4(c0.w, c1.x, c1.y, c1.z);
    }
}

__global__ void __launch_bounds__(kXentThreads, 2)
    xent_kernel(int64_t rows, int64_t V, const float *logits, int64_t ld,
                const int32_t *__restrict__ labels, float *__restrict__ loss,
                float *dlogits, int64_t ldd, float dscale, int32_t *dev_status) {
    __shared__ float red[kXentThreads / 32];
    __shared__ float bcast;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t drop = l2_policy_evict_first();
    const int64_t ngroups = (V + 3) / 4;
    const bool in_place = dlogits != nullptr && dlogits == logits;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float *x = logits + row * ld;
        const int64_t y = labels[row];
        if (y < 0 || y >= V) {
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
        const int h = int((reinterpret_cast<uintptr_t>(x) >> 2) & 3);
        const float *xa = x - h;                     // 16-byte aligned
        const int64_t nchunks = (V + h + 3) / 4;     // granules touching the row
        // 1. m = max (order-free, NaN-propagating); kU independent loads in
        // flight a thread
        float m = x[0];
        for (int64_t q0 = tid; q0 < nchunks; q0 += int64_t(kXentThreads) * kU) {
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t q = q0 + int64_t(u) * kXentThreads;
                if (q < nchunks) v[u] = ld4_policy(xa + 4 * q, keep);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t q = q0 + int64_t(u) * kXentThreads;
                if (q >= nchunks) break;
                const int64_t j0 = 4 * q - h;
                if (j0 >= 0 && j0 + 3 < V) {
                    m = nan_max(v[u].x, m); m = nan_max(v[u].y, m);
                    m = nan_max(v[u].z, m); m = nan_max(v[u].w, m);
                } else {
                    if (j0 >= 0 && j0 < V) m = nan_max(v[u].x, m);
                    if (j0 + 1 >= 0 && j0 + 1 < V) m = nan_max(v[u].y, m);
                    if (j0 + 2 >= 0 && j0 + 2 < V) m = nan_max(v[u].z, m);
                    if (j0 + 3 >= 0 && j0 + 3 < V) m = nan_max(v[u].w, m);
                }
            }
        }
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
        const bool finite_m = fabsf(m) <= 3.402823466e38f;   // false for NaN / inf
        float *drow = dlogits ? dlogits + row * ldd : nullptr;
        const bool store_e = drow != nullptr && !in_place && finite_m;

        // 2. chain sums over the logical groups, kU2 sweeps' loads in flight
        float s = 0.0f;
        const int64_t titers = (ngroups + kXentThreads - 1) / kXentThreads;
        for (int64_t t0 = 0; t0 < titers; t0 += kU2) {
          float4 c0s[kU2], c1s[kU2];
#pragma unroll
          for (int u = 0; u < kU2; ++u) {
            const int64_t g = tid + (t0 + u) * kXentThreads;
            c0s[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            c1s[u] = c0s[u];
            if (t0 + u < titers && 4 * g - h < V) c0s[u] = ld4_policy(xa + 4 * g, drop);
            if (h != 0 && lane == 31 && t0 + u < titers && 4 * (g + 1) - h < V)
                c1s[u] = ld4_policy(xa + 4 * (g + 1), drop);
          }
#pragma unroll
          for (int u = 0; u < kU2; ++u) {
            if (t0 + u >= titers) break;    // uniform across the CTA
            const int64_t g = tid + (t0 + u) * kXentThreads;
            const float4 c0 = c0s[u];
            float4 c1 = c1s[u];
            if (h != 0) {
                const float nx = __shfl_down_sync(0xffffffffu, c0.x, 1);
                const float ny = __shfl_down_sync(0xffffffffu, c0.y, 1);
                const float nz = __shfl_down_sync(0xffffffffu, c0.z, 1);
                if (lane != 31) { c1.x = nx; c1.y = ny; c1.z = nz; }
            }
            if (g < ngroups) {
                const float4 v = pick_group(c0, c1, h);
                const int64_t j0 = 4 * g;
                if (finite_m) {
                    float e[4];
                    e[0] = det_exp_le0(__fsub_rn(v.x, m));
                    e[1] = det_exp_le0(__fsub_rn(v.y, m));
                    e[2] = det_exp_le0(__fsub_rn(v.z, m));
                    e[3] = det_exp_le0(__fsub_rn(v.w, m));
                    const int cnt = j0 + 3 < V ? 4 : int(V - j0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < cnt) s = __fadd_rn(s, e[k]);
                    if (store_e) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k < cnt) st_policy(drow + j0 + k, e[k], keep);
                    }
                } else {
                    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (j0 + k < V) s = __fadd_rn(s, det_exp(__fsub_rn(vv[k], m)));
                }
            }
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
        if (drow) {
            const float inv = __fdiv_rn(1.0f, bcast);
            if (store_e) {
                const int hd = int((reinterpret_cast<uintptr_t>(drow) >> 2) & 3);
                float *da = drow - hd;
                const int64_t dchunks = (V + hd + 3) / 4;
                for (int64_t q0 = tid; q0 < dchunks; q0 += int64_t(kXentThreads) * kU) {
                  float4 es[kU];
#pragma unroll
                  for (int u = 0; u < kU; ++u) {
                    const int64_t q = q0 + int64_t(u) * kXentThreads;
                    const int64_t j0 = 4 * q - hd;
                    if (q < dchunks && j0 >= 0 && j0 + 3 < V) es[u] = ld4_policy(da + 4 * q, drop);
                  }
#pragma unroll
                  for (int u = 0; u < kU; ++u) {
                    const int64_t q = q0 + int64_t(u) * kXentThreads;
                    if (q >= dchunks) break;
                    const int64_t j0 = 4 * q - hd;
                    if (j0 >= 0 && j0 + 3 < V) {
                        const float4 e = es[u];
                        float4 o;
                        o.x = __fmul_rn(__fsub_rn(__fmul_rn(e.x, inv), j0 == y ? 1.0f : 0.0f), dscale);
                        o.y = __fmul_rn(__fsub_rn(__fmul_rn(e.y, inv), j0 + 1 == y ? 1.0f : 0.0f), dscale);
                        o.z = __fmul_rn(__fsub_rn(__fmul_rn(e.z, inv), j0 + 2 == y ? 1.0f : 0.0f), dscale);
                        o.w = __fmul_rn(__fsub_rn(__fmul_rn(e.w, inv), j0 + 3 == y ? 1.0f : 0.0f), dscale);
                        __stcs(reinterpret_cast<float4 *>(da + 4 * q), o);
                    } else {
                        for (int k = 0; k < 4; ++k) {
                            const int64_t j = j0 + k;
                            if (j >= 0 && j < V) {
                                const float e = da[4 * q + k];
                                da[4 * q + k] = __fmul_rn(
                                    __fsub_rn(__fmul_rn(e, inv), j == y ? 1.0f : 0.0f), dscale);
                            }
                        }
                    }
                  }
                }
            } else {
                // in place, or a non-finite max: recompute e_j element-wise
                for (int64_t j = tid; j < V; j += kXentThreads) {
                    const float e = det_exp(__fsub_rn(x[j], m));
                    drow[j] = __fmul_rn(__fsub_rn(__fmul_rn(e, inv), j == y ? 1.0f : 0.0f),
                                        dscale);
                }
            }
        }
        __syncthreads();    // bcast / red reuse by the next row
    }
}

// Mean of n floats: 32 chains (groups of 4, plain adds), butterfly, / n.
// The CTA stages blocks of kMeanBlock floats in shared memory with coalesced
// loads; warp 0 then runs the 32 chains over the block. kMeanBlock is a
// multiple of 4 * 32, so a block starts at chain 0 and chain l's groups keep
// their ascending order across blocks.
constexpr int kMeanThreads = 1024;
constexpr int kMeanBlock = 8192;
static_assert(kMeanBlock % (4 * 32) == 0, "blocks start at chain 0");

__global__ void __launch_bounds__(kMeanThreads)
    mean_kernel(int64_t n, const float *__restrict__ v, float *out) {
    __shared__ float buf[kMeanBlock];
    const int tid = threadIdx.x;
    float s = 0.0f;
    for (int64_t base = 0; base < n; base += kMeanBlock) {
        const int cnt = int(n - base < kMeanBlock ? n - base : kMeanBlock);
        __syncthreads();
        for (int i = tid; i < cnt; i += kMeanThreads) buf[i] = v[base + i];
        __syncthreads();
        if (tid < 32) {
            for (int g = tid; 4 * g < cnt; g += 32) {
                const int j0 = 4 * g;
                const int jn = j0 + 4 < cnt ? j0 + 4 : cnt;
                for (int j = j0; j < jn; ++j) s = __fadd_rn(s, buf[j]);
            }
        }
    }
    if (tid < 32) {
        s = warp_butterfly_sum(s);
        if (tid == 0) *out = __fdiv_rn(s, __ll2float_rn(n));
    }
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
    const bool vec = (D % 4 == 0) && (ldx % 4 == 0) && (ldy % 4 == 0) && al16(x) &&
                     al16(y) && al16(gain) && D <= int64_t(kRmsMaxNG) * 128;
    const int64_t blocks = (rows + kRmsWarps - 1) / kRmsWarps;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid{unsigned(blocks)}, block{unsigned(kRmsWarps * 32)};
    if (!vec) {
        rmsnorm_kernel<<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms);
        return cudaGetLastError();
    }
    switch ((D + 127) / 128) {
        case 1: rmsnorm_vec_kernel<1><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 2: rmsnorm_vec_kernel<2><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 3: rmsnorm_vec_kernel<3><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 4: rmsnorm_vec_kernel<4><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 5: rmsnorm_vec_kernel<5><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 6: rmsnorm_vec_kernel<6><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 7: rmsnorm_vec_kernel<7><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        default: rmsnorm_vec_kernel<8><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                        const int32_t *labels, float *loss, float *loss_mean,
                        float *dlogits, int64_t ldd, float dscale, int32_t *dev_status,
                        cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>(rows, int64_t(sm_count_current_device()) * 2);
    xent_kernel<<<unsigned(grid), kXentThreads, 0, s>>>(rows, V, logits, ld, labels, loss,
                                                        dlogits, ldd, dscale, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !loss_mean) return e;
    mean_kernel<<<1, kMeanThreads, 0, s>>>(rows, loss, loss_mean);
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
