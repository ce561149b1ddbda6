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
// exp for arguments d <= 0 (or -inf), never NaN, without branches: the same
// bits as det_exp(d) whenever the returned n satisfies n >= -125; otherwise the
// caller must use det_exp(d). n = rint(t) is formed as (t + 1.5 2^23) -
// 1.5 2^23, which rounds t to an integer with ties to even for |t| < 2^22; it
// can differ from rintf only in the sign of a zero n, which reaches the
// result only through r = d - n ln2 and the polynomial's products with r,
// where it is inert. For n >= -125 the scaling p 2^n is exact and is done on
// the exponent bits.
constexpr float kRoundMagic = 0x1.8p23f;

__device__ __forceinline__ float exp_le0_fast(float d, int &ni) {
    const float t = __fmul_rn(d, kLog2e);
    const float tm = __fadd_rn(t, kRoundMagic);
    ni = __float_as_int(tm) - __float_as_int(kRoundMagic);
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

// The general exp as an out-of-line call, for the rarely taken paths of the
// cross-entropy (deep underflow, -inf, non-finite maxima), so they cost no
// registers in the hot loops.
__device__ __noinline__ float det_exp_call(float x) { return det_exp(x); }

// The profile's row max: NaN if any element is NaN, else the largest (ties
// between +0 and -0 are bit-inert for the loss and dlogits).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
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
__device__ __forceinline__ void st4_policy(float *p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_policy(float *p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol)
                 : "memory");
}

// One 256-thread CTA per row at a time (thread l = chain l of the 256-chain
// profile), a persistent grid of two CTAs an SM so a row's re-reads hit L2.
// Rows of 50,257 floats start anywhere mod 16 bytes; each row is processed by
// xent_row<H> with its misalignment H (elements) known at compile time.
// Granule q of a row is the 16-byte aligned float4 holding elements
// 4q - H .. 4q + 3 - H; the profile's group g (elements 4g .. 4g+3) is the last
// 4 - H elements of granule g and the first H of granule g + 1.
//  1. m = max over the granules (elements outside the row masked), loads kept
//     in L2 (evict_last);
//  2. chain l loads granule g (g = l, l + 256, ...), computes its 4 exps,
//     stores them to the dlogits row (one 16-byte store where the two rows
//     share their alignment), takes the first H exps of granule g + 1 from
//     lane l + 1 by shuffles (lane 31 computes them itself) and adds group g's
//     4 exps to its chain in ascending order;
//  3. the butterfly 16..1 by shuffles, 32/64/128 through shared memory; thread
//     0 forms loss = log(S) - (x_y - m);
//  4. d_j = (e_j * (1/S) - [j == y]) * dscale over the dlogits granules.
// Main sweeps have no bounds checks; the first and last granules take a
// checked path with the same arithmetic. Rows with a non-finite max, a bad
// label, or dlogits equal to the logits recompute e_j element-wise instead of
// storing it.
constexpr int kXentThreads = 256;
constexpr int kU = 4;    // independent 16-byte loads a thread keeps in flight
static_assert(kXentThreads == kXentLanes, "one thread per chain");

__device__ __forceinline__ float dl_of(float e, float inv, float dscale) {
    return __fmul_rn(__fmul_rn(e, inv), dscale);        // e * inv - 0 == e * inv
}
__device__ __forceinline__ float dl_of_label(float e, float inv, float dscale) {
    return __fmul_rn(__fsub_rn(__fmul_rn(e, inv), 1.0f), dscale);
}

// exp(v - m) for the 4 lanes of a granule; d <= 0 for every element of a row
// with a finite max. Rare deep-underflow elements take the general routine.
__device__ __forceinline__ float4 exp4(float4 v, float m) {
    const float d0 = __fsub_rn(v.x, m), d1 = __fsub_rn(v.y, m);
    const float d2 = __fsub_rn(v.z, m), d3 = __fsub_rn(v.w, m);
    int n0, n1, n2, n3;
    float4 e;
    e.x = exp_le0_fast(d0, n0);
    e.y = exp_le0_fast(d1, n1);
    e.z = exp_le0_fast(d2, n2);
    e.w = exp_le0_fast(d3, n3);
    if (min(min(n0, n1), min(n2, n3)) < -125) {
        if (n0 < -125) e.x = det_exp_call(d0);
        if (n1 < -125) e.y = det_exp_call(d1);
        if (n2 < -125) e.z = det_exp_call(d2);
        if (n3 < -125) e.w = det_exp_call(d3);
    }
    return e;
}

// The profile's group g (elements 4g .. 4g+3) from granule g (cur) and
// granule g + 1 (nxt): the last 4 - H elements of cur, then the first H of nxt.
template <int H>
__device__ __forceinline__ float4 group_of(float4 cur, float4 nxt) {
    if (H == 0) return cur;
    if (H == 1) return make_float4(cur.y, cur.z, cur.w, nxt.x);
    if (H == 2) return make_float4(cur.z, cur.w, nxt.x, nxt.y);
    return make_float4(cur.w, nxt.x, nxt.y, nxt.z);
}

__device__ __forceinline__ float comp(float4 v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Granule g+1 for lanes 0..30 comes from the next lane; lane 31 loaded it.
template <int H>
__device__ __forceinline__ float4 next_granule(float4 c0, float4 own_next, int lane) {
    float4 c1 = own_next;
    if (H != 0) {
        const float a = __shfl_down_sync(0xffffffffu, c0.x, 1);
        const float b = H > 1 ? __shfl_down_sync(0xffffffffu, c0.y, 1) : 0.f;
        const float d = H > 2 ? __shfl_down_sync(0xffffffffu, c0.z, 1) : 0.f;
        if (lane != 31) c1 = make_float4(a, b, d, 0.f);
    }
    return c1;
}

// A sweep with bounds checks (the first sweep, the row's end, non-finite
// maxima): the same operations as the fast sweep, element by element. Returns
// the updated chain value.
template <int H>
__device__ __noinline__ float xent_checked_sweep(const float *xa, int V, int g, float m,
                                                 bool finite_m, float *drow, bool store_e,
                                                 float s, uint64_t keep) {
    const int lane = threadIdx.x & 31;
    const int ngroups = (V + 3) >> 2;
    float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), own = c0;
    if (4 * g - H < V) c0 = *reinterpret_cast<const float4 *>(xa + 4 * g);
    if (H != 0 && lane == 31 && 4 * (g + 1) - H < V)
        own = *reinterpret_cast<const float4 *>(xa + 4 * (g + 1));
    const float4 v = group_of<H>(c0, next_granule<H>(c0, own, lane));
    if (g < ngroups) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = 4 * g + k;
            if (j < V) {
                const float e = det_exp_call(__fsub_rn(comp(v, k), m));
                s = __fadd_rn(s, e);
                if (store_e) st_policy(drow + j, e, keep);
            }
        }
    }
    (void)finite_m;
    return s;
}

template <int H>
__device__ __noinline__ void xent_row(const float *x, int V, int y, float *drow, bool in_place,
                                         float dscale, float *loss_out, float *red, float *bcast,
                                         uint64_t keep, uint64_t drop) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *xa = x - H;                        // 16-byte aligned
    const int nch = (V + H + 3) >> 2;               // granules touching the row
    const int q_lo = H == 0 ? 0 : 1;                // granules fully inside the row:
    const int q_hi = (V + H) >> 2;                  //   [q_lo, q_hi)
    // 1. m = max (order-free, NaN-propagating)
    float m = x[0];
    for (int q0 = q_lo + tid; q0 < q_hi; q0 += kXentThreads * kU) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int q = q0 + u * kXentThreads;
            if (q < q_hi) v[u] = ld4_policy(xa + 4 * q, keep);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (q0 + u * kXentThreads < q_hi)
                m = max_nan(m, max_nan(max_nan(v[u].x, v[u].y), max_nan(v[u].z, v[u].w)));
    }
    if (tid < 2) {      // the partial granules at the two ends
        const int q = tid == 0 ? 0 : q_hi;
        if ((tid == 0 && q_lo == 1) || (tid == 1 && q_hi < nch && q_hi >= q_lo)) {
            const float4 v = *reinterpret_cast<const float4 *>(xa + 4 * q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * q - H + i;
                if (j >= 0 && j < V) m = max_nan(m, comp(v, i));
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = max_nan(__shfl_xor_sync(0xffffffffu, m, off), m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (tid == 0) {
        float mm = red[0];
        for (int w = 1; w < kXentThreads / 32; ++w) mm = max_nan(red[w], mm);
        *bcast = mm;
    }
    __syncthreads();
    m = *bcast;
    const bool finite_m = fabsf(m) <= 3.402823466e38f;     // false for NaN / inf
    const bool store_e = drow != nullptr && !in_place && finite_m;
    const int hd = drow ? int((reinterpret_cast<uintptr_t>(drow) >> 2) & 3) : 0;
    float *da = drow ? drow - hd : nullptr;          // 16-byte aligned dlogits row

    // 2. chain sums: sweep t covers groups g = tid + 256 t
    float s = 0.0f;
    const int ngroups = (V + 3) >> 2;
    const int t_all = (ngroups + kXentThreads - 1) / kXentThreads;
    // sweeps 1 .. t_fast-1 have every group full and inside the row
    const int t_fast = finite_m ? (V >> 2) / kXentThreads : 0;
    s = xent_checked_sweep<H>(xa, V, tid, m, finite_m, drow, store_e, s, keep);
    for (int t = 1; t < t_fast; ++t) {
        const int g = tid + t * kXentThreads;
        const float4 c0 = ld4_policy(xa + 4 * g, drop);
        float4 own = make_float4(0.f, 0.f, 0.f, 0.f);
        if (H != 0 && lane == 31) own = ld4_policy(xa + 4 * (g + 1), drop);
        const float4 v = group_of<H>(c0, next_granule<H>(c0, own, lane));
        const float4 e = exp4(v, m);
        s = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(s, e.x), e.y), e.z), e.w);
        if (store_e) {
            float *dp = drow + 4 * g;
            st_policy(dp, e.x, keep); st_policy(dp + 1, e.y, keep);
            st_policy(dp + 2, e.z, keep); st_policy(dp + 3, e.w, keep);
        }
    }
    for (int t = t_fast < 1 ? 1 : t_fast; t < t_all; ++t)
        s = xent_checked_sweep<H>(xa, V, tid + t * kXentThreads, m, finite_m, drow, store_e, s,
                                  keep);
    // 3. butterfly: 16..1 in the warp, then 32, 64, 128 across warps
    s = warp_butterfly_sum(s);
    __syncthreads();    // red[] reuse
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (tid == 0) {
        const float a01 = __fadd_rn(red[0], red[1]), a23 = __fadd_rn(red[2], red[3]);
        const float a45 = __fadd_rn(red[4], red[5]), a67 = __fadd_rn(red[6], red[7]);
        const float S = __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67));
        *bcast = S;
        *loss_out = __fsub_rn(det_log(S), __fsub_rn(x[y], m));
    }
    __syncthreads();
    // 4. dlogits
    if (drow) {
        const float inv = __fdiv_rn(1.0f, *bcast);
        if (store_e) {
            const int dq_lo = hd == 0 ? 0 : 1, dq_hi = (V + hd) >> 2, dch = (V + hd + 3) >> 2;
            for (int q0 = dq_lo + tid; q0 < dq_hi; q0 += kXentThreads * kU) {
                float4 es[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int q = q0 + u * kXentThreads;
                    if (q < dq_hi) es[u] = ld4_policy(da + 4 * q, drop);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int q = q0 + u * kXentThreads;
                    if (q >= dq_hi) break;
                    const float4 e = es[u];
                    float4 o = make_float4(dl_of(e.x, inv, dscale), dl_of(e.y, inv, dscale),
                                           dl_of(e.z, inv, dscale), dl_of(e.w, inv, dscale));
                    const unsigned k = unsigned(y - (4 * q - hd));
                    if (k < 4) {      // the label's element: rare
                        if (k == 0) o.x = dl_of_label(e.x, inv, dscale);
                        if (k == 1) o.y = dl_of_label(e.y, inv, dscale);
                        if (k == 2) o.z = dl_of_label(e.z, inv, dscale);
                        if (k == 3) o.w = dl_of_label(e.w, inv, dscale);
                    }
                    __stcs(reinterpret_cast<float4 *>(da + 4 * q), o);
                }
            }
            if (tid < 2) {    // the partial granules at the two ends
                const int q = tid == 0 ? 0 : dq_hi;
                if ((tid == 0 && dq_lo == 1) || (tid == 1 && dq_hi < dch && dq_hi >= dq_lo)) {
                    for (int i = 0; i < 4; ++i) {
                        const int j = 4 * q - hd + i;
                        if (j >= 0 && j < V) {
                            const float e = drow[j];
                            drow[j] = j == y ? dl_of_label(e, inv, dscale) : dl_of(e, inv, dscale);
                        }
                    }
                }
            }
        } else {
            // in place, or a non-finite max: recompute e_j element-wise
            for (int j = tid; j < V; j += kXentThreads) {
                const float e = det_exp_call(__fsub_rn(x[j], m));
                drow[j] = __fmul_rn(__fsub_rn(__fmul_rn(e, inv), j == y ? 1.0f : 0.0f), dscale);
            }
        }
    }
    __syncthreads();    // bcast / red reuse by the next row
}

__global__ void __launch_bounds__(kXentThreads, 2)
    xent_kernel(int64_t rows, int64_t V, const float *logits, int64_t ld,
                const int32_t *__restrict__ labels, float *__restrict__ loss,
                float *dlogits, int64_t ldd, float dscale, int32_t *dev_status) {
    __shared__ float red[kXentThreads / 32];
    __shared__ float bcast;
    const int tid = threadIdx.x;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t drop = l2_policy_evict_first();
    const bool in_place = dlogits != nullptr && dlogits == logits;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const float *x = logits + row * ld;
        const int64_t y = labels[row];
        float *drow = dlogits ? dlogits + row * ldd : nullptr;
        if (y < 0 || y >= V) {
            if (tid == 0) {
                loss[row] = __uint_as_float(0x7fc00000u);
                if (dev_status) atomicOr(reinterpret_cast<int *>(dev_status), 1);
            }
            if (drow)
                for (int64_t j = tid; j < V; j += kXentThreads) drow[j] = __uint_as_float(0x7fc00000u);
            continue;   // uniform across the CTA
        }
        switch (int((reinterpret_cast<uintptr_t>(x) >> 2) & 3)) {
            case 0: xent_row<0>(x, int(V), int(y), drow, in_place, dscale, loss + row, red, &bcast, keep, drop); break;
            case 1: xent_row<1>(x, int(V), int(y), drow, in_place, dscale, loss + row, red, &bcast, keep, drop); break;
            case 2: xent_row<2>(x, int(V), int(y), drow, in_place, dscale, loss + row, red, &bcast, keep, drop); break;
            default: xent_row<3>(x, int(V), int(y), drow, in_place, dscale, loss + row, red, &bcast, keep, drop); break;
        }
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
