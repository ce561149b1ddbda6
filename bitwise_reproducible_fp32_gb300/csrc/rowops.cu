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
#include "det_math.cuh"

namespace det {
namespace {

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

template <int NG, int RPW>
__global__ void __launch_bounds__(kRmsWarps * 32, 4)
    rmsnorm_vec_kernel(int64_t rows, int64_t D, const float *__restrict__ x, int64_t ldx,
                       const float *__restrict__ gain, float eps, float *__restrict__ y,
                       int64_t ldy, float *__restrict__ inv_rms) {
    // RPW rows a warp: every row's loads are issued before any is used
    const int lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t(blockIdx.x) * kRmsWarps + (threadIdx.x >> 5)) * RPW;
    const int ngroups = int(D >> 2);
    float4 v[RPW][NG];
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
        if (row0 + q >= rows) break;
        const float4 *xr = reinterpret_cast<const float4 *>(x + (row0 + q) * ldx);
#pragma unroll
        for (int t = 0; t < NG; ++t) {
            const int g = lane + 32 * t;
            if (g < ngroups) v[q][t] = __ldcs(xr + g);
        }
    }
    const float4 *g4 = reinterpret_cast<const float4 *>(gain);
    const float Df = __ll2float_rn(D);
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
        const int64_t row = row0 + q;
        if (row >= rows) break;
        float s = 0.0f;
#pragma unroll
        for (int t = 0; t < NG; ++t) {
            if (lane + 32 * t < ngroups) {
                s = __fmaf_rn(v[q][t].x, v[q][t].x, s);
                s = __fmaf_rn(v[q][t].y, v[q][t].y, s);
                s = __fmaf_rn(v[q][t].z, v[q][t].z, s);
                s = __fmaf_rn(v[q][t].w, v[q][t].w, s);
            }
        }
        const float ss = warp_butterfly_sum(s);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Df), eps)));
        float4 *yr = reinterpret_cast<float4 *>(y + row * ldy);
#pragma unroll
        for (int t = 0; t < NG; ++t) {
            const int g = lane + 32 * t;
            if (g < ngroups) {
                const float4 gg = __ldg(g4 + g);
                float4 o;
                o.x = __fmul_rn(__fmul_rn(v[q][t].x, r), gg.x);
                o.y = __fmul_rn(__fmul_rn(v[q][t].y, r), gg.y);
                o.z = __fmul_rn(__fmul_rn(v[q][t].z, r), gg.z);
                o.w = __fmul_rn(__fmul_rn(v[q][t].w, r), gg.w);
                __stcs(yr + g, o);
            }
        }
        if (inv_rms && lane == 0) inv_rms[row] = r;
    }
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
constexpr int kP = 4;    // chain-pass sweeps loaded ahead
static_assert(kXentThreads == kXentLanes, "one thread per chain");

__device__ __forceinline__ float dl_of(float e, float inv, float dscale) {
    return __fmul_rn(__fmul_rn(e, inv), dscale);        // e * inv - 0 == e * inv
}
__device__ __forceinline__ float dl_of_label(float e, float inv, float dscale) {
    return __fmul_rn(__fsub_rn(__fmul_rn(e, inv), 1.0f), dscale);
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

// Pass 1: this thread's share of the row max over granules (order-free,
// NaN-propagating); the granules fully inside the row are read kU at a time
// and kept in L2 for pass 2.
template <int H>
__device__ __noinline__ float xent_max_part(const float *x, int V, uint64_t keep) {
    const int tid = threadIdx.x;
    const float *xa = x - H;
    const int nch = (V + H + 3) >> 2;
    const int q_lo = H == 0 ? 0 : 1, q_hi = (V + H) >> 2;   // granules inside the row
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
    return m;
}

// Pass 2: chain tid's sum over its groups g = tid + 256 t, storing each e_j to
// drow when store_e.
template <int H>
__device__ __noinline__ float xent_chain(const float *x, int V, float m, bool finite_m,
                                         float *drow, bool store_e, uint64_t keep,
                                         uint64_t drop) {
    const int tid = threadIdx.x, lane = tid & 31;
    const float *xa = x - H;
    float s = 0.0f;
    const int ngroups = (V + 3) >> 2;
    const int t_all = (ngroups + kXentThreads - 1) / kXentThreads;
    // sweeps 1 .. t_fast-1 have every group full and inside the row
    const int t_fast = finite_m ? (V >> 2) / kXentThreads : 0;
    s = xent_checked_sweep<H>(xa, V, tid, m, finite_m, drow, store_e, s, keep);
    // fast sweeps, kP at a time: all their loads are issued before any is used
    for (int t0 = 1; t0 < t_fast; t0 += kP) {
        float4 c0[kP], own[kP];
#pragma unroll
        for (int u = 0; u < kP; ++u) {
            const int g = tid + (t0 + u) * kXentThreads;
            own[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t0 + u < t_fast) {
                c0[u] = ld4_policy(xa + 4 * g, drop);
                if (H != 0 && lane == 31) own[u] = ld4_policy(xa + 4 * (g + 1), drop);
            }
        }
#pragma unroll
        for (int u = 0; u < kP; ++u) {
            if (t0 + u >= t_fast) break;             // uniform across the CTA
            const int g = tid + (t0 + u) * kXentThreads;
            const float4 v = group_of<H>(c0[u], next_granule<H>(c0[u], own[u], lane));
            const float4 e = exp4(v, m);
            s = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(s, e.x), e.y), e.z), e.w);
            if (store_e) {
                float *dp = drow + 4 * g;
                st_policy(dp, e.x, keep); st_policy(dp + 1, e.y, keep);
                st_policy(dp + 2, e.z, keep); st_policy(dp + 3, e.w, keep);
            }
        }
    }
    for (int t = t_fast < 1 ? 1 : t_fast; t < t_all; ++t)
        s = xent_checked_sweep<H>(xa, V, tid + t * kXentThreads, m, finite_m, drow, store_e, s,
                                  keep);
    return s;
}

// Pass 4: d_j = (e_j * inv - [j == y]) * dscale over the dlogits row, reading
// back the e_j that pass 2 stored.
__device__ __noinline__ void xent_dlogits_from_e(float *drow, int V, int y, float inv,
                                                 float dscale, uint64_t drop) {
    const int tid = threadIdx.x;
    const int hd = int((reinterpret_cast<uintptr_t>(drow) >> 2) & 3);
    float *da = drow - hd;                           // 16-byte aligned
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
}

template <int H>
__device__ __forceinline__ void xent_row(const float *x, int V, int y, float *drow, bool in_place,
                                         float dscale, float *loss_out, float *red, float *bcast,
                                         uint64_t keep, uint64_t drop) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // 1. m = max
    float m = xent_max_part<H>(x, V, keep);
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
    // 2. chain sums
    float s = xent_chain<H>(x, V, m, finite_m, drow, store_e, keep, drop);
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
            xent_dlogits_from_e(drow, V, y, inv, dscale, drop);
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

// ---------------------------------------------------------------- cross-entropy, row in shared memory
// For rows that fit in shared memory (V up to ~58,000 floats: the 162M model's
// 50,257-id vocabulary is 201 KB), one 1024-thread CTA per SM keeps the whole
// row on chip, so DRAM sees one read of the logits and one write of dlogits:
//  A. the row's 16-byte granules arrive by TMA bulk copies (two halves, each
//     on its own mbarrier); the next row's halves are copied in while this
//     row's dlogits are written out;
//  B. m = max over the granules (NaN-propagating, elements outside the row
//     masked);
//  C. e = exp(x - m) in place, element-wise, by all 32 warps;
//  D. chains 0..255 add their groups' e values in ascending order from shared
//     memory; butterfly; loss = log(S) - (x_y - m);
//  E. d_j = (e_j (1/S) - [j == y]) dscale, written as 16-byte granules where
//     the dlogits row shares the logits row's alignment.
// The operations and their order are those of the register kernel below.
constexpr int kXsThreads = 1024;
constexpr int kXsMaxGranules = 14400;            // 230,400 bytes of row buffer
constexpr int kXsPiece = 1024;                   // granules per bulk copy (16 KB)
// Row parts, each with its mbarrier: a part is refilled with the next row as
// soon as its dlogits are out. Two measured fastest (three: +1%, four: +3%,
// eight: +8%; each part costs a CTA barrier a row).
constexpr int kXsParts = 2;
// The max, exp and dlogits loops unrolled by two: two granules' loads and
// exps in flight a thread (8192 x 50257: 710 -> 697 us; by four: no better).
constexpr int kXsUnroll = 2;
constexpr int kXsMaxUnroll = 2;
constexpr unsigned kWatchdogXent = 2u;

__device__ unsigned int g_rowops_watchdog;


// Asks L2 to fetch granules [0, n) of the row whose aligned base is xa. Every
// granule holds at least one element of the row, so no byte outside the
// row's pages is touched.
__device__ __forceinline__ void prefetch_granules_l2(const float *xa, int n) {
    for (int q = 0; q < n; q += kXsPiece) {
        const int c = min(kXsPiece, n - q);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(xa + 4 * q),
                     "r"(uint32_t(c) * 16u)
                     : "memory");
    }
}

// Thread 0: copies granules [q0, q1) of the row whose aligned base is xa into
// the same granules of buf, completing on bar.
__device__ __forceinline__ void load_granules(float4 *buf, const float *xa, int q0, int q1,
                                              uint64_t *bar) {
    const uint32_t b = smem_u32(bar);
    mbar_arrive_expect_tx(b, uint32_t(q1 - q0) * 16u);
    for (int q = q0; q < q1; q += kXsPiece) {
        const int n = min(kXsPiece, q1 - q);
        bulk_load(smem_u32(buf + q), xa + 4 * q, uint32_t(n) * 16u, b);
    }
}

// Stage D for a row with misalignment H: chain l (< 256) adds the exps of its
// groups g = l, l + 256, ... in ascending order. Group g is the last 4 - H
// elements of granule g and the first H of granule g + 1; both granules are
// read with 16-byte loads (consecutive chains, consecutive granules: no bank
// conflicts), one sweep ahead of the adds.
// 16-byte load from shared memory by shared-window address: the chain runs in
// an out-of-line function, where a plain pointer would compile to a generic
// load (slower, and tracked as a long-latency access).
__device__ __forceinline__ float4 lds4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds1(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

template <int H>
__device__ __noinline__ float xent_smem_chain(uint32_t buf, int V) {
    const int l = threadIdx.x;
    const int ngroups = (V + 3) >> 2, gfull = V >> 2;
    float s = 0.0f;
    int g = l;
    if (g < gfull) {
        float4 c0 = lds4(buf + 16u * g), c1 = H ? lds4(buf + 16u * (g + 1)) : c0;
        for (; g < gfull; g += kXentLanes) {
            const int gn = g + kXentLanes;
            float4 n0 = c0, n1 = c1;
            if (gn < gfull) {
                n0 = lds4(buf + 16u * gn);
                if (H) n1 = lds4(buf + 16u * (gn + 1));
            }
            const float4 v = group_of<H>(c0, c1);
            s = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(s, v.x), v.y), v.z), v.w);
            c0 = n0;
            c1 = n1;
        }
    }
    if (g < ngroups) {     // the last, partial group
        for (int j = 4 * g; j < V; ++j) s = __fadd_rn(s, lds1(buf + 4u * (j + H)));
    }
    return s;
}

__global__ void __launch_bounds__(kXsThreads, 1)
    xent_smem_kernel(int64_t rows, int V, const float *logits, int64_t ld,
                     const int32_t *__restrict__ labels, float *__restrict__ loss,
                     float *dlogits, int64_t ldd, float dscale, int32_t *dev_status) {
    extern __shared__ float4 buf[];
    __shared__ uint64_t bar[kXsParts];
    __shared__ float red[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int part = ((V + 3) >> 2) / kXsParts;     // granules of parts 0 .. kXsParts-2
    auto part_begin = [&](int pt) { return pt * part; };
    auto part_end = [&](int pt, int n) { return pt + 1 < kXsParts ? (pt + 1) * part : n; };
    auto aligned_row = [&](int64_t r) {
        const float *x = logits + r * ld;
        return x - int((reinterpret_cast<uintptr_t>(x) >> 2) & 3);
    };
    auto granules = [&](int64_t r) {
        const float *x = logits + r * ld;
        return (V + int((reinterpret_cast<uintptr_t>(x) >> 2) & 3) + 3) >> 2;
    };
    if (tid == 0) {
        for (int pt = 0; pt < kXsParts; ++pt) mbar_init(smem_u32(&bar[pt]), 1);
        fence_mbar_init();
        if (int64_t(blockIdx.x) < rows) {
            const int n = granules(blockIdx.x);
            for (int pt = 0; pt < kXsParts; ++pt)
                load_granules(buf, aligned_row(blockIdx.x), part_begin(pt), part_end(pt, n),
                              &bar[pt]);
        }
    }
    __syncthreads();
    int k = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++k) {
        const float *x = logits + row * ld;
        const int h = int((reinterpret_cast<uintptr_t>(x) >> 2) & 3);
        const int nch = (V + h + 3) >> 2;
        const int64_t next = row + gridDim.x;
        const int y32 = labels[row];
        const bool bad = y32 < 0 || y32 >= V;
        const int y = y32;
        float *drow = dlogits ? dlogits + row * ldd : nullptr;
        if (tid == 0 && next < rows) prefetch_granules_l2(aligned_row(next), granules(next));
        // A/B. each part of the row as it lands; its share of the max meanwhile
        float m = x[0];
        bool ok = true;
        for (int hf = 0; hf < kXsParts; ++hf) {
            ok = mbar_wait_bounded(smem_u32(&bar[hf]), uint32_t(k) & 1u) && ok;
            const int q0 = part_begin(hf), q1 = part_end(hf, nch);
            if (!bad && ok) {
                #pragma unroll kXsMaxUnroll
                for (int q = q0 + tid; q < q1; q += kXsThreads) {
                    const float4 v = buf[q];
                    const int j0 = 4 * q - h;
                    if (j0 >= 0 && j0 + 3 < V) {
                        m = max_nan(m, max_nan(max_nan(v.x, v.y), max_nan(v.z, v.w)));
                    } else {
                        if (j0 >= 0 && j0 < V) m = max_nan(m, v.x);
                        if (j0 + 1 >= 0 && j0 + 1 < V) m = max_nan(m, v.y);
                        if (j0 + 2 >= 0 && j0 + 2 < V) m = max_nan(m, v.z);
                        if (j0 + 3 >= 0 && j0 + 3 < V) m = max_nan(m, v.w);
                    }
                }
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&g_rowops_watchdog, kWatchdogXent);
                for (int pt = 0; pt < kXsParts; ++pt)
                    (void)mbar_wait_bounded(smem_u32(&bar[pt]), uint32_t(k) & 1u);
            }
            return;
        }
        float inv = 0.0f;
        bool vec_out = false;
        if (!bad) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = max_nan(__shfl_xor_sync(0xffffffffu, m, off), m);
            if (lane == 0) red[warp] = m;
            __syncthreads();
            // every warp folds the 32 warp maxima itself (the max's order is
            // free: NaN wins, and a +0/-0 tie is bit-inert downstream)
            m = red[lane];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = max_nan(__shfl_xor_sync(0xffffffffu, m, off), m);
            const bool finite_m = fabsf(m) <= 3.402823466e38f;
            // C. e = exp(x - m) in place (elements outside the row are never read)
            if (finite_m) {
#pragma unroll kXsUnroll
                for (int q = tid; q < nch; q += kXsThreads) buf[q] = exp4(buf[q], m);
            } else {
                for (int q = tid; q < nch; q += kXsThreads) {
                    const float4 v = buf[q];
                    buf[q] = make_float4(det_exp_call(__fsub_rn(v.x, m)), det_exp_call(__fsub_rn(v.y, m)),
                                         det_exp_call(__fsub_rn(v.z, m)), det_exp_call(__fsub_rn(v.w, m)));
                }
            }
            __syncthreads();
            // D. the 256 chains, groups g = l, l + 256, ... in ascending order
            if (tid < kXentLanes) {
                float s;
                switch (h) {
                    case 0: s = xent_smem_chain<0>(smem_u32(buf), V); break;
                    case 1: s = xent_smem_chain<1>(smem_u32(buf), V); break;
                    case 2: s = xent_smem_chain<2>(smem_u32(buf), V); break;
                    default: s = xent_smem_chain<3>(smem_u32(buf), V); break;
                }
                s = warp_butterfly_sum(s);
                if (lane == 0) red[warp] = s;
            }
            __syncthreads();
            // every thread folds the 8 chain-warp totals (the same tree)
            const float a01 = __fadd_rn(red[0], red[1]), a23 = __fadd_rn(red[2], red[3]);
            const float a45 = __fadd_rn(red[4], red[5]), a67 = __fadd_rn(red[6], red[7]);
            const float S = __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67));
            if (tid == 0) loss[row] = __fsub_rn(det_log(S), __fsub_rn(x[y], m));
            inv = __fdiv_rn(1.0f, S);
            vec_out = drow != nullptr &&
                      int((reinterpret_cast<uintptr_t>(drow) >> 2) & 3) == h;
        } else {
            if (tid == 0) {
                loss[row] = __uint_as_float(0x7fc00000u);
                if (dev_status) atomicOr(reinterpret_cast<int *>(dev_status), 1);
            }
        }
        const f32x2 inv2 = splat2(inv), dscale2 = splat2(dscale);
        // E. dlogits, part by part; each part's buffer is refilled with the
        // next row as soon as it is free
        for (int hf = 0; hf < kXsParts; ++hf) {
            const int q0 = part_begin(hf), q1 = part_end(hf, nch);
            if (drow) {
                #pragma unroll kXsUnroll
                for (int q = q0 + tid; q < q1; q += kXsThreads) {
                    const int j0 = 4 * q - h;
                    if (bad) {
                        for (int i = 0; i < 4; ++i)
                            if (j0 + i >= 0 && j0 + i < V) drow[j0 + i] = __uint_as_float(0x7fc00000u);
                        continue;
                    }
                    const float4 e = buf[q];
                    float4 o;      // dl_of on both pairs
                    unpack2(mul2(mul2(pack2(e.x, e.y), inv2), dscale2), o.x, o.y);
                    unpack2(mul2(mul2(pack2(e.z, e.w), inv2), dscale2), o.z, o.w);
                    const unsigned kk = unsigned(y - j0);
                    if (kk < 4) {
                        if (kk == 0) o.x = dl_of_label(e.x, inv, dscale);
                        if (kk == 1) o.y = dl_of_label(e.y, inv, dscale);
                        if (kk == 2) o.z = dl_of_label(e.z, inv, dscale);
                        if (kk == 3) o.w = dl_of_label(e.w, inv, dscale);
                    }
                    if (vec_out && j0 >= 0 && j0 + 3 < V) {
                        __stcs(reinterpret_cast<float4 *>(drow + j0), o);
                    } else {
                        if (j0 >= 0 && j0 < V) drow[j0] = o.x;
                        if (j0 + 1 >= 0 && j0 + 1 < V) drow[j0 + 1] = o.y;
                        if (j0 + 2 >= 0 && j0 + 2 < V) drow[j0 + 2] = o.z;
                        if (j0 + 3 >= 0 && j0 + 3 < V) drow[j0 + 3] = o.w;
                    }
                }
            }
            __syncthreads();
            if (tid == 0 && next < rows)
                load_granules(buf, aligned_row(next), part_begin(hf),
                              part_end(hf, granules(next)), &bar[hf]);
        }
    }
}


// ---------------------------------------------------------------- RMSNorm, streamed
// For dense rows (row stride D, 16-byte aligned, D % 4 == 0): one persistent
// CTA per SM takes a contiguous block of rows. A producer lane streams them
// into a ring of shared-memory slots of 4 rows, one 1-D bulk copy a slot
// (many small copies measured slower: 3 KB copies ran at 20 us for the
// 8192 x 768 case, 9 KB copies at 12.4), refilling a slot as soon as its
// rows are released (empty mbarrier, one arrival a row); 16 consumer warps
// each take every 16th row: the 32 chains and the butterfly over the slot,
// then y = (x r) g straight to global memory. Rows are requested in order, so
// the first rows are written while later ones are still arriving. Same
// operations and order as rmsnorm_vec_kernel.
// A consumer's wait on a slot names only the parity of the phase it wants,
// and a wait for phase q passes at once while phase q - 1 is still pending
// (a parity wait cannot tell q from q - 2). So a warp must never wait on a
// slot whose previous copy it has not itself seen land: the 16 consumers form
// 4 groups of 4 (a slot's rows), group g taking the slots' blocks g, g + 4,
// g + 8, ..., and the slot count is a multiple of 4, so the block a slot held
// before block b (block b - S) is one the same warp consumed. (Bulk copies can
// land out of order; with 3-row slots and 16 consumers a warp could reach
// block b while block b - S was still in flight, and read the slot's old
// rows.)
constexpr int kStreamConsumers = 16;
constexpr int kStreamThreads = (kStreamConsumers + 1) * 32;
constexpr int kStreamMaxSlots = 64;
constexpr size_t kStreamSmemBudget = 200 * 1024;
constexpr unsigned kWatchdogRmsNorm = 8u;
constexpr int kRowsPerSlot = 4;            // rows a slot: one bulk copy
constexpr int kStreamGroups = kStreamConsumers / kRowsPerSlot;
static_assert(kStreamConsumers % kRowsPerSlot == 0, "a slot's rows go to one group of warps");
static_assert(kStreamMaxSlots % kStreamGroups == 0, "slot counts are multiples of the groups");

// The ring's slot count for rows of D floats and 1 or 2 inputs: as many as
// the shared-memory budget holds, rounded down to a multiple of the consumer
// groups (0 when fewer than one slot a group fit).
constexpr int stream_slots(int64_t D, int inputs) {
    const int64_t fit = ((int64_t(kStreamSmemBudget) - 256) / (4 * D) - 1) /
                        (int64_t(inputs) * kRowsPerSlot);
    const int64_t s = (fit < kStreamMaxSlots ? fit : kStreamMaxSlots) / kStreamGroups *
                      kStreamGroups;
    return s > 0 ? int(s) : 0;
}

// inputs: 1, or 2 for the fused residual add (a slot then holds a's rows and
// b's rows)
__host__ __device__ constexpr size_t stream_smem(int D, int S, int inputs = 1) {
    return 128 + size_t(inputs * S * kRowsPerSlot + 1) * size_t(D) * 4 + size_t(2 * S + 1) * 8;
}

// With b_in given (the fused residual add), a slot holds the rows of x and of
// b_in (two bulk copies on its mbarrier; both dense with row stride ldx), each
// consumer forms v = x + b_in (one rounding), writes it to xs (row stride
// ldxs) and normalises v: the bits of detadd_f32 followed by detrmsnorm_f32
// on its output.
__global__ void __launch_bounds__(kStreamThreads, 1)
    rmsnorm_stream_kernel(int64_t rows, int D, const float *__restrict__ x, int64_t ldx,
                          const float *__restrict__ gain, float eps, float *__restrict__ y,
                          int64_t ldy, float *__restrict__ inv_rms, int S,
                          const float *__restrict__ b_in, float *__restrict__ xs,
                          int64_t ldxs) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ volatile int abort_flag;
    float4 *gs = reinterpret_cast<float4 *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int ng = D >> 2;
    const int inputs = b_in != nullptr ? 2 : 1;
    float4 *ring = gs + ng;
    float4 *ring_b = ring + size_t(S) * kRowsPerSlot * ng;   // b's rows (fused add)
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + size_t(inputs) * S * kRowsPerSlot * ng);
    uint64_t *empty = full + S;
    uint64_t *gbar = empty + S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = int64_t(blockIdx.x) * per;
    const int n = int(max(int64_t(0), min(per, rows - r0)));
    const int nblk = (n + kRowsPerSlot - 1) / kRowsPerSlot;
    const uint32_t rb = uint32_t(D) * 4u;
    // launched as a programmatic dependent: wait for the previous grid before
    // any global access, then let the next dependent grid's CTAs be placed as
    // this one's retire (each of them waits for this grid in turn)
    grid_dependency_wait();
    allow_dependents();
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(smem_u32(&full[k]), 1);
            mbar_init(smem_u32(&empty[k]), kRowsPerSlot);
        }
        mbar_init(smem_u32(gbar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;
    if (warp == kStreamConsumers) {
        if (lane == 0 && n > 0) {
            mbar_arrive_expect_tx(smem_u32(gbar), rb);
            bulk_load(smem_u32(gs), gain, rb, smem_u32(gbar));
            for (int b = 0; b < nblk; ++b) {
                const int slot = b % S;
                if (b >= S && !mbar_wait_or_abort(smem_u32(&empty[slot]),
                                                  uint32_t(b / S - 1) & 1u, &abort_flag))
                    break;
                const int k = min(kRowsPerSlot, n - b * kRowsPerSlot);
                mbar_arrive_expect_tx(smem_u32(&full[slot]), rb * uint32_t(k) * uint32_t(inputs));
                float4 *dst = ring + size_t(slot) * kRowsPerSlot * ng;
                const int64_t row0 = r0 + int64_t(b) * kRowsPerSlot;
                bulk_load(smem_u32(dst), x + row0 * ldx, rb * uint32_t(k), smem_u32(&full[slot]));
                if (inputs == 2)
                    bulk_load(smem_u32(ring_b + size_t(slot) * kRowsPerSlot * ng),
                              b_in + row0 * ldx, rb * uint32_t(k), smem_u32(&full[slot]));
                issued = b + 1;
            }
        }
    } else if (n > 0 && mbar_wait_or_abort(smem_u32(gbar), 0, &abort_flag)) {
        const float Df = __int2float_rn(D);
        for (int i = warp; i < n; i += kStreamConsumers) {
            const int b = i / kRowsPerSlot, slot = b % S;
            if (!mbar_wait_or_abort(smem_u32(&full[slot]), uint32_t(b / S) & 1u, &abort_flag))
                break;
            const size_t off = (size_t(slot) * kRowsPerSlot + i % kRowsPerSlot) * ng;
            const float4 *xr = ring + off, *br = ring_b + off;
            const int64_t row = r0 + i;
            // the row's values: x, or x + b (written out once)
            auto value = [&](int g) {
                float4 v = xr[g];
                if (inputs == 2) {
                    const float4 u = br[g];
                    v = make_float4(__fadd_rn(v.x, u.x), __fadd_rn(v.y, u.y), __fadd_rn(v.z, u.z),
                                    __fadd_rn(v.w, u.w));
                }
                return v;
            };
            float4 *xsr = inputs == 2 ? reinterpret_cast<float4 *>(xs + row * ldxs) : nullptr;
            float s = 0.0f;
            for (int g = lane; g < ng; g += 32) {
                const float4 v = value(g);
                if (inputs == 2) xsr[g] = v;
                s = __fmaf_rn(v.x, v.x, s);
                s = __fmaf_rn(v.y, v.y, s);
                s = __fmaf_rn(v.z, v.z, s);
                s = __fmaf_rn(v.w, v.w, s);
            }
            const float ss = warp_butterfly_sum(s);
            const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, Df), eps)));
            float4 *yr = reinterpret_cast<float4 *>(y + row * ldy);
            for (int g = lane; g < ng; g += 32) {
                const float4 v = value(g), gg = gs[g];
                __stcs(yr + g, make_float4(__fmul_rn(__fmul_rn(v.x, r), gg.x),
                                           __fmul_rn(__fmul_rn(v.y, r), gg.y),
                                           __fmul_rn(__fmul_rn(v.z, r), gg.z),
                                           __fmul_rn(__fmul_rn(v.w, r), gg.w)));
            }
            if (inv_rms && lane == 0) inv_rms[row] = r;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        }
    }
    __syncthreads();
    if (abort_flag && warp == kStreamConsumers && lane == 0) {
        // a wait gave up: record it, then let every copy still in flight land
        // (or give up on it too) before the shared memory is released
        atomicOr(&g_rowops_watchdog, kWatchdogRmsNorm);
        (void)mbar_wait_bounded(smem_u32(gbar), 0);
        for (int b = max(0, issued - S); b < issued; ++b)
            (void)mbar_wait_bounded(smem_u32(&full[b % S]), uint32_t(b / S) & 1u);
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
    // launched as a programmatic dependent of the kernel that writes v: its
    // launch overlaps that kernel, and this wait returns once that grid has
    // completed and its writes are visible (a plain launch returns at once)
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

cudaError_t rowops_watchdog(unsigned int *code, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_rowops_watchdog, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear && *code) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_rowops_watchdog, &zero, sizeof(unsigned int));
    }
    return e;
}

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
    // streamed: dense aligned rows, D % 4 == 0, and room for a slot a group
    const int S = stream_slots(D, 1);
    if ((D % 4 == 0) && ldx == D && (ldy % 4 == 0) && al16(x) && al16(y) && al16(gain) &&
        S >= kStreamGroups) {
        const size_t smem = stream_smem(int(D), S);
        cudaError_t e = cudaFuncSetAttribute(rmsnorm_stream_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        const int64_t g = std::min<int64_t>(rows, sm_count_current_device());
        return launch_dependent(rmsnorm_stream_kernel, dim3(unsigned(g)), dim3(kStreamThreads),
                                smem, s, rows, int(D), x, ldx, gain, eps, y, ldy, inv_rms, S,
                                static_cast<const float *>(nullptr), static_cast<float *>(nullptr),
                                int64_t(0));
    }
    if (!vec) {
        rmsnorm_kernel<<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms);
        return cudaGetLastError();
    }
    // two rows a warp up to 6 groups a lane (D <= 768), one beyond
    const int64_t blocks2 = (rows + 2 * kRmsWarps - 1) / (2 * kRmsWarps);
    const dim3 grid2{unsigned(blocks2)};
    switch ((D + 127) / 128) {
        case 1: rmsnorm_vec_kernel<1, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 2: rmsnorm_vec_kernel<2, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 3: rmsnorm_vec_kernel<3, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 4: rmsnorm_vec_kernel<4, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 5: rmsnorm_vec_kernel<5, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 6: rmsnorm_vec_kernel<6, 2><<<grid2, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        case 7: rmsnorm_vec_kernel<7, 1><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
        default: rmsnorm_vec_kernel<8, 1><<<grid, block, 0, s>>>(rows, D, x, ldx, gain, eps, y, ldy, inv_rms); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_add_rmsnorm(int64_t rows, int64_t D, const float *a, const float *b,
                               float *x, int64_t ldx, const float *gain, float eps, float *y,
                               int64_t ldy, float *inv_rms, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    auto al16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    const int S = stream_slots(D, 2);
    if ((D % 4 == 0) && (ldx % 4 == 0) && (ldy % 4 == 0) && al16(a) && al16(b) && al16(x) &&
        al16(y) && al16(gain) && S >= kStreamGroups) {
        const size_t smem = stream_smem(int(D), S, 2);
        cudaError_t e = cudaFuncSetAttribute(rmsnorm_stream_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        const int64_t g = std::min<int64_t>(rows, sm_count_current_device());
        return launch_dependent(rmsnorm_stream_kernel, dim3(unsigned(g)), dim3(kStreamThreads),
                                smem, s, rows, int(D), a, D, gain, eps, y, ldy, inv_rms, S, b, x,
                                ldx);
    }
    return cudaErrorNotSupported;   // the caller runs the add and the RMSNorm apart
}

cudaError_t launch_xent(int64_t rows, int64_t V, const float *logits, int64_t ld,
                        const int32_t *labels, float *loss, float *loss_mean,
                        float *dlogits, int64_t ldd, float dscale, int32_t *dev_status,
                        cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t max_granules = (V + 3 + 3) / 4 + 1;
    cudaError_t e;
    if (max_granules <= kXsMaxGranules) {
        const size_t smem = size_t(max_granules) * 16;
        e = cudaFuncSetAttribute(xent_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return e;
        const int64_t grid = std::min<int64_t>(rows, int64_t(sm_count_current_device()));
        xent_smem_kernel<<<unsigned(grid), kXsThreads, smem, s>>>(
            rows, int(V), logits, ld, labels, loss, dlogits, ldd, dscale, dev_status);
    } else {
        const int64_t grid = std::min<int64_t>(rows, int64_t(sm_count_current_device()) * 2);
        xent_kernel<<<unsigned(grid), kXentThreads, 0, s>>>(rows, V, logits, ld, labels, loss,
                                                            dlogits, ldd, dscale, dev_status);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess || !loss_mean) return e;
    // the mean as a programmatic dependent of the row kernel (its launch
    // latency hidden behind the rows; griddepcontrol.wait orders the reads)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kMeanThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mean_kernel, int64_t(rows), static_cast<const float *>(loss),
                           loss_mean);
    if (e != cudaSuccess) return e;
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
