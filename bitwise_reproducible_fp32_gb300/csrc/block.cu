// block.cu -- the rest of a decoder block's forward for sm_103a: SwiGLU's gate,
// the residual add, the causal softmax of attention scores, rotary position
// embedding, and the sin/cos maps.
//
// What each computes (profile v1; "MojoLearn 162M" model card, table
// "Compared with GPT-3 Small": 12 heads of 64, rotary positions with
// theta = 10,000, SwiGLU 2,048 wide, pre-norm residual blocks; the pages fix
// the reduction order and the transcendental spellings but print none):
//   swiglu   h = (g / (1 + exp(-g))) * u
//   add      y = a + b
//   softmax  row r keeps columns j <= (r mod period) + diag of x = s * scale;
//            m = max (NaN-propagating), e = exp(x - m), S = the 256-chain sum
//            folded by the butterfly (the cross-entropy's arrangement),
//            p = e * (1 / S); masked columns +0
//   rope     pairs (2i, 2i+1) of each head turn by a = pos * w_i,
//            w_i = exp(-((2i)/d) * log(theta)): y0 = x0 c - x1 s,
//            y1 = x0 s + x1 c
//
// Design for GB300: all four are HBM-bound. The element-wise ones stream
// float4s through a persistent grid; the softmax takes a row per 256-thread
// CTA (thread l = chain l, the row's 16-byte granules read with float4
// loads when the row allows, three passes hitting L1/L2 after the first);
// the rotary kernel gives a thread one (row, pair) and turns that pair in
// every head, so each angle's sin and cos are formed once.
#include <algorithm>

#include "det_internal.cuh"
#include "det_math.cuh"

namespace det {

// Set when a bounded wait of the bulk-staged causal softmax gave up.
__device__ unsigned int g_block_watchdog;

namespace {

constexpr unsigned kWatchdogSoftmax = 16u;   // det_watchdog_status bit 4

constexpr int kSmaxChains = 32 * 8;       // 8 chains a lane of a warp
static_assert(kSmaxChains == kXentLanes, "the 256 chains of the row reductions");

__global__ void __launch_bounds__(256)
    swiglu_kernel(int64_t n, const float *__restrict__ g, const float *__restrict__ u,
                  float *out, int vec) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    auto one = [](float gv, float uv) {
        const float den = __fadd_rn(1.0f, det_exp(-gv));
        return __fmul_rn(__fdiv_rn(gv, den), uv);
    };
    if (vec) {
        const int64_t n4 = n >> 2;
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += stride) {
            const float4 a = __ldcs(reinterpret_cast<const float4 *>(g) + i);
            const float4 b = __ldcs(reinterpret_cast<const float4 *>(u) + i);
            __stcs(reinterpret_cast<float4 *>(out) + i,
                   make_float4(one(a.x, b.x), one(a.y, b.y), one(a.z, b.z), one(a.w, b.w)));
        }
        for (int64_t i = 4 * n4 + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
             i += stride)
            out[i] = one(g[i], u[i]);
    } else {
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += stride)
            out[i] = one(g[i], u[i]);
    }
}

// SwiGLU backward: silu = g / den, sig = 1 / den, den = 1 + exp(-g);
// d_up = dh silu; d_gate = (dh u) (sig (1 + g (1 - sig))).
__global__ void __launch_bounds__(256)
    swiglu_bwd_kernel(int64_t n, const float *__restrict__ g, const float *__restrict__ u,
                      const float *__restrict__ dh, float *dg, float *du) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float gv = g[i], uv = u[i], d = dh[i];
        const float den = __fadd_rn(1.0f, det_exp(-gv));
        const float silu = __fdiv_rn(gv, den);
        const float sig = __fdiv_rn(1.0f, den);
        const float ds =
            __fmul_rn(sig, __fadd_rn(1.0f, __fmul_rn(gv, __fsub_rn(1.0f, sig))));
        du[i] = __fmul_rn(d, silu);
        dg[i] = __fmul_rn(__fmul_rn(d, uv), ds);
    }
}

__global__ void __launch_bounds__(256)
    add_kernel(int64_t n, const float *__restrict__ a, const float *__restrict__ b,
               float *out, int vec) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    if (vec) {
        const int64_t n4 = n >> 2;
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += stride) {
            const float4 x = __ldcs(reinterpret_cast<const float4 *>(a) + i);
            const float4 y = __ldcs(reinterpret_cast<const float4 *>(b) + i);
            f32x2 lo = add2(pack2(x.x, x.y), pack2(y.x, y.y));
            f32x2 hi = add2(pack2(x.z, x.w), pack2(y.z, y.w));
            float4 o;
            unpack2(lo, o.x, o.y);
            unpack2(hi, o.z, o.w);
            __stcs(reinterpret_cast<float4 *>(out) + i, o);
        }
        for (int64_t i = 4 * n4 + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
             i += stride)
            out[i] = __fadd_rn(a[i], b[i]);
    } else {
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += stride)
            out[i] = __fadd_rn(a[i], b[i]);
    }
}

__device__ __forceinline__ float max_nan2(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float butterfly32(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// The causal-softmax kernels give a row to a warp. Lane l carries chains
// l + 32w (w = 0..7) of the 256, so chain ch still owns the 4-wide groups
// g = ch, ch + 256, ... of the kept columns and adds them in ascending order;
// the 32 chains of each w fold by the butterfly and the 8 totals by the tree
// ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7)), as with a thread a chain
// and a warp per 32 chains. Segment sg of a row is groups 256 sg .. 256 sg +
// 255 (columns 1024 sg ..). The backward holds its first segment of P and dP
// in registers (kSmaxBwdCache) and reads later segments again; the forward
// reads its row in each pass (see there).
constexpr int kSmaxMinBlocks = 4;     // the forward: 56 registers a thread
// The forward stages a row's kept columns in shared memory when they number at
// most kSmaxStage: a lane's slots are the 16-byte groups it reads in every
// pass (groups lane, lane + 32, ...), so no pass waits on another lane.
constexpr int kSmaxStage = 2048;
constexpr int kSmaxBwdCache = 1;
constexpr int kSmaxWarps = 8;

// Kept values of columns j .. j+3 (j a multiple of 4); columns >= nr are not
// read and come back as 0.
__device__ __forceinline__ float4 ld4_kept(const float *r, int64_t j, int64_t nr, bool vec) {
    if (vec && j + 3 < nr) return *reinterpret_cast<const float4 *>(r + j);
    float4 v;
    v.x = j < nr ? r[j] : 0.0f;
    v.y = j + 1 < nr ? r[j + 1] : 0.0f;
    v.z = j + 2 < nr ? r[j + 2] : 0.0f;
    v.w = j + 3 < nr ? r[j + 3] : 0.0f;
    return v;
}

__device__ __forceinline__ void st4_kept(float *r, int64_t j, int64_t nr, bool vec, float4 v) {
    if (vec && j + 3 < nr) {
        *reinterpret_cast<float4 *>(r + j) = v;
        return;
    }
    if (j < nr) r[j] = v.x;
    if (j + 1 < nr) r[j + 1] = v.y;
    if (j + 2 < nr) r[j + 2] = v.z;
    if (j + 3 < nr) r[j + 3] = v.w;
}

// +0 in the masked columns nr .. cols-1 of a row, by the 32 lanes (16-byte
// stores from the first 16-byte boundary at or after nr when vec). Columns
// below nr are never touched.
__device__ __forceinline__ void zero_masked(float *r, int64_t nr, int64_t cols, int lane,
                                            bool vec) {
    if (nr >= cols) return;
    if (!vec) {
        for (int64_t j = nr + lane; j < cols; j += 32) r[j] = 0.0f;
        return;
    }
    const int64_t j4 = ((nr + 3) & ~int64_t(3)) < cols ? ((nr + 3) & ~int64_t(3)) : cols;
    for (int64_t j = nr + lane; j < j4; j += 32) r[j] = 0.0f;
    const int64_t jend = j4 + ((cols - j4) & ~int64_t(3));
    for (int64_t j = j4 + 4 * lane; j < jend; j += 128)
        *reinterpret_cast<float4 *>(r + j) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int64_t j = jend + lane; j < cols; j += 32) r[j] = 0.0f;
}

// Asks L2 to fetch floats [0, n) of a 16-byte aligned row, n a multiple of 4,
// in pieces of at most 16 KB.
__device__ __forceinline__ void prefetch_row_l2(const float *row, int64_t n) {
    for (int64_t q = 0; q < n; q += 4096) {
        const int64_t c = n - q < 4096 ? n - q : 4096;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row + q),
                     "r"(uint32_t(c) * 4u)
                     : "memory");
    }
}

__device__ __forceinline__ float fold_chains(const float (&c)[8]) {
    float t[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) t[w] = butterfly32(c[w]);
    return __fadd_rn(__fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3])),
                     __fadd_rn(__fadd_rn(t[4], t[5]), __fadd_rn(t[6], t[7])));
}

__device__ __forceinline__ int64_t kept_columns(int64_t r, int64_t period, int64_t diag,
                                                int64_t cols) {
    const int64_t nr = (r % period) + diag + 1;
    return nr < 0 ? 0 : (nr > cols ? cols : nr);
}

// Causal softmax: pass 1 the max of x = s * scale (order free), pass 2 the
// chains of exp(x - max), pass 3 p = exp(x - max) * (1 / S). A row of at most
// kSmaxStage kept columns is read from global memory once: pass 1 stores x in
// the warp's shared-memory slots, pass 2 replaces it by the exps, pass 3
// scales them. Longer rows read the row again in each pass (it stays in L1
// between the passes) and form the exps again in pass 3 (the same bits). The
// warp's next row is prefetched into L2. Holding the first 2048 columns in
// registers instead (128 a thread, two CTAs an SM) measured slower than the
// three global passes: 416 against 373 us for 48 x 2048 rows of 2048.
__global__ void __launch_bounds__(32 * kSmaxWarps, kSmaxMinBlocks)
    softmax_causal_kernel(int64_t rows, int64_t cols, const float *s, int64_t lds, float scale,
                          int64_t diag, int64_t period, float *p, int64_t ldp, int vec_s,
                          int vec_p, const int *chunk_zeros) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * kSmaxWarps;
    // With chunk_zeros given and *chunk_zeros == 0, masked columns are zeroed
    // only up to the end of the row's 256-row block of queries: the product
    // that reads P (P V, skipping the +0 chunks past a row block when V is
    // finite, which *chunk_zeros == 0 says) reads no column beyond it.
    const bool to_chunk = chunk_zeros != nullptr && *chunk_zeros == 0;
    extern __shared__ float4 smax_slots[];
    float4 *slots = smax_slots + (threadIdx.x >> 5) * (kSmaxStage / 4);
    for (int64_t r = int64_t(blockIdx.x) * kSmaxWarps + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const float *sr = s + r * lds;
        float *pr = p + r * ldp;
        const int64_t nr = kept_columns(r, period, diag, cols);
        // ask L2 for this warp's next row (its whole 16-byte granules of kept
        // columns), so its loads find it there
        if (vec_s && lane == 0 && r + nwarps < rows) {
            const int64_t rn = r + nwarps;
            prefetch_row_l2(s + rn * lds, kept_columns(rn, period, diag, cols) & ~int64_t(3));
        }
        const int64_t chunk_end = ((r % period) / kKChunk + 1) * kKChunk;
        const int64_t zend = to_chunk && chunk_end < cols ? chunk_end : cols;
        zero_masked(pr, nr, zend, lane, vec_p);
        if (nr == 0) continue;     // uniform across the warp
        if (vec_s && nr <= kSmaxStage) {
            // staged: one read of the row; lane l owns groups l + 32 i
            const int ng = int((nr + 3) / 4);
            float m = __fmul_rn(sr[0], scale);
            for (int g = lane; g < ng; g += 32) {
                float4 v = ld4_kept(sr, 4 * int64_t(g), nr, true);
                v.x = __fmul_rn(v.x, scale); v.y = __fmul_rn(v.y, scale);
                v.z = __fmul_rn(v.z, scale); v.w = __fmul_rn(v.w, scale);
                slots[g] = v;
                const int j = 4 * g;
                if (j < nr) m = max_nan2(m, v.x);
                if (j + 1 < nr) m = max_nan2(m, v.y);
                if (j + 2 < nr) m = max_nan2(m, v.z);
                if (j + 3 < nr) m = max_nan2(m, v.w);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = max_nan2(m, __shfl_xor_sync(0xffffffffu, m, off));
            const bool finite = fabsf(m) <= 0x1.fffffep127f;
            float c[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) c[w] = 0.0f;
            // chain lane + 32 w adds groups lane + 32 w + 256 sg, sg ascending
            for (int sg = 0; 256 * sg < ng; ++sg)
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const int g = lane + 32 * w + 256 * sg;
                    if (g >= ng) continue;
                    const float4 v = slots[g];
                    const float4 e = finite ? exp4(v, m)
                                            : make_float4(det_exp_call(__fsub_rn(v.x, m)),
                                                          det_exp_call(__fsub_rn(v.y, m)),
                                                          det_exp_call(__fsub_rn(v.z, m)),
                                                          det_exp_call(__fsub_rn(v.w, m)));
                    slots[g] = e;
                    const int j = 4 * g;
                    if (j < nr) c[w] = __fadd_rn(c[w], e.x);
                    if (j + 1 < nr) c[w] = __fadd_rn(c[w], e.y);
                    if (j + 2 < nr) c[w] = __fadd_rn(c[w], e.z);
                    if (j + 3 < nr) c[w] = __fadd_rn(c[w], e.w);
                }
            const float inv = __fdiv_rn(1.0f, fold_chains(c));
            for (int g = lane; g < ng; g += 32) {
                const float4 e = slots[g];
                st4_kept(pr, 4 * int64_t(g), nr, vec_p,
                         make_float4(__fmul_rn(e.x, inv), __fmul_rn(e.y, inv),
                                     __fmul_rn(e.z, inv), __fmul_rn(e.w, inv)));
            }
            continue;
        }
        const int64_t nseg = (nr + 1023) / 1024;
        auto scaled = [&](int64_t j) {
            float4 v = ld4_kept(sr, j, nr, vec_s);
            v.x = __fmul_rn(v.x, scale); v.y = __fmul_rn(v.y, scale);
            v.z = __fmul_rn(v.z, scale); v.w = __fmul_rn(v.w, scale);
            return v;
        };
        auto col = [&](int64_t sg, int w) { return 4 * (int64_t(lane) + 32 * w + 256 * sg); };
        // pass 1
        float m = __fmul_rn(sr[0], scale);
        for (int64_t sg = 0; sg < nseg; ++sg)
            for (int w = 0; w < 8; ++w) {
                const int64_t j = col(sg, w);
                const float4 v = scaled(j);
                if (j < nr) m = max_nan2(m, v.x);
                if (j + 1 < nr) m = max_nan2(m, v.y);
                if (j + 2 < nr) m = max_nan2(m, v.z);
                if (j + 3 < nr) m = max_nan2(m, v.w);
            }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            m = max_nan2(m, __shfl_xor_sync(0xffffffffu, m, off));
        // pass 2
        float c[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) c[w] = 0.0f;
        // with a finite max every x - m <= 0: the branch-free exp4 (same bits)
        const bool finite_max = fabsf(m) <= 0x1.fffffep127f;
        auto exps = [&](int64_t j) {
            const float4 v = scaled(j);
            if (finite_max) return exp4(v, m);
            return make_float4(det_exp_call(__fsub_rn(v.x, m)), det_exp_call(__fsub_rn(v.y, m)),
                               det_exp_call(__fsub_rn(v.z, m)), det_exp_call(__fsub_rn(v.w, m)));
        };
        for (int64_t sg = 0; sg < nseg; ++sg)
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int64_t j = col(sg, w);
                const float4 e = exps(j);
                if (j < nr) c[w] = __fadd_rn(c[w], e.x);
                if (j + 1 < nr) c[w] = __fadd_rn(c[w], e.y);
                if (j + 2 < nr) c[w] = __fadd_rn(c[w], e.z);
                if (j + 3 < nr) c[w] = __fadd_rn(c[w], e.w);
            }
        const float inv = __fdiv_rn(1.0f, fold_chains(c));
        // pass 3
        for (int64_t sg = 0; sg < nseg; ++sg)
            for (int w = 0; w < 8; ++w) {
                const int64_t j = col(sg, w);
                const float4 e = exps(j);
                st4_kept(pr, j, nr, vec_p,
                         make_float4(__fmul_rn(e.x, inv), __fmul_rn(e.y, inv),
                                     __fmul_rn(e.z, inv), __fmul_rn(e.w, inv)));
            }
    }
}

// One staged row of the bulk kernel: the passes and every arithmetic step of
// softmax_causal_kernel's staged path (the same bits) on the row's kept
// columns s[0 .. nr) in slots: pass 1 the max of x = s * scale, pass 2a
// e = exp(x - m) into the slots, pass 2b the chains, pass 3 p = e * (1 / S)
// to pr. A lane touches only the groups g = lane (mod 32) in every pass, so
// no pass waits on another lane. The loops over whole groups run without
// per-group conditions (four exps in flight a lane in pass 2a): with the
// conditions inside the unrolled loop the compiler ran the exps one after
// another, and the warps stalled on their dependent steps. The products by
// scale and by 1/S are packed pairs (each half rounded as __fmul_rn).
__device__ __forceinline__ float4 scaled4(float4 v, f32x2 sc2) {
    float4 r;
    unpack2(mul2(pack2(v.x, v.y), sc2), r.x, r.y);
    unpack2(mul2(pack2(v.z, v.w), sc2), r.z, r.w);
    return r;
}
__device__ __forceinline__ void softmax_row_from_slots(float4 *slots, int64_t nr, float *pr,
                                                       float scale, int lane, bool vec_p) {
    const int ng = int((nr + 3) / 4);     // groups holding a kept column
    const int nfull = int(nr / 4);        // groups of 4 kept columns
    const f32x2 sc2 = splat2(scale);
    // pass 1: the max (order free: NaN wins, a +0/-0 tie is bit-inert)
    float m = __fmul_rn(reinterpret_cast<const float *>(slots)[0], scale);
    for (int g = lane; g < nfull; g += 32) {
        const float4 v = scaled4(slots[g], sc2);
        m = max_nan2(m, max_nan2(max_nan2(v.x, v.y), max_nan2(v.z, v.w)));
    }
    if (nfull < ng && lane == (nfull & 31)) {
        const float4 v = scaled4(slots[nfull], sc2);
        const int64_t j = 4 * int64_t(nfull);
        m = max_nan2(m, v.x);
        if (j + 1 < nr) m = max_nan2(m, v.y);
        if (j + 2 < nr) m = max_nan2(m, v.z);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        m = max_nan2(m, __shfl_xor_sync(0xffffffffu, m, off));
    // pass 2a: e = exp(x - m) in place for every group (a partial group's
    // other columns are formed too and never used)
    if (fabsf(m) <= 0x1.fffffep127f) {
        int g = lane;
        for (; g + 96 < ng; g += 128) {
            const float4 v0 = scaled4(slots[g], sc2), v1 = scaled4(slots[g + 32], sc2);
            const float4 v2 = scaled4(slots[g + 64], sc2), v3 = scaled4(slots[g + 96], sc2);
            slots[g] = exp4(v0, m);
            slots[g + 32] = exp4(v1, m);
            slots[g + 64] = exp4(v2, m);
            slots[g + 96] = exp4(v3, m);
        }
        for (; g < ng; g += 32) slots[g] = exp4(scaled4(slots[g], sc2), m);
    } else {
        for (int g = lane; g < ng; g += 32) {
            const float4 v = scaled4(slots[g], sc2);
            slots[g] = make_float4(det_exp_call(__fsub_rn(v.x, m)), det_exp_call(__fsub_rn(v.y, m)),
                                   det_exp_call(__fsub_rn(v.z, m)),
                                   det_exp_call(__fsub_rn(v.w, m)));
        }
    }
    // pass 2b: chain lane + 32 w adds groups lane + 32 w + 256 sg, sg ascending
    float c[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) c[w] = 0.0f;
    int sg = 0;
    for (; 256 * sg + 255 < nfull; ++sg)
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 e = slots[lane + 32 * w + 256 * sg];
            c[w] = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(c[w], e.x), e.y), e.z), e.w);
        }
    for (; 256 * sg < ng; ++sg)
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const int g = lane + 32 * w + 256 * sg;
            if (g >= ng) continue;
            const float4 e = slots[g];
            const int64_t j = 4 * int64_t(g);
            c[w] = __fadd_rn(c[w], e.x);
            if (j + 1 < nr) c[w] = __fadd_rn(c[w], e.y);
            if (j + 2 < nr) c[w] = __fadd_rn(c[w], e.z);
            if (j + 3 < nr) c[w] = __fadd_rn(c[w], e.w);
        }
    const f32x2 inv2 = splat2(__fdiv_rn(1.0f, fold_chains(c)));
    // pass 3: p = e * (1 / S)
    for (int g = lane; g < ng; g += 32)
        st4_kept(pr, 4 * int64_t(g), nr, vec_p, scaled4(slots[g], inv2));
}

// The causal softmax for rows of at most kSmaxStage columns, 16-byte aligned
// (the attention's score rows): each warp keeps two row buffers in shared
// memory, and its lane 0 brings the warp's next row in by one bulk copy
// (cp.async.bulk, completing on the buffer's mbarrier) while the warp works
// on the current one, so a warp's HBM reads are in flight back to back with
// no load instructions of its own. The row's arithmetic is
// softmax_row_from_slots. (Pairs of rows, i and period - 1 - i, a copy of
// about twice the bytes an item, measured 7% slower.) A wait for a copy gives
// up after kWaitLimitNs: the kernel then sets kWatchdogSoftmax, lets its
// copies in flight land (bounded) and returns.
constexpr int kSmaxBulkWarps = 4;    // 64 KB of buffers a block, 3 blocks an SM
constexpr int kSmaxBulkBlocksPerSm = 3;
__global__ void __launch_bounds__(32 * kSmaxBulkWarps)
    softmax_causal_bulk_kernel(int64_t rows, int64_t cols, const float *s, int64_t lds,
                               float scale, int64_t diag, int64_t period, float *p,
                               int64_t ldp, int vec_p, const int *chunk_zeros) {
    extern __shared__ float4 smax_bufs[];
    __shared__ uint64_t sbar[kSmaxBulkWarps][2];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    float4 *bufs = smax_bufs + wib * 2 * (kSmaxStage / 4);
    const uint32_t bar0 = smem_u32(&sbar[wib][0]), bar1 = smem_u32(&sbar[wib][1]);
    const int64_t nwarps = int64_t(gridDim.x) * kSmaxBulkWarps;
    const int64_t first = int64_t(blockIdx.x) * kSmaxBulkWarps + wib;
    const bool to_chunk = chunk_zeros != nullptr && *chunk_zeros == 0;
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // lane 0: row r's kept columns, rounded up to whole 16-byte groups (within
    // the row's cols, a multiple of 4), into buffer b; the proxy fence orders
    // the warp's earlier shared-memory accesses to that buffer before the copy
    auto issue = [&](int64_t r, int b) {
        const int64_t nr = kept_columns(r, period, diag, cols);
        if (nr == 0) return;
        const uint32_t bytes = uint32_t((nr + 3) & ~int64_t(3)) * 4u;
        const uint32_t bar = b ? bar1 : bar0;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(smem_u32(bufs + b * (kSmaxStage / 4)), s + r * lds, bytes, bar);
    };
    if (lane == 0 && first < rows) issue(first, 0);
    uint32_t ph = 0;   // bit b: the parity of the next wait on buffer b
    int k = 0;
    for (int64_t r = first; r < rows; r += nwarps, ++k) {
        const int b = k & 1;
        // the other buffer held the previous row, which the warp is done with
        if (lane == 0 && r + nwarps < rows) issue(r + nwarps, b ^ 1);
        const int64_t nr = kept_columns(r, period, diag, cols);
        float *pr = p + r * ldp;
        if (nr > 0) {
            const bool ok = mbar_wait_bounded(b ? bar1 : bar0, (ph >> b) & 1u);
            ph ^= 1u << b;
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    atomicOr(&g_block_watchdog, kWatchdogSoftmax);
                    (void)mbar_wait_bounded(b ? bar1 : bar0, ((ph >> b) & 1u) ^ 1u);
                    if (r + nwarps < rows && kept_columns(r + nwarps, period, diag, cols) > 0)
                        (void)mbar_wait_bounded(b ? bar0 : bar1, (ph >> (b ^ 1)) & 1u);
                }
                __syncwarp();
                return;
            }
        }
        const int64_t chunk_end = ((r % period) / kKChunk + 1) * kKChunk;
        const int64_t zend = to_chunk && chunk_end < cols ? chunk_end : cols;
        zero_masked(pr, nr, zend, lane, vec_p);
        if (nr > 0)   // uniform across the warp
            softmax_row_from_slots(bufs + b * (kSmaxStage / 4), nr, pr, scale, lane, vec_p);
        __syncwarp();
    }
}

// Softmax backward: dot = the chains of fmaf(dP_j, P_j, .) over the kept
// columns, folded as the forward's sum; dS_j = (P_j (dP_j - dot)) scale;
// masked columns +0. ds may be dp itself (each dS_j is written after dP_j is
// read).
__global__ void __launch_bounds__(32 * kSmaxWarps)
    softmax_causal_bwd_kernel(int64_t rows, int64_t cols, const float *p, const float *dp,
                              int64_t ld, float scale, int64_t diag, int64_t period,
                              float *ds, int64_t ldd, int vec_in, int vec_out) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * kSmaxWarps;
    for (int64_t r = int64_t(blockIdx.x) * kSmaxWarps + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const float *pr = p + r * ld, *dpr = dp + r * ld;
        float *dr = ds + r * ldd;
        const int64_t nr = kept_columns(r, period, diag, cols);
        if (vec_in && lane == 0 && r + nwarps < rows) {
            const int64_t rn = r + nwarps, nn = kept_columns(rn, period, diag, cols) & ~int64_t(3);
            prefetch_row_l2(p + rn * ld, nn);
            prefetch_row_l2(dp + rn * ld, nn);
        }
        zero_masked(dr, nr, cols, lane, vec_out);
        if (nr == 0) continue;
        const int64_t nseg = (nr + 1023) / 1024;
        float4 pc[kSmaxBwdCache][8], dc[kSmaxBwdCache][8];
        auto col = [&](int64_t sg, int w) { return 4 * (int64_t(lane) + 32 * w + 256 * sg); };
        float c[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) c[w] = 0.0f;
        auto chain = [&](float4 pv, float4 dv, int64_t j, float &cw) {
            if (j < nr) cw = __fmaf_rn(dv.x, pv.x, cw);
            if (j + 1 < nr) cw = __fmaf_rn(dv.y, pv.y, cw);
            if (j + 2 < nr) cw = __fmaf_rn(dv.z, pv.z, cw);
            if (j + 3 < nr) cw = __fmaf_rn(dv.w, pv.w, cw);
        };
#pragma unroll
        for (int sg = 0; sg < kSmaxBwdCache; ++sg)
            if (sg < nseg)
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    pc[sg][w] = ld4_kept(pr, col(sg, w), nr, vec_in);
                    dc[sg][w] = ld4_kept(dpr, col(sg, w), nr, vec_in);
                    chain(pc[sg][w], dc[sg][w], col(sg, w), c[w]);
                }
        for (int64_t sg = kSmaxBwdCache; sg < nseg; ++sg)
#pragma unroll
            for (int w = 0; w < 8; ++w)
                chain(ld4_kept(pr, col(sg, w), nr, vec_in), ld4_kept(dpr, col(sg, w), nr, vec_in),
                      col(sg, w), c[w]);
        const float dot = fold_chains(c);
        auto grad = [&](float4 pv, float4 dv) {
            return make_float4(__fmul_rn(__fmul_rn(pv.x, __fsub_rn(dv.x, dot)), scale),
                               __fmul_rn(__fmul_rn(pv.y, __fsub_rn(dv.y, dot)), scale),
                               __fmul_rn(__fmul_rn(pv.z, __fsub_rn(dv.z, dot)), scale),
                               __fmul_rn(__fmul_rn(pv.w, __fsub_rn(dv.w, dot)), scale));
        };
#pragma unroll
        for (int sg = 0; sg < kSmaxBwdCache; ++sg)
            if (sg < nseg)
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    st4_kept(dr, col(sg, w), nr, vec_out, grad(pc[sg][w], dc[sg][w]));
        for (int64_t sg = kSmaxBwdCache; sg < nseg; ++sg)
            for (int w = 0; w < 8; ++w)
                st4_kept(dr, col(sg, w), nr, vec_out,
                         grad(ld4_kept(pr, col(sg, w), nr, vec_in),
                              ld4_kept(dpr, col(sg, w), nr, vec_in)));
    }
}

// +0 in columns chunk_end .. cols-1 of each row, chunk_end the end of the
// row's 256-row block of queries (what a softmax given chunk_zeros left
// unwritten), when *flag is not 0; nothing otherwise (the kernel reads the
// flag first). A warp a row.
__global__ void __launch_bounds__(256)
    zero_past_chunks_kernel(int64_t rows, int64_t cols, int64_t period, float *p, int64_t ld,
                            const int *flag, int vec) {
    if (*flag == 0) return;
    const int lane = threadIdx.x & 31;
    for (int64_t r = blockIdx.x * 8 + (threadIdx.x >> 5); r < rows;
         r += int64_t(gridDim.x) * 8) {
        const int64_t chunk_end = ((r % period) / kKChunk + 1) * kKChunk;
        if (chunk_end < cols) zero_masked(p + r * ld, chunk_end, cols, lane, vec);
    }
}

// Counts the non-finite values of a rows x cols block (row stride ld) into
// *bad: a warp a row, one atomic add a warp that saw any.
__global__ void __launch_bounds__(256)
    count_nonfinite_kernel(int64_t rows, int64_t cols, const float *base, int64_t ld,
                           int *bad) {
    const int lane = threadIdx.x & 31;
    int found = 0;
    for (int64_t r = blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += int64_t(gridDim.x) * 8) {
        const float *row = base + r * ld;
        for (int64_t c = lane; c < cols; c += 32) found |= !(fabsf(row[c]) <= 0x1.fffffep127f);
    }
    if (__any_sync(0xffffffffu, found) && lane == 0) atomicAdd(bad, 1);
}

// Embedding backward: a CTA per id v. It scans the tokens 256 at a time,
// lists the positions holding v in ascending order (warp ballots and a prefix
// over the 8 warps), and thread j adds the listed gradient rows' column j to
// its running sum in that order, the first as is; +0 for an id no token uses.
// Columns go 1024 at a time, 4 a thread.
__global__ void __launch_bounds__(256)
    embedding_bwd_kernel(int64_t ntok, int64_t dim, const int32_t *__restrict__ tokens,
                         const float *__restrict__ dx, int64_t lddx, int64_t vocab, float *de,
                         int64_t ldde) {
    __shared__ int32_t list[256];
    __shared__ int wcount[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t v = blockIdx.x; v < vocab; v += gridDim.x) {
        for (int64_t j0 = 0; j0 < dim; j0 += 1024) {
            float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            bool first = true;
            for (int64_t k0 = 0; k0 < ntok; k0 += 256) {
                const int64_t k = k0 + tid;
                const bool hit = k < ntok && tokens[k] == v;
                const unsigned m = __ballot_sync(0xffffffffu, hit);
                if (lane == 0) wcount[warp] = __popc(m);
                __syncthreads();
                int before = 0, total = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    before += w < warp ? wcount[w] : 0;
                    total += wcount[w];
                }
                if (hit) list[before + __popc(m & ((1u << lane) - 1u))] = tid;
                __syncthreads();
                for (int i = 0; i < total; ++i) {
                    const float *row = dx + (k0 + list[i]) * lddx;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int64_t j = j0 + tid + 256 * c;
                        if (j < dim) t[c] = first ? row[j] : __fadd_rn(t[c], row[j]);
                    }
                    first = false;
                }
                __syncthreads();   // list and wcount are rewritten next
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int64_t j = j0 + tid + 256 * c;
                if (j < dim) de[v * ldde + j] = t[c];
            }
        }
    }
}

// Thread per (row, pair i): a = pos * w_i, its sin and cos once, then the
// pair turned in every head (by -a for the backward).
__global__ void __launch_bounds__(256)
    rope_kernel(int64_t rows, int heads, int d, float *x, int64_t ldx, int64_t seq,
                float theta, int backward) {
    const int half = d / 2;
    const int64_t total = rows * half;
    const float L = det_log(theta);
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = e / half;
        const int i = int(e - t * half);
        const float pos = float(t % seq);
        const float ex = __fdiv_rn(float(2 * i), float(d));
        const float w = det_exp(__fmul_rn(-ex, L));
        const float a = __fmul_rn(pos, w);
        float sn, cs;
        det_sincos(a, sn, cs);
        float *row = x + t * ldx + 2 * i;
        for (int h = 0; h < heads; ++h) {
            float *q = row + h * d;
            const float x0 = q[0], x1 = q[1];
            if (!backward) {
                q[0] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
                q[1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
            } else {
                q[0] = __fadd_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
                q[1] = __fsub_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
            }
        }
    }
}

// Embedding rows: out[t] = table[token[t]] (copies, exact). A token outside
// [0, vocab) writes a NaN row and sets the caller's status word.
__global__ void __launch_bounds__(256)
    embedding_kernel(int64_t ntok, int64_t dim, const float *table, int64_t ldt, int64_t vocab,
                     const int32_t *tokens, float *out, int64_t ldo, int32_t *status) {
    const int64_t total = ntok * dim;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = e / dim, j = e - t * dim;
        const int64_t id = tokens[t];
        if (id < 0 || id >= vocab) {
            out[t * ldo + j] = __uint_as_float(0x7fc00000u);
            if (status && j == 0) atomicOr(reinterpret_cast<int *>(status), 1);
        } else {
            out[t * ldo + j] = table[id * ldt + j];
        }
    }
}

__global__ void sincos_map_kernel(int64_t n, const float *x, float *y, int want_cos) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        float sn, cs;
        det_sincos(x[i], sn, cs);
        y[i] = want_cos ? cs : sn;
    }
}

int64_t ew_blocks(int64_t n) {
    return std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256,
                                                  int64_t(sm_count_current_device()) * 8));
}
bool al16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

cudaError_t block_watchdog(unsigned int *code, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_block_watchdog, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear && *code) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_block_watchdog, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_swiglu(int64_t n, const float *g, const float *u, float *out,
                          cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int vec = al16(g) && al16(u) && al16(out);
    swiglu_kernel<<<unsigned(ew_blocks(vec ? n / 4 : n)), 256, 0, s>>>(n, g, u, out, vec);
    return cudaGetLastError();
}

cudaError_t launch_add(int64_t n, const float *a, const float *b, float *out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int vec = al16(a) && al16(b) && al16(out);
    add_kernel<<<unsigned(ew_blocks(vec ? n / 4 : n)), 256, 0, s>>>(n, a, b, out, vec);
    return cudaGetLastError();
}

cudaError_t launch_softmax_causal(int64_t rows, int64_t cols, const float *sc, int64_t lds,
                                  float scale, int64_t diag, int64_t period, float *p,
                                  int64_t ldp, cudaStream_t s, const int *chunk_zeros) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((rows + kSmaxWarps - 1) / kSmaxWarps,
                                             int64_t(sm_count_current_device()) * 16);
    const int vec_s = al16(sc) && lds % 4 == 0, vec_p = al16(p) && ldp % 4 == 0;
    if (vec_s && cols <= kSmaxStage && cols % 4 == 0) {
        // every row fits a buffer, and a copy rounded up to whole 16-byte
        // groups stays within the row's columns: the bulk-staged kernel,
        // persistent
        const size_t bsmem = size_t(kSmaxBulkWarps) * 2 * kSmaxStage * 4;
        const int64_t bblocks = std::min<int64_t>(
            (rows + kSmaxBulkWarps - 1) / kSmaxBulkWarps,
            int64_t(sm_count_current_device()) * kSmaxBulkBlocksPerSm);
        cudaError_t eb = cudaFuncSetAttribute(softmax_causal_bulk_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              int(bsmem));
        if (eb != cudaSuccess) return eb;
        softmax_causal_bulk_kernel<<<unsigned(bblocks), 32 * kSmaxBulkWarps, bsmem, s>>>(
            rows, cols, sc, lds, scale, diag, period, p, ldp, vec_p, chunk_zeros);
        return cudaGetLastError();
    }
    const size_t smem = size_t(kSmaxWarps) * kSmaxStage * 4;
    const cudaError_t e = cudaFuncSetAttribute(
        softmax_causal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    softmax_causal_kernel<<<unsigned(blocks), 32 * kSmaxWarps, smem, s>>>(
        rows, cols, sc, lds, scale, diag, period, p, ldp, vec_s, vec_p, chunk_zeros);
    return cudaGetLastError();
}

cudaError_t launch_rope(int64_t rows, int heads, int head_dim, float *x, int64_t ldx,
                        int64_t seq_len, float theta, int backward, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    rope_kernel<<<unsigned(ew_blocks(rows * (head_dim / 2))), 256, 0, s>>>(
        rows, heads, head_dim, x, ldx, seq_len, theta, backward);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(int64_t n, const float *g, const float *u, const float *dh,
                              float *dg, float *du, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    swiglu_bwd_kernel<<<unsigned(ew_blocks(n)), 256, 0, s>>>(n, g, u, dh, dg, du);
    return cudaGetLastError();
}

cudaError_t launch_softmax_causal_bwd(int64_t rows, int64_t cols, const float *p,
                                      const float *dp, int64_t ld, float scale, int64_t diag,
                                      int64_t period, float *ds, int64_t ldd, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((rows + kSmaxWarps - 1) / kSmaxWarps,
                                             int64_t(sm_count_current_device()) * 16);
    const int vec_in = al16(p) && al16(dp) && ld % 4 == 0, vec_out = al16(ds) && ldd % 4 == 0;
    softmax_causal_bwd_kernel<<<unsigned(blocks), 32 * kSmaxWarps, 0, s>>>(
        rows, cols, p, dp, ld, scale, diag, period, ds, ldd, vec_in, vec_out);
    return cudaGetLastError();
}

cudaError_t launch_zero_past_chunks(int64_t rows, int64_t cols, int64_t period, float *p,
                                   int64_t ld, const int *flag, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, int64_t(sm_count_current_device()) * 8);
    const int vec = al16(p) && ld % 4 == 0;
    zero_past_chunks_kernel<<<unsigned(blocks), 256, 0, s>>>(rows, cols, period, p, ld, flag, vec);
    return cudaGetLastError();
}

cudaError_t launch_count_nonfinite(int64_t rows, int64_t cols, const float *base, int64_t ld,
                                   int *bad, cudaStream_t s) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, int64_t(sm_count_current_device()) * 8);
    count_nonfinite_kernel<<<unsigned(blocks), 256, 0, s>>>(rows, cols, base, ld, bad);
    return cudaGetLastError();
}

cudaError_t launch_embedding_bwd(int64_t ntok, int64_t dim, const int32_t *tokens,
                                 const float *dx, int64_t lddx, int64_t vocab, float *de,
                                 int64_t ldde, cudaStream_t s) {
    const int64_t blocks = std::min<int64_t>(vocab, int64_t(sm_count_current_device()) * 8);
    embedding_bwd_kernel<<<unsigned(blocks), 256, 0, s>>>(ntok, dim, tokens, dx, lddx, vocab,
                                                         de, ldde);
    return cudaGetLastError();
}

cudaError_t launch_embedding(int64_t ntok, int64_t dim, const float *table, int64_t ldt,
                             int64_t vocab, const int32_t *tokens, float *out, int64_t ldo,
                             int32_t *status, cudaStream_t s) {
    if (ntok == 0) return cudaSuccess;
    embedding_kernel<<<unsigned(ew_blocks(ntok * dim)), 256, 0, s>>>(ntok, dim, table, ldt,
                                                                     vocab, tokens, out, ldo,
                                                                     status);
    return cudaGetLastError();
}

cudaError_t launch_sincos_map(int64_t n, const float *x, float *y, int want_cos,
                              cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    sincos_map_kernel<<<unsigned(ew_blocks(n)), 256, 0, s>>>(n, x, y, want_cos);
    return cudaGetLastError();
}

}  // namespace det
