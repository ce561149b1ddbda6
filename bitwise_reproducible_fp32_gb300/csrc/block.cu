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
namespace {

constexpr int kSmaxThreads = 256;        // = the 256 chains
static_assert(kSmaxThreads == kXentLanes, "one thread a chain");

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

// One row per CTA, thread l = chain l: chain l owns the 4-element groups
// g = l, l + 256, ... of the kept columns and adds their exps in ascending
// order. Pass 1 the max, pass 2 the chains, pass 3 the probabilities (the
// exps recomputed; rows of an attention batch stay in L1/L2 between passes).
__global__ void __launch_bounds__(kSmaxThreads)
    softmax_causal_kernel(int64_t rows, int64_t cols, const float *s, int64_t lds, float scale,
                          int64_t diag, int64_t period, float *p, int64_t ldp) {
    __shared__ float red[kSmaxThreads / 32];
    const int l = threadIdx.x, lane = l & 31, warp = l >> 5;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *sr = s + r * lds;
        float *pr = p + r * ldp;
        int64_t nr = (r % period) + diag + 1;
        nr = nr < 0 ? 0 : (nr > cols ? cols : nr);
        for (int64_t j = nr + l; j < cols; j += kSmaxThreads) pr[j] = 0.0f;
        if (nr == 0) continue;     // uniform across the CTA
        // pass 1: the max (its order is free)
        float m = __fmul_rn(sr[0], scale);
        for (int64_t j = l; j < nr; j += kSmaxThreads) m = max_nan2(m, __fmul_rn(sr[j], scale));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            m = max_nan2(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int w = 1; w < kSmaxThreads / 32; ++w) m = max_nan2(m, red[w]);
        __syncthreads();
        // pass 2: chain l over its groups, ascending
        float c = 0.0f;
        for (int64_t g = l; 4 * g < nr; g += kSmaxThreads) {
            const int64_t j1 = 4 * g + 4 < nr ? 4 * g + 4 : nr;
            for (int64_t j = 4 * g; j < j1; ++j)
                c = __fadd_rn(c, det_exp(__fsub_rn(__fmul_rn(sr[j], scale), m)));
        }
        c = butterfly32(c);
        if (lane == 0) red[warp] = c;
        __syncthreads();
        const float a01 = __fadd_rn(red[0], red[1]), a23 = __fadd_rn(red[2], red[3]);
        const float a45 = __fadd_rn(red[4], red[5]), a67 = __fadd_rn(red[6], red[7]);
        const float inv = __fdiv_rn(1.0f, __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67)));
        __syncthreads();
        // pass 3: p = e * (1 / S)
        for (int64_t j = l; j < nr; j += kSmaxThreads)
            pr[j] = __fmul_rn(det_exp(__fsub_rn(__fmul_rn(sr[j], scale), m)), inv);
    }
}

// Softmax backward, one row per CTA, thread l = chain l: dot = the 256 chains
// of fmaf(dP_j, P_j, .) over the kept columns, folded like the forward's sum;
// then dS_j = (P_j (dP_j - dot)) scale; masked columns +0.
__global__ void __launch_bounds__(kSmaxThreads)
    softmax_causal_bwd_kernel(int64_t rows, int64_t cols, const float *p, const float *dp,
                              int64_t ld, float scale, int64_t diag, int64_t period,
                              float *ds, int64_t ldd) {
    __shared__ float red[kSmaxThreads / 32];
    const int l = threadIdx.x, lane = l & 31, warp = l >> 5;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *pr = p + r * ld, *dpr = dp + r * ld;
        float *dr = ds + r * ldd;
        int64_t nr = (r % period) + diag + 1;
        nr = nr < 0 ? 0 : (nr > cols ? cols : nr);
        for (int64_t j = nr + l; j < cols; j += kSmaxThreads) dr[j] = 0.0f;
        if (nr == 0) continue;
        float c = 0.0f;
        for (int64_t g = l; 4 * g < nr; g += kSmaxThreads) {
            const int64_t j1 = 4 * g + 4 < nr ? 4 * g + 4 : nr;
            for (int64_t j = 4 * g; j < j1; ++j) c = __fmaf_rn(dpr[j], pr[j], c);
        }
        c = butterfly32(c);
        if (lane == 0) red[warp] = c;
        __syncthreads();
        const float a01 = __fadd_rn(red[0], red[1]), a23 = __fadd_rn(red[2], red[3]);
        const float a45 = __fadd_rn(red[4], red[5]), a67 = __fadd_rn(red[6], red[7]);
        const float dot = __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67));
        __syncthreads();
        for (int64_t j = l; j < nr; j += kSmaxThreads)
            dr[j] = __fmul_rn(__fmul_rn(pr[j], __fsub_rn(dpr[j], dot)), scale);
    }
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
                                  int64_t ldp, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>(rows, int64_t(sm_count_current_device()) * 8);
    softmax_causal_kernel<<<unsigned(blocks), kSmaxThreads, 0, s>>>(rows, cols, sc, lds, scale,
                                                                   diag, period, p, ldp);
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
    const int64_t blocks = std::min<int64_t>(rows, int64_t(sm_count_current_device()) * 8);
    softmax_causal_bwd_kernel<<<unsigned(blocks), kSmaxThreads, 0, s>>>(
        rows, cols, p, dp, ld, scale, diag, period, ds, ldd);
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
