// shardsum.cu -- the fixed-order sum of gathered shard gradients, for sm_103a.
//
// What it computes ("MojoLearn 162M" model card, table "Training": 64 logical
// shards, each a mean over 4 x 2,048 tokens, their gradients summed in a fixed
// order; profile v1 reads the order as left to right over the shard index):
//   out[i] = scale * (((g_0[i] + g_1[i]) + g_2[i]) + ... + g_{S-1}[i])
// with one rounding per addition and one multiply. The shards are whatever an
// unreduced gather left in one buffer (shard s at shards + s * ld); a
// collective's own reduction is never used, since its order is not the
// profile's.
//
// Design for GB300: HBM-bound (4 S bytes read and 4 written an element). A
// persistent grid of 8 CTAs an SM walks float4 columns; each thread issues the
// loads of 8 shards before it adds them in order, so ~256 KB of loads an SM
// stay in flight, and the adds run on packed f32x2 pairs (each half rounded
// as the scalar add). Rows that are not 16-byte aligned take a scalar kernel
// with the same order.
#include <algorithm>

#include "det_internal.cuh"

namespace det {
namespace {

constexpr int kSumAhead = 8;     // shards loaded before their adds

__global__ void __launch_bounds__(256)
    shardsum_vec_kernel(int64_t nshards, int64_t n4, const float4 *__restrict__ g,
                        int64_t ld4, float scale, float4 *out) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float4 v0 = __ldcs(g + i);
        f32x2 lo = pack2(v0.x, v0.y), hi = pack2(v0.z, v0.w);
        for (int64_t s0 = 1; s0 < nshards; s0 += kSumAhead) {
            float4 v[kSumAhead];
#pragma unroll
            for (int k = 0; k < kSumAhead; ++k)
                if (s0 + k < nshards) v[k] = __ldcs(g + (s0 + k) * ld4 + i);
#pragma unroll
            for (int k = 0; k < kSumAhead; ++k) {
                if (s0 + k < nshards) {
                    lo = add2(lo, pack2(v[k].x, v[k].y));
                    hi = add2(hi, pack2(v[k].z, v[k].w));
                }
            }
        }
        float4 o;
        unpack2(lo, o.x, o.y);
        unpack2(hi, o.z, o.w);
        o = make_float4(__fmul_rn(o.x, scale), __fmul_rn(o.y, scale),
                        __fmul_rn(o.z, scale), __fmul_rn(o.w, scale));
        __stcs(out + i, o);
    }
}

__global__ void __launch_bounds__(256)
    shardsum_kernel(int64_t nshards, int64_t n, const float *__restrict__ g, int64_t ld,
                    float scale, float *out) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        float t = g[i];
        for (int64_t s = 1; s < nshards; ++s) t = __fadd_rn(t, g[s * ld + i]);
        out[i] = __fmul_rn(t, scale);
    }
}

}  // namespace

cudaError_t launch_shardsum(int64_t nshards, int64_t n, const float *shards, int64_t ld,
                            float scale, float *out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int64_t cap = int64_t(sm_count_current_device()) * 8;
    const bool vec = n % 4 == 0 && ld % 4 == 0 &&
                     reinterpret_cast<uintptr_t>(shards) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(out) % 16 == 0;
    if (vec) {
        const int64_t n4 = n / 4;
        const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256, cap));
        shardsum_vec_kernel<<<unsigned(blocks), 256, 0, s>>>(
            nshards, n4, reinterpret_cast<const float4 *>(shards), ld / 4, scale,
            reinterpret_cast<float4 *>(out));
    } else {
        const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, cap));
        shardsum_kernel<<<unsigned(blocks), 256, 0, s>>>(nshards, n, shards, ld, scale, out);
    }
    return cudaGetLastError();
}

}  // namespace det
