// gemm.cu -- fixed-order FP32 GEMM on CUDA-core FFMA for sm_103a.
//
// What it computes ("mojolearn" PyPI page, section "What bitwise identity
// means, and why it is not the default": reduction order, partitioning and FMA
// policy are fixed by the profile; "MojoLearn 162M" model card, table
// "Compared with GPT-3 Small", for the shapes): every C[i,j] is, for each
// 256-wide chunk of k, a sequential fmaf chain from +0 in ascending k, and the
// chunk partials are added left to right. Each output element belongs to one
// thread for the whole of K, so the chain is exactly the thread's accumulator
// sequence, whatever the tiling.
//
// Why CUDA cores and not tcgen05: a tensor-core FP32 product (TF32 or split
// bf16 emulation) rounds differently from a chain of fmaf, so the profile's
// bits require FFMA.
//
// Design for GB300:
//  * CTA tile 128 x 128, k-tile 32 (divides the 256-wide chunk, so chunk
//    boundaries fall on k-tile boundaries), 256 threads, 8 x 8 outputs per
//    thread, one CTA per SM (up to 255 registers a thread).
//  * Operand tiles arrive by TMA (cp.async.bulk.tensor) into a 4-stage ring
//    with one mbarrier per stage; thread 0 is the producer. Tiles whose k is
//    the contiguous dimension use the 128-byte swizzle, so 16-byte shared loads
//    of 4 consecutive k for 8 different rows are bank-conflict free; tiles
//    whose m/n is contiguous are stored plain and read as float4 along m/n.
//  * Per 4-wide k group a thread issues 16 LDS.128 and 256 FFMA (6% of issue).
//  * Chunk partials: the running left-to-right total lives in shared memory
//    (64 KB), touched once per 256 k, which keeps registers for the operand
//    fragments.
//  * Operands whose base or row stride is not 16-byte aligned (TMA cannot
//    describe them) take the same kernel with a plain-load producer; the
//    arithmetic, and so the bits, are identical.
//  * Tile order: the dimension whose operand is smaller runs fastest, so the
//    smaller operand stays resident in the 129 MB L2 and the larger one
//    streams from HBM once.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "det_internal.cuh"

namespace det {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 32;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int TILES_PER_CHUNK = kKChunk / BK;   // 8
constexpr int TILE_FLOATS = BM * BK;            // 4096 (BN == BM)
constexpr int STAGE_FLOATS = 2 * TILE_FLOATS;   // A tile then B tile
constexpr int TOTAL_FLOAT4 = THREADS * 16;      // 64 running totals a thread
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_FLOATS * 4 +
                              size_t(TOTAL_FLOAT4) * 16 + STAGES * 8;
static_assert(kKChunk % BK == 0, "chunk boundaries must fall on k-tiles");

__device__ unsigned int g_gemm_watchdog;

// Shared-memory float index of element (row r, k) of a 128 x 32 operand tile.
// KMAJ: rows of 32 k (128 bytes), 16-byte chunk q of row r stored at chunk
// q ^ (r & 7) -- the TMA 128-byte swizzle pattern. Otherwise: rows of 128
// m/n values for each k.
template <bool KMAJ>
__device__ __forceinline__ int tile_idx(int r, int k) {
    if (KMAJ) return r * 32 + ((((k >> 2) ^ (r & 7)) << 2) | (k & 3));
    return k * 128 + r;
}

struct KArgs {
    int M, N, K;
    int64_t lda, ldb, ldc;
    const float *A, *B;
    float *C;
    int mt, nt;        // tiles along M and N
    int m_fast;        // tile order
    int vec_store;     // C rows 16-byte aligned
};

// Loads the operand fragments of k group q (k = 4q .. 4q+3 of the tile) and
// runs the 256 FFMAs: acc[r][c] = fmaf(a[r][kk], b[c][kk], acc[r][c]) for
// kk ascending.
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void mma_group(const float *__restrict__ As,
                                          const float *__restrict__ Bs, int q,
                                          int arow, int bcol, int lm, int ln,
                                          float (&acc)[8][8]) {
    float a[8][4], b[8][4];
    if (A_KM) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float4 v = *reinterpret_cast<const float4 *>(
                As + (arow + 8 * r) * 32 + ((q ^ lm) << 2));
            a[r][0] = v.x; a[r][1] = v.y; a[r][2] = v.z; a[r][3] = v.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *p = As + (4 * q + kk) * 128 + arow;
            const float4 lo = *reinterpret_cast<const float4 *>(p);
            const float4 hi = *reinterpret_cast<const float4 *>(p + 32);
            a[0][kk] = lo.x; a[1][kk] = lo.y; a[2][kk] = lo.z; a[3][kk] = lo.w;
            a[4][kk] = hi.x; a[5][kk] = hi.y; a[6][kk] = hi.z; a[7][kk] = hi.w;
        }
    }
    if (B_KM) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int sw = ln + 4 * (c & 1);          // (bcol + 4c) & 7
            const float4 v = *reinterpret_cast<const float4 *>(
                Bs + (bcol + 4 * c) * 32 + ((q ^ sw) << 2));
            b[c][0] = v.x; b[c][1] = v.y; b[c][2] = v.z; b[c][3] = v.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *p = Bs + (4 * q + kk) * 128 + bcol;
            const float4 lo = *reinterpret_cast<const float4 *>(p);
            const float4 hi = *reinterpret_cast<const float4 *>(p + 16);
            b[0][kk] = lo.x; b[1][kk] = lo.y; b[2][kk] = lo.z; b[3][kk] = lo.w;
            b[4][kk] = hi.x; b[5][kk] = hi.y; b[6][kk] = hi.z; b[7][kk] = hi.w;
        }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[r][c] = __fmaf_rn(a[r][kk], b[c][kk], acc[r][c]);
}

// The last k-tile when K is not a multiple of 32: k ascending up to kcount.
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void mma_partial(const float *__restrict__ As,
                                         const float *__restrict__ Bs, int kcount,
                                         const int (&rows)[8], const int (&cols)[8],
                                         float (&acc)[8][8]) {
    for (int k = 0; k < kcount; ++k) {
        float a[8], b[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) a[r] = As[tile_idx<A_KM>(rows[r], k)];
#pragma unroll
        for (int c = 0; c < 8; ++c) b[c] = Bs[tile_idx<B_KM>(cols[c], k)];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[r][c] = __fmaf_rn(a[r], b[c], acc[r][c]);
    }
}

// Plain-load producer: the whole CTA copies one 128 x 32 tile into the same
// layout TMA would produce, zero-filling outside the matrix.
template <bool KMAJ>
__device__ __forceinline__ void load_tile_plain(float *dst, const float *src,
                                                int64_t ld, int rows_total,
                                                int k_total, int r0, int k0,
                                                int tid) {
#pragma unroll 4
    for (int e = tid; e < TILE_FLOATS; e += THREADS) {
        int r, k;
        if (KMAJ) { r = e >> 5; k = e & 31; }        // consecutive threads: consecutive k
        else      { k = e >> 7; r = e & 127; }       // consecutive threads: consecutive m/n
        const int gr = r0 + r, gk = k0 + k;
        float v = 0.0f;
        if (gr < rows_total && gk < k_total)
            v = KMAJ ? src[int64_t(gr) * ld + gk] : src[int64_t(gk) * ld + gr];
        dst[tile_idx<KMAJ>(r, k)] = v;
    }
}

template <bool A_KM, bool B_KM, bool TMA>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB, const KArgs p) {
    extern __shared__ unsigned char smem_raw[];
    float *smem = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *stages = smem;
    float4 *totals = reinterpret_cast<float4 *>(smem + STAGES * STAGE_FLOATS);
    uint64_t *full = reinterpret_cast<uint64_t *>(totals + TOTAL_FLOAT4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;
    const int lm = lane >> 2, ln = lane & 3;

    int mb, nb;
    if (p.m_fast) { mb = blockIdx.x % p.mt; nb = blockIdx.x / p.mt; }
    else          { nb = blockIdx.x % p.nt; mb = blockIdx.x / p.nt; }
    const int m0 = mb * BM, n0 = nb * BN;

    // the thread's 8 rows of op(A) and 8 columns of op(B), tile-relative
    const int arow = A_KM ? wm * 64 + lm : wm * 64 + lm * 4;
    const int bcol = B_KM ? wn * 32 + ln : wn * 32 + ln * 4;
    int rows[8], cols[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) rows[r] = A_KM ? arow + 8 * r : arow + (r & 3) + (r >> 2) * 32;
#pragma unroll
    for (int c = 0; c < 8; ++c) cols[c] = B_KM ? bcol + 4 * c : bcol + (c & 3) + (c >> 2) * 16;

    const int nkt = (p.K + BK - 1) / BK;
    const int nchunks = (p.K + kKChunk - 1) / kKChunk;

    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.0f;

    constexpr uint32_t kStageBytes = STAGE_FLOATS * 4;
    int issued = 0;   // producer (thread 0): tiles issued so far
    if (TMA) {
        if (tid == 0) {
            for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(&full[s]), 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            for (; issued < STAGES && issued < nkt; ++issued) {
                float *st = stages + issued * STAGE_FLOATS;
                const uint32_t bar = smem_u32(&full[issued]);
                mbar_arrive_expect_tx(bar, kStageBytes);
                const int k0 = issued * BK;
                if (A_KM) tma_load_2d(smem_u32(st), &tmA, k0, m0, bar);
                else      tma_load_2d(smem_u32(st), &tmA, m0, k0, bar);
                if (B_KM) tma_load_2d(smem_u32(st + TILE_FLOATS), &tmB, k0, n0, bar);
                else      tma_load_2d(smem_u32(st + TILE_FLOATS), &tmB, n0, k0, bar);
            }
        }
    }

    bool aborted = false;
    int kt = 0;
    for (; kt < nkt; ++kt) {
        const int s = TMA ? kt % STAGES : 0;
        const float *As = stages + s * STAGE_FLOATS;
        const float *Bs = As + TILE_FLOATS;
        int ok = 1;
        if (TMA) {
            ok = mbar_wait_bounded(smem_u32(&full[s]), (kt / STAGES) & 1);
        } else {
            __syncthreads();   // everyone is done with the previous tile
            load_tile_plain<A_KM>(stages, p.A, p.lda, p.M, p.K, m0, kt * BK, tid);
            load_tile_plain<B_KM>(stages + TILE_FLOATS, p.B, p.ldb, p.N, p.K, n0,
                                  kt * BK, tid);
            __syncthreads();
        }
        if (ok) {
            const int kcount = min(BK, p.K - kt * BK);
            if (kcount == BK) {
#pragma unroll
                for (int q = 0; q < BK / 4; ++q)
                    mma_group<A_KM, B_KM>(As, Bs, q, arow, bcol, lm, ln, acc);
            } else {
                mma_partial<A_KM, B_KM>(As, Bs, kcount, rows, cols, acc);
            }
        }
        // chunk boundary: fold the finished partial into the running total
        const bool last = (kt == nkt - 1);
        if (((kt + 1) % TILES_PER_CHUNK == 0) || last) {
            const int chunk = kt / TILES_PER_CHUNK;
            if (!(chunk == 0 && last)) {
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float4 &t = totals[(r * 2 + h) * THREADS + tid];
                        float *a4 = &acc[r][4 * h];
                        if (chunk == 0) {
                            t = make_float4(a4[0], a4[1], a4[2], a4[3]);
                        } else {
                            float4 v = t;
                            v.x = __fadd_rn(v.x, a4[0]);
                            v.y = __fadd_rn(v.y, a4[1]);
                            v.z = __fadd_rn(v.z, a4[2]);
                            v.w = __fadd_rn(v.w, a4[3]);
                            if (last) { a4[0] = v.x; a4[1] = v.y; a4[2] = v.z; a4[3] = v.w; }
                            else t = v;
                        }
                    }
                if (!last) {
#pragma unroll
                    for (int r = 0; r < 8; ++r)
#pragma unroll
                        for (int c = 0; c < 8; ++c) acc[r][c] = 0.0f;
                }
            }
        }
        if (TMA) {
            if (__syncthreads_or(!ok)) { aborted = true; break; }
            if (tid == 0 && issued < nkt) {
                float *st = stages + s * STAGE_FLOATS;
                const uint32_t bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, kStageBytes);
                const int k0 = issued * BK;
                if (A_KM) tma_load_2d(smem_u32(st), &tmA, k0, m0, bar);
                else      tma_load_2d(smem_u32(st), &tmA, m0, k0, bar);
                if (B_KM) tma_load_2d(smem_u32(st + TILE_FLOATS), &tmB, k0, n0, bar);
                else      tma_load_2d(smem_u32(st + TILE_FLOATS), &tmB, n0, k0, bar);
                ++issued;
            }
        }
    }
    (void)nchunks;

    if (TMA && aborted) {
        if (tid == 0) {
            atomicOr(&g_gemm_watchdog, kWatchdogGemm);
            // let the copies still in flight land before the CTA exits
            for (int t = kt; t < issued; ++t)
                (void)mbar_wait_bounded(smem_u32(&full[t % STAGES]), (t / STAGES) & 1);
        }
        return;
    }

    // epilogue: C[m0 + rows[r], n0 + cols[c]]
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = m0 + rows[r];
        if (i >= p.M) continue;
        float *crow = p.C + int64_t(i) * p.ldc;
        if (!B_KM && p.vec_store) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = n0 + cols[4 * h];
                if (j + 3 < p.N) {
                    *reinterpret_cast<float4 *>(crow + j) =
                        make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2],
                                    acc[r][4 * h + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (j + c < p.N) crow[j + c] = acc[r][4 * h + c];
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int j = n0 + cols[c];
                if (j < p.N) crow[j] = acc[r][c];
            }
        }
    }
}

// K == 0: the empty sum, +0 everywhere.
__global__ void fill_zero_kernel(float *C, int64_t ldc, int64_t M, int64_t N) {
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        C[i * ldc + j] = 0.0f;
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// A 2-D fp32 tensor map over a row-major matrix (inner = contiguous extent,
// outer = rows, ld = row stride in elements) with a 32 x 128 or 128 x 32 box.
bool make_map(CUtensorMap *map, const float *base, int64_t inner, int64_t outer,
              int64_t ld, bool kmajor_box) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
    cuuint32_t box[2];
    CUtensorMapSwizzle swz;
    if (kmajor_box) { box[0] = 32; box[1] = 128; swz = CU_TENSOR_MAP_SWIZZLE_128B; }
    else            { box[0] = 128; box[1] = 32; swz = CU_TENSOR_MAP_SWIZZLE_NONE; }
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tma_ok(const float *base, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(base) % 16 == 0) && (ld % 4 == 0) &&
           (ld * 4 < (int64_t(1) << 40));
}

template <bool A_KM, bool B_KM, bool TMA>
cudaError_t launch_variant(const CUtensorMap &ma, const CUtensorMap &mb, const KArgs &k,
                           cudaStream_t s) {
    auto kern = gemm_kernel<A_KM, B_KM, TMA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(int64_t(k.mt) * k.nt);
    kern<<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, k);
    return cudaGetLastError();
}

template <bool TMA>
cudaError_t launch_layout(bool a_km, bool b_km, const CUtensorMap &ma,
                          const CUtensorMap &mb, const KArgs &k, cudaStream_t s) {
    if (a_km && b_km) return launch_variant<true, true, TMA>(ma, mb, k, s);
    if (a_km) return launch_variant<true, false, TMA>(ma, mb, k, s);
    if (b_km) return launch_variant<false, true, TMA>(ma, mb, k, s);
    return launch_variant<false, false, TMA>(ma, mb, k, s);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.K == 0) {
        const int64_t total = a.M * a.N;
        const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
        fill_zero_kernel<<<unsigned(blocks), 256, 0, s>>>(a.C, a.ldc, a.M, a.N);
        return cudaGetLastError();
    }
    KArgs k;
    k.M = int(a.M); k.N = int(a.N); k.K = int(a.K);
    k.lda = a.lda; k.ldb = a.ldb; k.ldc = a.ldc;
    k.A = a.A; k.B = a.B; k.C = a.C;
    k.mt = int((a.M + BM - 1) / BM);
    k.nt = int((a.N + BN - 1) / BN);
    k.m_fast = a.M <= a.N;
    k.vec_store = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 4 == 0);
    // op(A) is k-contiguous when A is not transposed; op(B) when B is.
    const bool a_km = !a.transA, b_km = a.transB != 0;
    CUtensorMap ma{}, mb{};
    bool tma = tma_ok(a.A, a.lda) && tma_ok(a.B, a.ldb);
    if (tma) {
        tma = a_km ? make_map(&ma, a.A, a.K, a.M, a.lda, true)
                   : make_map(&ma, a.A, a.M, a.K, a.lda, false);
        tma = tma && (b_km ? make_map(&mb, a.B, a.K, a.N, a.ldb, true)
                           : make_map(&mb, a.B, a.N, a.K, a.ldb, false));
    }
    if (tma) return launch_layout<true>(a_km, b_km, ma, mb, k, s);
    return launch_layout<false>(a_km, b_km, ma, mb, k, s);
}

cudaError_t gemm_watchdog(unsigned int *code, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemm_watchdog, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear && *code) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_watchdog, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace det
