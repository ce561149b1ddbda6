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
//  * Shared memory bandwidth sets the register tile. A 16-byte shared load
//    costs 4 wavefronts of the SM's one-wavefront-a-clock pipe, while the 4
//    sub-partitions issue 4 warp-FFMAs a clock. With a TM x TN register tile a
//    thread loads TM + TN floats per k for TM*TN FFMAs, so 8 x 8 saturates the
//    pipe exactly at full FFMA rate; 16 x 8 leaves it 25% headroom. So: CTA
//    tile 256 x 128, 256 threads (2 x 4 warps of 128 x 32), 16 x 8 outputs a
//    thread, one CTA per SM (up to 255 registers a thread).
//  * k-tile 32 divides the 256-wide chunk, so chunk boundaries fall on k-tile
//    boundaries. Operand tiles arrive by TMA (cp.async.bulk.tensor) into a
//    2-stage ring (48 KB a stage) with one mbarrier per stage. A stage is
//    refilled by the last warp to finish with it (a shared counter per stage),
//    so no warp ever waits for the others; thread 0 only issues the first
//    stages. Tiles whose k is contiguous use the 128-byte swizzle, so
//    16-byte loads of 4 consecutive k from 8 different rows are free of bank
//    conflicts; tiles whose m/n is contiguous are stored plain and read as
//    float4 along m/n.
//  * Per 4-wide k group a thread issues 24 LDS.128 and 512 FMAs; one operand's
//    4-k fragment is held while the other streams. The FMAs go out as packed
//    pairs (fma.rn.f32x2, each half rounded as fmaf) where a 16-byte load
//    yields the pairs: two rows of op(A) when A is m-contiguous, which
//    measured fastest. A large GEMM with a k-contiguous A therefore first
//    copies A transposed into the caller's workspace (transpose_kernel).
//  * Chunk partials: the running left-to-right total lives in shared memory
//    (128 KB), touched once per 256 k, which keeps registers for the
//    accumulators and fragments.
//  * Persistent: one CTA per SM walks its tiles; the k-tiles of consecutive
//    tiles share the stage ring, so the next tile's loads overlap the
//    epilogue.
//  * Operands whose base or row stride is not 16-byte aligned (TMA cannot
//    describe them) take the same kernel with a plain-load producer; the
//    arithmetic, and so the bits, are identical.
//  * Tile order: the dimension whose operand is smaller runs fastest, so the
//    smaller operand stays resident in the 129 MB L2 and the larger one
//    streams from HBM once.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "det_internal.cuh"

#ifdef DET_GEMM_SECONDARY_NS
// Another build of this file (gemm_n64.cu, gemm_m128.cu): its kernels and batched
// launcher live in their own namespace; the shared helpers, plans and the
// single-product launchers come from the primary build.
#define DET_GEMM_PRIMARY 0
#else
#define DET_GEMM_PRIMARY 1
#endif

namespace det {
#if !DET_GEMM_PRIMARY
namespace DET_GEMM_SECONDARY_NS {
#endif
namespace {

#ifndef DET_GEMM_TM
#define DET_GEMM_TM 16
#endif
#ifndef DET_GEMM_STAGES
#define DET_GEMM_STAGES 2
#endif
#ifndef DET_GEMM_TN
#define DET_GEMM_TN 8
#endif
#ifndef DET_GEMM_WARPS_M
#define DET_GEMM_WARPS_M 2
#endif
#ifndef DET_GEMM_WARPS_N
#define DET_GEMM_WARPS_N 4
#endif
#ifndef DET_GEMM_CTAS_PER_SM
#define DET_GEMM_CTAS_PER_SM 1
#endif
#ifndef DET_GEMM_TMEM
#define DET_GEMM_TMEM 0
#endif
constexpr int TM = DET_GEMM_TM;                 // outputs a thread: TM x TN
constexpr int TN = DET_GEMM_TN;
static_assert(TN == 4 || TN == 8, "fragment loads take one or two float4 along n");
constexpr int WTM = 8 * TM;                     // warp tile rows (8 lanes along m)
constexpr int WTN = 4 * TN;                     // warp tile columns (4 lanes along n)
constexpr int WARPS_M = DET_GEMM_WARPS_M;       // warps of the CTA along m and n
constexpr int WARPS_N = DET_GEMM_WARPS_N;
constexpr int BM = WARPS_M * WTM;               // CTA tile rows (op(A) rows)
constexpr int BN = WARPS_N * WTN;               // CTA tile columns
constexpr int BK = 32;                          // k-tile
constexpr int STAGES = DET_GEMM_STAGES;
static_assert(TM % 4 == 0 && BM <= 256 && BN <= 256, "TMA boxes and fragment loads");
constexpr int THREADS = 32 * WARPS_M * WARPS_N;
constexpr int CTAS_PER_SM = DET_GEMM_CTAS_PER_SM;   // resident CTAs the grid counts on
constexpr int TILES_PER_CHUNK = kKChunk / BK;   // 8
constexpr int A_FLOATS = BM * BK;               // 8192
constexpr int B_FLOATS = BN * BK;               // 4096
constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
// The running chunk totals: in shared memory, or (kTmemTotals) in Tensor
// Memory, where a thread's TM x TN totals fill TM * TN columns of its lane and
// the warps sharing a lane quarter (warp % 4) take consecutive column blocks.
constexpr bool kTmemTotals = DET_GEMM_TMEM != 0;
constexpr int TOTAL_FLOAT4 = kTmemTotals ? 0 : THREADS * TM * TN / 4;
constexpr uint32_t kTmemCols = uint32_t(TM * TN) * uint32_t((THREADS / 32 + 3) / 4);
static_assert(!kTmemTotals || ((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols >= 32 &&
                               kTmemCols * CTAS_PER_SM <= 512),
              "a TMEM allocation is a power of two of 32..512 columns, all CTAs of an SM fit");
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_FLOATS * 4 +
                              size_t(TOTAL_FLOAT4) * 16 + STAGES * 8;
static_assert(kKChunk % BK == 0, "chunk boundaries must fall on k-tiles");
static_assert(SMEM_BYTES <= 232448 && (SMEM_BYTES + 2048) * CTAS_PER_SM <= 233472,
              "the CTAs of an SM fit its 228 KB of shared memory");

__device__ unsigned int g_gemm_watchdog;

// The limit of the consumers' wait for a k-tile's operands. The shipped
// library uses the common bound; the test suite builds a separate copy with
// DET_TEST_GEMM_WAIT_NS=0, whose consumers give up at the first wait that is
// not already complete, to run the give-up path (watchdog bit, drain of the
// copies in flight, skipped stores) on healthy copies.
#ifdef DET_TEST_GEMM_WAIT_NS
constexpr unsigned long long kGemmConsumerWaitNs = DET_TEST_GEMM_WAIT_NS;
#else
constexpr unsigned long long kGemmConsumerWaitNs = kWaitLimitNs;
#endif

// Shared-memory float index of element (row r, k) of an operand tile with R
// rows. KMAJ: rows of 32 k (128 bytes); 16-byte chunk q of row r is stored at
// chunk q ^ (r & 7), the TMA 128-byte swizzle pattern. Otherwise one row of R
// m/n values for each k.
template <bool KMAJ, int R>
__device__ __forceinline__ int tile_idx(int r, int k) {
    if (KMAJ) return r * 32 + ((((k >> 2) ^ (r & 7)) << 2) | (k & 3));
    return k * R + r;
}

struct KArgs {
    int M, N, K;
    int64_t lda, ldb, ldc;
    const float *A, *B;
    float *C;
    int mt, nt;        // tiles along M and N
    int m_fast;        // tile order
    int vec_store;     // C rows 16-byte aligned
    // Work units. Without split, a unit is a tile over all of K. With split,
    // a unit is (tile, group of consecutive 256-wide chunks); it writes every
    // chunk partial P_c of the tile to the workspace in the tile-blocked layout
    // of ws_index(), and a second kernel adds them left to right into C.
    int split;
    int units_per_tile;
    int kt_per_unit;   // multiple of the k-tiles a chunk spans
    float4 *W;
    int accumulate;    // C = C + result (beta = 1): one rounded add, C on the left
    // Batched products (never split): product z = zb * zinner + zh reads its
    // operands and writes C at element offsets zb * X_zb + zh * X_zh from the
    // base pointers; one tensor map spans each whole buffer and a TMA
    // coordinate adds the offset's row (offset / ld) and column (offset % ld).
    int zcount;        // 1: a single product
    int zinner;
    int64_t a_zb, a_zh, b_zb, b_zh, c_zb, c_zh;
    // The TMA coordinates of those offsets: offset / ld and offset % ld split
    // into the parts of zb and zh (the launcher takes TMA only when the
    // column parts never carry into the next row), so the producer needs no
    // 64-bit division: row = (z / zinner) * X_rb + (z % zinner) * X_rh, and
    // column likewise.
    int a_rb, a_cb, a_rh, a_ch, b_rb, b_cb, b_rh, b_ch;
    // Causal: only the tiles holding some output with j <= i are computed
    // (row-major over those tiles); the others are left unwritten.
    int causal;
    int live_tiles;    // tiles computed per product
    // Triangular op(A) (square, batched only): tri 1: op(A)[i][k] = +0 for
    // k > i, so the chunks after a row tile's last row are skipped; tri 2:
    // op(A)[i][k] = +0 for k < i, so the chunks before its first row are. A
    // skipped chunk's partial would be +0 and leaves the left-to-right sum
    // unchanged, but only when every op(B) value it meets is finite (0 * inf
    // is NaN): the kernel skips only if *tri_bad == 0, a count of non-finite
    // op(B) values written before the launch.
    int tri;
    const int *tri_bad;
    // Two independent products in one launch (the GROUP instances): the
    // kernel's second KArgs describes the other product; CTAs below ctas0
    // work on this one, the rest on the other, each set persistent over its
    // own product's units.
    int ctas0;
};

__device__ __forceinline__ int64_t z_offset(int64_t zb_stride, int64_t zh_stride, int z,
                                            int zinner) {
    return int64_t(z / zinner) * zb_stride + int64_t(z % zinner) * zh_stride;
}

// Causal tile rows: tile row mb holds rows mb*BM .. mb*BM + BM - 1, so its
// tiles nb with nb*BN <= mb*BM + BM - 1 hold an output with j <= i.
__device__ __forceinline__ int causal_row_tiles(int mb, int nt);

// Workspace layout of split mode: float4 slot of (chunk c, tile t, accumulator
// quad q of the thread, thread tid), consecutive threads adjacent so each
// store instruction writes 4 KB contiguously.
constexpr int QUADS = TM * TN / 4;   // 32
__device__ __forceinline__ int64_t ws_index(int c, int ntiles, int t, int q, int tid) {
    return ((int64_t(c) * ntiles + t) * QUADS + q) * THREADS + tid;
}

// One 4-wide k group q (k = 4q .. 4q+3 of the k-tile): for every accumulator,
// acc[r][c] = fmaf(a[r][kk], b[c][kk], acc[r][c]) with kk = 0, 1, 2, 3 in that
// order. The order across different accumulators is free, so each layout
// gets the loop nest that keeps the fewest fragment registers live. A
// k-contiguous tile yields the 4 k of one row per 16-byte load; an
// m/n-contiguous tile yields 4 rows of one k.
//   thread rows (op(A)): KMAJ arow + 8r;  else arow + (r & 3) + 32 (r >> 2)
//   thread cols (op(B)): KMAJ bcol + 4c;  else bcol + (c & 3) + 16 (c >> 2)
// Packed FP32 pairs (fma.rn.f32x2, det_internal.cuh): two accumulators of a
// row, columns 2c2 and 2c2 + 1, advance by one instruction. Each half is
// rounded exactly as fmaf, so every accumulator still follows its own
// ascending-k chain; the pair only halves the issue slots the FFMA stream
// takes.

// B with m/n contiguous (B_KM false): one 16-byte load holds columns
// {c, c+1, c+2, c+3} at one k, i.e. two column pairs ready for fma.rn.f32x2;
// A's value is paired with itself. A k-contiguous B would need its pairs
// assembled from two loads, so with a k-contiguous A as well the scalar form
// (mma_group_scalar) is used.
template <bool A_KM>
__device__ __forceinline__ void mma_group_packed(const float *__restrict__ As,
                                                 const float *__restrict__ Bs, int q,
                                                 int arow, int bcol, int lm,
                                                 float (&acc)[TM][TN]) {
    f32x2 b[TN / 2][4];      // b[c2][kk] = columns {2c2, 2c2 + 1} at k = 4q + kk
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const float *pb = Bs + (4 * q + kk) * BN + bcol;
        const ulonglong2 lo = *reinterpret_cast<const ulonglong2 *>(pb);
        b[0][kk] = lo.x; b[1][kk] = lo.y;
        if (TN == 8) {
            const ulonglong2 hi = *reinterpret_cast<const ulonglong2 *>(pb + 16);
            b[TN / 2 - 2][kk] = hi.x; b[TN / 2 - 1][kk] = hi.y;
        }
    }
    auto row_step = [&](int r, float a, int kk) {
        const f32x2 aa = pack2(a, a);
#pragma unroll
        for (int c2 = 0; c2 < TN / 2; ++c2) {
            f32x2 v = pack2(acc[r][2 * c2], acc[r][2 * c2 + 1]);
            v = fma2(aa, b[c2][kk], v);
            unpack2(v, acc[r][2 * c2], acc[r][2 * c2 + 1]);
        }
    };
    if (A_KM) {
        // A streamed one row (4 k) at a time
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            const float4 v = *reinterpret_cast<const float4 *>(
                As + (arow + 8 * r) * 32 + ((q ^ lm) << 2));
            row_step(r, v.x, 0);
            row_step(r, v.y, 1);
            row_step(r, v.z, 2);
            row_step(r, v.w, 3);
        }
    } else {
        // A streamed one k (16 rows) at a time
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *pa = As + (4 * q + kk) * BM + arow;
            float a[TM];
#pragma unroll
            for (int h = 0; h < TM / 4; ++h) {
                const float4 v = *reinterpret_cast<const float4 *>(pa + 32 * h);
                a[4 * h] = v.x; a[4 * h + 1] = v.y; a[4 * h + 2] = v.z; a[4 * h + 3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < TM; ++r) row_step(r, a[r], kk);
        }
    }
}

template <bool A_KM, bool B_KM>
__device__ __forceinline__ void mma_group_scalar(const float *__restrict__ As,
                                          const float *__restrict__ Bs, int q,
                                          int arow, int bcol, int lm, int ln,
                                          float (&acc)[TM][TN]) {
    // B fragment: 8 columns x 4 k
    float b[TN][4];
    if (B_KM) {
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int sw = ln + 4 * (c & 1);          // (bcol + 4c) & 7
            const float4 v = *reinterpret_cast<const float4 *>(
                Bs + (bcol + 4 * c) * 32 + ((q ^ sw) << 2));
            b[c][0] = v.x; b[c][1] = v.y; b[c][2] = v.z; b[c][3] = v.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *pb = Bs + (4 * q + kk) * BN + bcol;
            const float4 lo = *reinterpret_cast<const float4 *>(pb);
            b[0][kk] = lo.x; b[1][kk] = lo.y; b[2][kk] = lo.z; b[3][kk] = lo.w;
            if (TN == 8) {
                const float4 hi = *reinterpret_cast<const float4 *>(pb + 16);
                b[TN - 4][kk] = hi.x; b[TN - 3][kk] = hi.y; b[TN - 2][kk] = hi.z;
                b[TN - 1][kk] = hi.w;
            }
        }
    }
    if (A_KM) {
        // A streamed one row (4 k) at a time
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            const float4 v = *reinterpret_cast<const float4 *>(
                As + (arow + 8 * r) * 32 + ((q ^ lm) << 2));
            const float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int c = 0; c < TN; ++c)
                    acc[r][c] = __fmaf_rn(a[kk], b[c][kk], acc[r][c]);
        }
    } else {
        // A streamed one k (16 rows) at a time
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *pa = As + (4 * q + kk) * BM + arow;
            float a[TM];
#pragma unroll
            for (int h = 0; h < TM / 4; ++h) {
                const float4 v = *reinterpret_cast<const float4 *>(pa + 32 * h);
                a[4 * h] = v.x; a[4 * h + 1] = v.y; a[4 * h + 2] = v.z; a[4 * h + 3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < TM; ++r)
#pragma unroll
                for (int c = 0; c < TN; ++c)
                    acc[r][c] = __fmaf_rn(a[r], b[c][kk], acc[r][c]);
        }
    }
}

// A with m contiguous (A_KM false): one 16-byte load holds rows {r, r+1, r+2,
// r+3} at one k, i.e. two row pairs ready for fma.rn.f32x2; B's value is
// paired with itself, TN splats a k against TM splats when pairing columns.
template <bool B_KM>
__device__ __forceinline__ void mma_group_mpair(const float *__restrict__ As,
                                                const float *__restrict__ Bs, int q,
                                                int arow, int bcol, int ln,
                                                float (&acc)[TM][TN]) {
    float b[TN][4];
    if (B_KM) {
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const int sw = ln + 4 * (c & 1);
            const float4 v = *reinterpret_cast<const float4 *>(
                Bs + (bcol + 4 * c) * 32 + ((q ^ sw) << 2));
            b[c][0] = v.x; b[c][1] = v.y; b[c][2] = v.z; b[c][3] = v.w;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *pb = Bs + (4 * q + kk) * BN + bcol;
            const float4 lo = *reinterpret_cast<const float4 *>(pb);
            b[0][kk] = lo.x; b[1][kk] = lo.y; b[2][kk] = lo.z; b[3][kk] = lo.w;
            if (TN == 8) {
                const float4 hi = *reinterpret_cast<const float4 *>(pb + 16);
                b[TN - 4][kk] = hi.x; b[TN - 3][kk] = hi.y; b[TN - 2][kk] = hi.z;
                b[TN - 1][kk] = hi.w;
            }
        }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const float *pa = As + (4 * q + kk) * BM + arow;
        f32x2 a[TM / 2];     // a[r2] = rows {2r2, 2r2 + 1} of the thread at this k
#pragma unroll
        for (int h = 0; h < TM / 4; ++h) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(pa + 32 * h);
            a[2 * h] = v.x; a[2 * h + 1] = v.y;
        }
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const f32x2 bb = pack2(b[c][kk], b[c][kk]);
#pragma unroll
            for (int r2 = 0; r2 < TM / 2; ++r2) {
                f32x2 v = pack2(acc[2 * r2][c], acc[2 * r2 + 1][c]);
                v = fma2(a[r2], bb, v);
                unpack2(v, acc[2 * r2][c], acc[2 * r2 + 1][c]);
            }
        }
    }
}

// Measured on the 162M shapes: row pairs (A m-contiguous) beat column pairs
// and scalar FFMA by 5-12%, which is why a k-contiguous A worth the copy is
// transposed first (transpose_kernel, gemm_plan).
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void mma_group(const float *__restrict__ As,
                                          const float *__restrict__ Bs, int q,
                                          int arow, int bcol, int lm, int ln,
                                          float (&acc)[TM][TN]) {
    if (!A_KM)     mma_group_mpair<B_KM>(As, Bs, q, arow, bcol, ln, acc);
    else if (B_KM) mma_group_scalar<A_KM, B_KM>(As, Bs, q, arow, bcol, lm, ln, acc);
    else           mma_group_packed<A_KM>(As, Bs, q, arow, bcol, lm, acc);
}

// The thread's r-th row of op(A) and c-th column of op(B), tile-relative.
template <bool A_KM>
__device__ __forceinline__ int row_of(int arow, int r) {
    return A_KM ? arow + 8 * r : arow + (r & 3) + (r >> 2) * 32;
}
template <bool B_KM>
__device__ __forceinline__ int col_of(int bcol, int c) {
    return B_KM ? bcol + 4 * c : bcol + (c & 3) + (c >> 2) * 16;
}

// The last k-tile when K is not a multiple of 32: k ascending up to kcount.
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void mma_partial(const float *__restrict__ As,
                                            const float *__restrict__ Bs, int kcount,
                                            int arow, int bcol, float (&acc)[TM][TN]) {
    for (int k = 0; k < kcount; ++k) {
        float a[TM], b[TN];
#pragma unroll
        for (int r = 0; r < TM; ++r) a[r] = As[tile_idx<A_KM, BM>(row_of<A_KM>(arow, r), k)];
#pragma unroll
        for (int c = 0; c < TN; ++c) b[c] = Bs[tile_idx<B_KM, BN>(col_of<B_KM>(bcol, c), k)];
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
            for (int c = 0; c < TN; ++c) acc[r][c] = __fmaf_rn(a[r], b[c], acc[r][c]);
    }
}

// Plain-load producer: the whole CTA copies one R x 32 tile into the layout
// TMA would produce, zero-filling outside the matrix.
template <bool KMAJ, int R>
__device__ __forceinline__ void load_tile_plain(float *dst, const float *src,
                                                int64_t ld, int rows_total,
                                                int k_total, int r0, int k0,
                                                int tid) {
#pragma unroll 4
    for (int e = tid; e < R * BK; e += THREADS) {
        int r, k;
        if (KMAJ) { r = e >> 5; k = e & 31; }        // consecutive threads: consecutive k
        else      { k = e / R; r = e % R; }          // consecutive threads: consecutive m/n
        const int gr = r0 + r, gk = k0 + k;
        float v = 0.0f;
        if (gr < rows_total && gk < k_total)
            v = KMAJ ? src[int64_t(gr) * ld + gk] : src[int64_t(gk) * ld + gr];
        dst[tile_idx<KMAJ, R>(r, k)] = v;
    }
}

// Issues the TMA loads of k-tile kt of the tile at (m0, n0) into stage `st`.
// (ar, ac), (br, bc): the row and column of the product's operands within
// the buffers the tensor maps span (0 for a single product).
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void issue_stage(float *st, uint64_t *bar_ptr,
                                            const CUtensorMap *tmA, const CUtensorMap *tmB,
                                            int m0, int n0, int kt, int ar, int ac, int br,
                                            int bc) {
    const uint32_t bar = smem_u32(bar_ptr);
    mbar_arrive_expect_tx(bar, STAGE_FLOATS * 4);
    const int k0 = kt * BK;
    if (A_KM) tma_load_2d(smem_u32(st), tmA, ac + k0, ar + m0, bar);
    else      tma_load_2d(smem_u32(st), tmA, ac + m0, ar + k0, bar);
    if (B_KM) tma_load_2d(smem_u32(st + A_FLOATS), tmB, bc + k0, br + n0, bar);
    else      tma_load_2d(smem_u32(st + A_FLOATS), tmB, bc + n0, br + k0, bar);
}

// Unit u: tiles run fastest, so concurrent CTAs share one k range (and, for
// the tiles, the smaller operand's blocks), keeping the working set in L2.
struct Unit {
    int t, m0, n0, kt0, kt1, z;
};

__device__ __forceinline__ int causal_row_tiles(int mb, int nt) {
    return min(nt, (mb * BM + BM - 1) / BN + 1);
}

// BATCH: the kernel instance for batched products (z, causal and triangular
// modes); the plain instance compiles none of that in.
template <bool BATCH>
__device__ __forceinline__ Unit unit_of(const KArgs &p, int u, int nkt, bool tri_on,
                                        int ncta) {
    if (BATCH && tri_on) {
        // Triangular products (never split, never causal) differ in work by
        // row tile: units go out in descending work (tri 1: last row tile
        // first; tri 2: first row tile first), and every other full round of
        // the grid runs backwards, so each CTA's units mix long and short.
        const int G = ncta, U = p.mt * p.nt * p.zcount;
        const int j = u / G, b = u - j * G;
        const int r = ((j & 1) && (j + 1) * G <= U) ? j * G + (G - 1 - b) : u;
        const int per = p.zcount * p.nt;
        const int level = r / per, rest = r - level * per;
        const int mb = p.tri == 1 ? p.mt - 1 - level : level;
        const int nb = rest % p.nt;
        Unit w;
        w.z = rest / p.nt;
        w.t = mb * p.nt + nb;
        w.m0 = mb * BM;
        w.n0 = nb * BN;
        w.kt0 = 0;
        w.kt1 = nkt;
        if (p.tri == 1)
            w.kt1 = min(nkt, ((mb * BM + BM - 1) / kKChunk + 1) * TILES_PER_CHUNK);
        else
            w.kt0 = ((mb * BM) / kKChunk) * TILES_PER_CHUNK;
        return w;
    }
    const int ntiles = p.live_tiles;
    const int per_z = ntiles * p.units_per_tile;
    const int z = BATCH ? u / per_z : 0;
    u -= z * per_z;
    const int t = u % ntiles, g = u / ntiles;
    int mb, nb;
    if (BATCH && p.causal) {
        mb = 0;
        int first = 0;
        while (first + causal_row_tiles(mb, p.nt) <= t) first += causal_row_tiles(mb++, p.nt);
        nb = t - first;
    } else if (p.m_fast) { mb = t % p.mt; nb = t / p.mt; }
    else                 { nb = t % p.nt; mb = t / p.nt; }
    Unit w;
    w.t = t;
    w.z = z;
    w.m0 = mb * BM;
    w.n0 = nb * BN;
    w.kt0 = g * p.kt_per_unit;
    w.kt1 = min(nkt, w.kt0 + p.kt_per_unit);
    return w;
}

// Stores a TM x TN register tile at rows m0 + row r, cols n0 + col c of a
// row-major M x N matrix with row stride ld (bounds-checked); with accum, each
// output becomes C + result.
template <bool A_KM, bool B_KM>
__device__ __forceinline__ void store_tile(const float (&acc)[TM][TN], float *base,
                                           int64_t ld, int M, int N, int m0, int n0,
                                           int arow, int bcol, int vec, int accum) {
    auto out = [accum](float *p, float v) { *p = accum ? __fadd_rn(*p, v) : v; };
#pragma unroll
    for (int r = 0; r < TM; ++r) {
        const int i = m0 + row_of<A_KM>(arow, r);
        if (i >= M) continue;
        float *crow = base + int64_t(i) * ld;
        if (!B_KM && vec) {
#pragma unroll
            for (int h = 0; h < TN / 4; ++h) {
                const int j = n0 + col_of<B_KM>(bcol, 4 * h);
                if (j + 3 < N) {
                    float4 v = make_float4(acc[r][4 * h], acc[r][4 * h + 1],
                                           acc[r][4 * h + 2], acc[r][4 * h + 3]);
                    if (accum) {
                        const float4 o = *reinterpret_cast<const float4 *>(crow + j);
                        v = make_float4(__fadd_rn(o.x, v.x), __fadd_rn(o.y, v.y),
                                        __fadd_rn(o.z, v.z), __fadd_rn(o.w, v.w));
                    }
                    *reinterpret_cast<float4 *>(crow + j) = v;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (j + c < N) out(crow + j + c, acc[r][4 * h + c]);
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < TN; ++c) {
                const int j = n0 + col_of<B_KM>(bcol, c);
                if (j < N) out(crow + j, acc[r][c]);
            }
        }
    }
}

// The epilogue through shared memory, for op(A) m-contiguous and op(B)
// k-contiguous (the LM head on its copy of X, the attention's score
// product). A thread's columns are 4 apart there, so direct stores write 16
// scattered bytes of 8 rows an instruction. Here the warp's 128 x 32 result
// first goes to the warp's own slots of the totals area (float4 slots
// q * THREADS + 32 * warp + lane, q = 0..31: 32 runs of 128 floats, 4 rows
// each), with the 16-byte groups of a row XOR-swizzled by (row / 4) mod 8 so
// that the scalar writes and the 16-byte reads are both conflict-free; it
// then leaves as whole 128-byte rows, four rows a store instruction. Only
// the store pattern changes: each output is the same value, written once
// (with accum, C + result as store_tile adds it). The slots belong to the
// warp's own threads, whose chunk folds are done; the area is free again
// after the final __syncwarp.
constexpr bool kStagedEpilogue = !kTmemTotals && TM == 16 && TN == 8 && WTM == 128 &&
                                 WTN == 32;
__device__ __forceinline__ void store_tile_staged(const float (&acc)[TM][TN], float *area,
                                                  float *base, int64_t ld, int M, int N, int r0,
                                                  int c0, int accum) {
    // the thread's place is read here, not passed in, so that the compiler
    // does not keep these offsets live through the main loop
    uint32_t tidx;
    asm volatile("mov.u32 %0, %%tid.x;" : "=r"(tidx));
    const int lane = int(tidx & 31u), warp = int(tidx >> 5);
    const int lm = lane >> 2, ln = lane & 3;
    float *mine = area + warp * 128;
    __syncwarp();
    {
        // thread rows 4 lm + (r & 3) + 32 (r >> 2), columns ln + 4c: row run
        // lm + 8 (r >> 2), row in run r & 3, swizzled column ln + 4 (c ^ lm)
        float *t = mine + lm * (THREADS * 4) + ln;
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            float *tc = t + 4 * (c ^ lm);
#pragma unroll
            for (int r = 0; r < TM; ++r)
                tc[(r >> 2) * 8 * (THREADS * 4) + (r & 3) * 32] = acc[r][c];
        }
    }
    __syncwarp();
    // lane: row 4 s + (lane >> 3) of the warp tile, columns 4 (lane & 7) .. + 3
    const int rl = lane >> 3, g = lane & 7;
    const int col = c0 + 4 * g;
    const bool full = col + 3 < N;
    float *crow = base + int64_t(r0 + rl) * ld + col;
#pragma unroll 1
    for (int s0 = 0; s0 < 8; ++s0) {
        const float *src = mine + s0 * (THREADS * 4) + rl * 32 + 4 * (g ^ s0);
        float *dst0 = crow + int64_t(4 * s0) * ld;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int s = s0 + 8 * t;
            if (r0 + rl + 4 * s >= M) continue;
            float4 v = *reinterpret_cast<const float4 *>(src + 8 * t * (THREADS * 4));
            float *dst = dst0 + int64_t(32 * t) * ld;
            if (full) {
                if (accum) {
                    const float4 o = *reinterpret_cast<const float4 *>(dst);
                    v = make_float4(__fadd_rn(o.x, v.x), __fadd_rn(o.y, v.y),
                                    __fadd_rn(o.z, v.z), __fadd_rn(o.w, v.w));
                }
                *reinterpret_cast<float4 *>(dst) = v;
            } else {
                const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < N) dst[e] = accum ? __fadd_rn(dst[e], vv[e]) : vv[e];
            }
        }
    }
    __syncwarp();
}

// The chunk fold with the running totals in Tensor Memory: 32 columns a copy.
// The first chunk's partial is stored as the total; a later one is added to
// it, total + partial, and after the last chunk the sum is the result (left
// in acc). Warp-wide: every lane takes part in the same call.
__device__ __forceinline__ void fold_tmem(float (&acc)[TM][TN], uint32_t taddr, bool first,
                                          bool last) {
    static_assert((TM * TN) % 32 == 0, "whole 32-column copies");
    __syncwarp();
#pragma unroll
    for (int g = 0; g < TM * TN / 32; ++g) {
        uint32_t v[32];
        if (first) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                v[i] = __float_as_uint(acc[(32 * g + i) / TN][(32 * g + i) % TN]);
            tmem_st32(taddr + 32u * g, v);
        } else {
            tmem_ld32(taddr + 32u * g, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float &a = acc[(32 * g + i) / TN][(32 * g + i) % TN];
                const float t = __fadd_rn(__uint_as_float(v[i]), a);
                if (last) a = t;
                else v[i] = __float_as_uint(t);
            }
            if (!last) tmem_st32(taddr + 32u * g, v);
        }
    }
}

// Persistent: CTA b computes tiles b, b + gridDim.x, ... The k-tiles of all its
// tiles form one sequence through the stage ring, so the loads of the next
// tile are in flight while the current one finishes and stores.
// Producer bookkeeping, kept in shared memory so it costs no registers. One
// lane at a time touches it: thread 0 for the first stages, then the lane
// that releases a stage last, which every other lane's release precedes.
struct Producer {
    int ui;          // index of the unit being issued, among this CTA's units
    int kt;          // next k-tile of that unit
    int more;        // units left to issue
    int count;       // k-tiles issued so far
    Unit u;
};

// GROUP: the instance for two products in one grid (never batched): a CTA
// takes its product once, at entry, from its index; the other instances
// compile none of that in.
template <bool A_KM, bool B_KM, bool TMA, bool SPLIT, bool BATCH, bool GROUP>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ KArgs p1,
                const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ KArgs p2) {
    __shared__ Producer prod;
    __shared__ volatile int abort_flag;
    __shared__ int released[STAGES];   // warps done with a stage (last one refills)
    __shared__ uint32_t tmem_base;     // the CTA's Tensor Memory (kTmemTotals)
    static_assert(!(SPLIT && kTmemTotals), "split partials pass through the totals area");

    extern __shared__ unsigned char smem_raw[];
    float *smem = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *stages = smem;
    float4 *totals = reinterpret_cast<float4 *>(smem + STAGES * STAGE_FLOATS);
    uint64_t *full = reinterpret_cast<uint64_t *>(totals + TOTAL_FLOAT4);   // data landed

    // launched as a programmatic dependent of the kernel before it on the
    // stream: nothing here reads or writes global memory before that grid is
    // complete (a plain launch passes this at once)
    grid_dependency_wait();

    // this CTA's product, and its place among the CTAs of that product
    const bool second = GROUP && int(blockIdx.x) >= p1.ctas0;
    const KArgs &p = second ? p2 : p1;
    const CUtensorMap *tmA = second ? &tmA2 : &tmA1;
    const CUtensorMap *tmB = second ? &tmB2 : &tmB1;
    const int cta = second ? int(blockIdx.x) - p1.ctas0 : int(blockIdx.x);
    const int ncta = !GROUP ? int(gridDim.x) : second ? int(gridDim.x) - p1.ctas0 : p1.ctas0;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / WARPS_N, wn = warp % WARPS_N;   // warp tile WTM x WTN
    const int lm = lane >> 2, ln = lane & 3;     // 8 x 4 lanes

    const int arow = A_KM ? wm * WTM + lm : wm * WTM + lm * 4;
    const int bcol = B_KM ? wn * WTN + ln : wn * WTN + ln * 4;

    if (kTmemTotals) {
        if (warp == 0) tmem_alloc(smem_u32(&tmem_base), kTmemCols);
        tmem_fence_before_sync();
        __syncthreads();
        tmem_fence_after_sync();
    }
    const uint32_t tmem_mine = kTmemTotals ? tmem_base + ((uint32_t(warp & 3) * 32u) << 16) +
                                                 uint32_t(warp >> 2) * uint32_t(TM * TN)
                                           : 0u;

    const int nunits = p.live_tiles * p.units_per_tile * p.zcount;
    const int my_units = (nunits - cta + ncta - 1) / ncta;
    const int nkt = (p.K + BK - 1) / BK;
    const bool tri_on = BATCH && p.tri != 0 && *p.tri_bad == 0;

    // producer: issues the next k-tile of the CTA's unit sequence into a slot
    // (thread 0 for the first stages, then the last warp done with a stage)
    auto issue_next = [&](int slot) {
        int ar = 0, ac = 0, br = 0, bc = 0;
        if (BATCH && p.zcount > 1) {
            const int zb = prod.u.z / p.zinner, zh = prod.u.z - zb * p.zinner;
            ar = zb * p.a_rb + zh * p.a_rh; ac = zb * p.a_cb + zh * p.a_ch;
            br = zb * p.b_rb + zh * p.b_rh; bc = zb * p.b_cb + zh * p.b_ch;
        }
        issue_stage<A_KM, B_KM>(stages + slot * STAGE_FLOATS, &full[slot], tmA, tmB,
                                prod.u.m0, prod.u.n0, prod.kt, ar, ac, br, bc);
        ++prod.count;
        if (++prod.kt == prod.u.kt1) {
            if (++prod.ui < my_units) {
                prod.u = unit_of<BATCH>(p, cta + prod.ui * ncta, nkt, tri_on, ncta);
                prod.kt = prod.u.kt0;
            } else {
                prod.more = 0;
            }
        }
    };
    if (TMA) {
        if (tid == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(smem_u32(&full[s]), 1);
                released[s] = 0;
            }
            abort_flag = 0;
            fence_mbar_init();
            prod.ui = 0;
            prod.count = 0;
            prod.more = my_units > 0;
            if (prod.more) {
                prod.u = unit_of<BATCH>(p, cta, nkt, tri_on, ncta);
                prod.kt = prod.u.kt0;
            }
            for (int s = 0; s < STAGES && prod.more; ++s) issue_next(s);
        }
        __syncthreads();
    }

    int64_t it = 0;            // consumer position in the k-tile sequence
    bool aborted = false;
    for (int ui = 0; ui < my_units && !aborted; ++ui) {
        const Unit w = unit_of<BATCH>(p, cta + ui * ncta, nkt, tri_on, ncta);
        float acc[TM][TN];
#pragma unroll
        for (int r = 0; r < TM; ++r)
#pragma unroll
            for (int c = 0; c < TN; ++c) acc[r][c] = 0.0f;

        for (int kt = w.kt0; kt < w.kt1; ++kt, ++it) {
            const int s = TMA ? int(it % STAGES) : 0;
            const float *As = stages + s * STAGE_FLOATS;
            const float *Bs = As + A_FLOATS;
            int ok = 1;
            if (TMA) {
                ok = mbar_wait_or_abort(smem_u32(&full[s]), uint32_t(it / STAGES) & 1u,
                                        &abort_flag, kGemmConsumerWaitNs);
            } else {
                __syncthreads();   // everyone is done with the previous k-tile
                load_tile_plain<A_KM, BM>(stages,
                                          p.A + (BATCH ? z_offset(p.a_zb, p.a_zh, w.z, p.zinner) : 0),
                                          p.lda, p.M, p.K, w.m0, kt * BK, tid);
                load_tile_plain<B_KM, BN>(stages + A_FLOATS,
                                          p.B + (BATCH ? z_offset(p.b_zb, p.b_zh, w.z, p.zinner) : 0),
                                          p.ldb,
                                          p.N, p.K, w.n0, kt * BK, tid);
                __syncthreads();
            }
            if (ok) {
                const int kcount = min(BK, p.K - kt * BK);
                if (kcount == BK) {
#pragma unroll 1
                    for (int q = 0; q < BK / 4; ++q)
                        mma_group<A_KM, B_KM>(As, Bs, q, arow, bcol, lm, ln, acc);
                } else {
                    mma_partial<A_KM, B_KM>(As, Bs, kcount, arow, bcol, acc);
                }
            }
            // the unit's last k-tile; a batched tile's chunks run from w.kt0 (0
            // unless skipped) to w.kt1 (nkt unless skipped)
            const bool last = (SPLIT || !BATCH) ? (kt == nkt - 1) : (kt == w.kt1 - 1);
            const int first_chunk = (SPLIT || !BATCH) ? 0 : w.kt0 / TILES_PER_CHUNK;
            if (((kt + 1) % TILES_PER_CHUNK == 0) || last) {
                const int chunk = kt / TILES_PER_CHUNK;
                if (SPLIT) {
                    // split: chunk partials go to the workspace through the
                    // thread's own slots of the totals area, so the
                    // accumulators are free again before the global stores.
                    // The tile's first chunk group (k from 0) keeps the left
                    // fold's running total there instead and writes it once,
                    // at its last chunk: the second pass starts from it.
                    const bool prefix = w.kt0 == 0;
#pragma unroll
                    for (int r = 0; r < TM; ++r)
#pragma unroll
                        for (int h = 0; h < TN / 4; ++h) {
                            float4 &t = totals[(r * (TN / 4) + h) * THREADS + tid];
                            const float *a4 = &acc[r][4 * h];
                            if (!prefix || chunk == 0) {
                                t = make_float4(a4[0], a4[1], a4[2], a4[3]);
                            } else {
                                float4 v = t;
                                v.x = __fadd_rn(v.x, a4[0]);
                                v.y = __fadd_rn(v.y, a4[1]);
                                v.z = __fadd_rn(v.z, a4[2]);
                                v.w = __fadd_rn(v.w, a4[3]);
                                t = v;
                            }
                        }
#pragma unroll
                    for (int r = 0; r < TM; ++r)
#pragma unroll
                        for (int c = 0; c < TN; ++c) acc[r][c] = 0.0f;
                    if (ok && (!prefix || kt == w.kt1 - 1)) {
                        float4 *wb = p.W + ws_index(chunk, p.mt * p.nt, w.t, 0, tid);
#pragma unroll 4
                        for (int q4 = 0; q4 < QUADS; ++q4)
                            __stcg(wb + q4 * THREADS, totals[q4 * THREADS + tid]);
                    }
                } else if (kTmemTotals && !(chunk == first_chunk && last)) {
                    // fold the finished partial into the running total (Tensor
                    // Memory); after the last chunk acc holds the result
                    fold_tmem(acc, tmem_mine, chunk == first_chunk, last);
                    if (!last) {
#pragma unroll
                        for (int r = 0; r < TM; ++r)
#pragma unroll
                            for (int c = 0; c < TN; ++c) acc[r][c] = 0.0f;
                    }
                } else if (!kTmemTotals && !(chunk == first_chunk && last)) {
                    // fold the finished partial into the running total; after the
                    // last chunk acc holds the result
#pragma unroll
                    for (int r = 0; r < TM; ++r)
#pragma unroll
                        for (int h = 0; h < TN / 4; ++h) {
                            float4 &t = totals[(r * (TN / 4) + h) * THREADS + tid];
                            float *a4 = &acc[r][4 * h];
                            if (chunk == first_chunk) {
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
                        for (int r = 0; r < TM; ++r)
#pragma unroll
                            for (int c = 0; c < TN; ++c) acc[r][c] = 0.0f;
                    }
                }
            }
            if (TMA) {
                // release the stage: the last warp to finish with it refills it,
                // so no warp ever waits for the others here (the fences order
                // the producer bookkeeping between successive issuing lanes)
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    if (atomicAdd(&released[s], 1) == THREADS / 32 - 1) {
                        atomicExch(&released[s], 0);
                        __threadfence_block();
                        if (prod.more && !abort_flag) issue_next(s);
                    }
                }
                __syncwarp();
                if (!ok || abort_flag) { aborted = true; ++it; break; }
            }
        }
        if (aborted) break;
        // epilogue (the next unit's loads are already in flight)
        if constexpr (!SPLIT && kStagedEpilogue && !A_KM && B_KM) {
            float *cbase = p.C + (BATCH ? z_offset(p.c_zb, p.c_zh, w.z, p.zinner) : 0);
            if (p.vec_store)
                store_tile_staged(acc, reinterpret_cast<float *>(totals), cbase, p.ldc, p.M,
                                  p.N, w.m0 + wm * WTM, w.n0 + wn * WTN, p.accumulate);
            else
                store_tile<A_KM, B_KM>(acc, cbase, p.ldc, p.M, p.N, w.m0, w.n0, arow, bcol, 0,
                                       p.accumulate);
        } else if constexpr (!SPLIT) {
            store_tile<A_KM, B_KM>(acc,
                                   p.C + (BATCH ? z_offset(p.c_zb, p.c_zh, w.z, p.zinner) : 0),
                                   p.ldc,
                                   p.M, p.N, w.m0, w.n0, arow, bcol,
                                   p.vec_store, p.accumulate);
        }
    }

    // any warp may have issued the last copies: once every thread is here no
    // more are issued, and thread 0 drains them
    if (kTmemTotals) tmem_fence_before_sync();
    __syncthreads();
    if (kTmemTotals) tmem_fence_after_sync();
    if (TMA && abort_flag && tid == 0) {
        // every warp sees the shared abort flag within one k-tile and leaves its
        // loop. Thread 0 records the event and lets the last copy issued on
        // each stage land before it exits (the CTA's shared memory lives until
        // its last thread exits); each wait is bounded.
        atomicOr(&g_gemm_watchdog, kWatchdogGemm);
        for (int64_t t = prod.count > STAGES ? prod.count - STAGES : 0; t < prod.count; ++t)
            (void)mbar_wait_bounded(smem_u32(&full[t % STAGES]), uint32_t(t / STAGES) & 1u);
    }
    if (kTmemTotals && warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Split-K second pass: C[i,j] = ((P_0 + P_1) + P_2) + ... over the chunk
// partials in the workspace, left to right. The first chunk group's slot
// holds that group's running total (the fold's prefix, in the slot of its
// last chunk g - 1), so the sum starts there. One thread per workspace quad:
// it sums the quad over the chunks and scatters the 4 outputs to the rows and
// columns the GEMM thread that wrote it owns.
__global__ void chunk_sum_kernel(KArgs p, int nchunks, int a_km, int b_km) {
    grid_dependency_wait();
    const int ntiles = p.mt * p.nt;
    const int64_t slots = int64_t(ntiles) * QUADS * THREADS;
    const int64_t cstride = slots;      // one chunk's worth of quads
    const int c0 = min(nchunks, p.kt_per_unit / TILES_PER_CHUNK) - 1;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < slots;
         e += int64_t(gridDim.x) * blockDim.x) {
        float4 t = __ldcs(p.W + c0 * cstride + e);
        for (int c = c0 + 1; c < nchunks; ++c) {
            const float4 v = __ldcs(p.W + c * cstride + e);
            t.x = __fadd_rn(t.x, v.x);
            t.y = __fadd_rn(t.y, v.y);
            t.z = __fadd_rn(t.z, v.z);
            t.w = __fadd_rn(t.w, v.w);
        }
        const int tid = int(e % THREADS);
        const int q = int((e / THREADS) % QUADS);
        const int tile = int(e / (int64_t(THREADS) * QUADS));
        int mb, nb;
        if (p.m_fast) { mb = tile % p.mt; nb = tile / p.mt; }
        else          { nb = tile % p.nt; mb = tile / p.nt; }
        const int warp = tid >> 5, lane = tid & 31;
        const int wm = warp / WARPS_N, wn = warp % WARPS_N, lm = lane >> 2, ln = lane & 3;
        const int r = q / (TN / 4), h = q % (TN / 4);
        const int arow = a_km ? wm * WTM + lm : wm * WTM + lm * 4;
        const int bcol = b_km ? wn * WTN + ln : wn * WTN + ln * 4;
        const int i = mb * BM + (a_km ? arow + 8 * r : arow + (r & 3) + (r >> 2) * 32);
        if (i >= p.M) continue;
        float *crow = p.C + int64_t(i) * p.ldc;
        const float v[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * h + cc;
            const int j = nb * BN + (b_km ? bcol + 4 * c : bcol + (c & 3) + (c >> 2) * 16);
            if (j < p.N) crow[j] = p.accumulate ? __fadd_rn(crow[j], v[cc]) : v[cc];
        }
    }
}

// T = A^T: A is M x K (row stride lda), T is K x M (row stride ldt). Data
// movement only, so the GEMM that reads T forms the same chains, bit for bit,
// as one reading A. 64 x 64 tiles through shared memory (one padding column
// against bank conflicts); interior tiles move float4s on both sides when A's
// rows are 16-byte aligned (T's always are), edge tiles and unaligned A go
// element by element. The grid strides over tiles. (32 x 32 tiles of single
// floats ran the 8192 x 768 copy at 21 us.)
constexpr int kTrTile = 64;
__global__ void __launch_bounds__(256)
    transpose_kernel(const float *__restrict__ A, int64_t lda, int M, int K,
                     float *__restrict__ T, int64_t ldt, int vec) {
    __shared__ float tile[kTrTile][kTrTile + 1];
    grid_dependency_wait();
    const int tid = threadIdx.x;
    const int64_t mtiles = (M + kTrTile - 1) / kTrTile, ktiles = (K + kTrTile - 1) / kTrTile;
    for (int64_t t = blockIdx.x; t < mtiles * ktiles; t += gridDim.x) {
        const int m0 = int(t / ktiles) * kTrTile, k0 = int(t % ktiles) * kTrTile;
        const bool full = vec && m0 + kTrTile <= M && k0 + kTrTile <= K;
        __syncthreads();   // the previous tile's reads are done
        if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {      // row tid / 16 + 16 i, float4 tid % 16
                const int r = tid / 16 + 16 * i, c = 4 * (tid % 16);
                const float4 v =
                    *reinterpret_cast<const float4 *>(A + int64_t(m0 + r) * lda + k0 + c);
                tile[r][c] = v.x; tile[r][c + 1] = v.y; tile[r][c + 2] = v.z; tile[r][c + 3] = v.w;
            }
        } else {
            for (int e = tid; e < kTrTile * kTrTile; e += 256) {
                const int r = e / kTrTile, c = e % kTrTile;
                if (m0 + r < M && k0 + c < K) tile[r][c] = A[int64_t(m0 + r) * lda + k0 + c];
            }
        }
        __syncthreads();
        if (full) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {      // T row k0 + tid / 16 + 16 i, float4 tid % 16
                const int kr = tid / 16 + 16 * i, mc = 4 * (tid % 16);
                *reinterpret_cast<float4 *>(T + int64_t(k0 + kr) * ldt + m0 + mc) =
                    make_float4(tile[mc][kr], tile[mc + 1][kr], tile[mc + 2][kr], tile[mc + 3][kr]);
            }
        } else {
            for (int e = tid; e < kTrTile * kTrTile; e += 256) {
                const int kr = e / kTrTile, mc = e % kTrTile;
                if (k0 + kr < K && m0 + mc < M) T[int64_t(k0 + kr) * ldt + m0 + mc] = tile[mc][kr];
            }
        }
    }
}

// K == 0: the empty sum, +0 everywhere (C + 0 when accumulating).
__global__ void fill_zero_kernel(float *C, int64_t ldc, int64_t M, int64_t N, int accum) {
    grid_dependency_wait();
    const int64_t total = M * N;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        C[i * ldc + j] = accum ? __fadd_rn(C[i * ldc + j], 0.0f) : 0.0f;
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
// outer = rows, ld = row stride in elements). A k-contiguous operand gets a
// 32 (k) x R box with the 128-byte swizzle; an m/n-contiguous one an R x 32
// box, unswizzled. R = the tile's extent along m or n.
bool make_map(CUtensorMap *map, const float *base, int64_t inner, int64_t outer,
              int64_t ld, bool kmajor_box, int R) {
    return kmajor_box ? make_tensor_map_2d(map, base, inner, outer, ld, 32, uint32_t(R), true)
                      : make_tensor_map_2d(map, base, inner, outer, ld, uint32_t(R), 32, false);
}

bool tma_ok(const float *base, int64_t ld) { return tma_operand_ok(base, ld); }

// One product ready to launch: its kernel arguments and tensor maps.
struct Prepared {
    KArgs k;
    CUtensorMap ma, mb;
    bool tma, a_km, b_km;
};

// Launches x alone, or x and y (same layout, staging and split mode; never
// batched) in one grid of `grid` CTAs, the first ctas0 of them on x.
template <bool A_KM, bool B_KM, bool TMA>
cudaError_t launch_variant(Prepared x, const Prepared *y, int ctas0, int grid, cudaStream_t s) {
    const KArgs &k = x.k;
    // batched products are never split or grouped
#if DET_GEMM_PRIMARY
    auto kern = y ? (k.split ? gemm_kernel<A_KM, B_KM, TMA, true, false, true>
                             : gemm_kernel<A_KM, B_KM, TMA, false, false, true>)
                : k.split ? gemm_kernel<A_KM, B_KM, TMA, true, false, false>
                : (k.zcount > 1 || k.causal || k.tri)
                    ? gemm_kernel<A_KM, B_KM, TMA, false, true, false>
                    : gemm_kernel<A_KM, B_KM, TMA, false, false, false>;
#else
    // the second build serves batched products only
    auto kern = gemm_kernel<A_KM, B_KM, TMA, false, true, false>;
#endif
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    if (CTAS_PER_SM > 1) {
        // the whole unified L1 as shared memory, so the CTAs of an SM fit
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
    }
    if (!y) {
        const int64_t units = int64_t(k.live_tiles) * k.units_per_tile * k.zcount;
        grid = int(std::min<int64_t>(units, int64_t(sm_count_current_device()) * CTAS_PER_SM));
        ctas0 = grid;
    }
    x.k.ctas0 = ctas0;
    const Prepared &z = y ? *y : x;
    return launch_dependent(kern, dim3(unsigned(grid)), dim3(THREADS), SMEM_BYTES, s, x.ma,
                            x.mb, x.k, z.ma, z.mb, z.k);
}

template <bool TMA>
cudaError_t launch_layout(const Prepared &x, const Prepared *y, int ctas0, int grid,
                          cudaStream_t s) {
    if (x.a_km && x.b_km) return launch_variant<true, true, TMA>(x, y, ctas0, grid, s);
    if (x.a_km) return launch_variant<true, false, TMA>(x, y, ctas0, grid, s);
    if (x.b_km) return launch_variant<false, true, TMA>(x, y, ctas0, grid, s);
    return launch_variant<false, false, TMA>(x, y, ctas0, grid, s);
}

cudaError_t launch_prepared(const Prepared &x, const Prepared *y, cudaStream_t s,
                            int ctas0 = 0, int grid = 0) {
    return x.tma ? launch_layout<true>(x, y, ctas0, grid, s)
                 : launch_layout<false>(x, y, ctas0, grid, s);
}

}  // namespace

#if DET_GEMM_PRIMARY
bool make_tensor_map_2d(CUtensorMap *map, const float *base, int64_t inner, int64_t outer,
                        int64_t ld, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tma_operand_ok(const float *base, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(base) % 16 == 0) && (ld % 4 == 0) &&
           (ld * 4 < (int64_t(1) << 40));
}

// Work plan: whether to split K across CTAs and into how many chunk groups.
// A split unit computes whole 256-wide chunks, so the bits never depend on the
// plan. The cost model takes the k-tile steps of the most loaded CTA under the
// kernel's round-robin unit order (units run tiles-fastest, so a CTA's units
// cycle through the chunk groups and the last, shorter group is counted as
// such) at ~6 us a step of a 256 x 128 tile, and adds the workspace traffic
// (each partial written once and read once) at HBM speed plus the second
// pass's launch.
namespace {
double busiest_cta_steps(int64_t T, int64_t S, int64_t G, int64_t nkt, int sms) {
    const int64_t units = T * S;
    const int64_t grid = std::min<int64_t>(units, sms);
    double worst = 0.0;
    // CTA b takes units b, b + grid, ...; unit u belongs to group u / T
    for (int64_t b = 0; b < grid; ++b) {
        double steps = 0.0;
        for (int64_t u = b; u < units; u += grid) {
            const int64_t g = u / T;
            const int64_t kt0 = g * G * TILES_PER_CHUNK;
            steps += double(std::min<int64_t>(nkt, kt0 + G * TILES_PER_CHUNK) - kt0);
        }
        worst = std::max(worst, steps);
    }
    return worst;
}
}  // namespace

// Row stride of the transposed copy of a k-contiguous A: M rounded up to 4
// floats, so the copy's rows are 16-byte aligned for TMA.
int64_t transposed_ld(int64_t M) { return (M + 3) / 4 * 4; }

namespace {
GemmPlan gemm_plan_core(int64_t M, int64_t N, int64_t K, int sms, bool a_kmajor, int b_kmajor);
}  // namespace

// A k-contiguous B (transB, B stored N x K) is read ~3.5% faster from a K x N
// copy (row stride N rounded up to 4): the row-pair loop then loads B's
// values as 16-byte rows of 4 columns, and the epilogue stores 16-byte groups
// directly (measured on the LM head, 11.03 -> 10.70 ms, and the backward's
// input-gradient products, 3-5%). Taken where that gain, at ~48 TFLOP/s,
// exceeds one and a half times the copy's launch and its read and write at
// HBM speed (a product over a few rows of a large B, such as a row block of
// the LM head, is better off reading B in place); the copy comes first in the
// workspace, and the product over it has its own plan.
GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sms, bool a_kmajor, int b_kmajor) {
    if (b_kmajor == 1 && M > 0 && N > 0 && K > 0) {
        const double gain = 0.035 * 2.0 * double(M) * double(N) * double(K) / 48.0e12;
        const double cost = 5.0e-6 + 8.0 * double(N) * double(K) / 6.0e12;
        if (gain > 1.5 * cost) {
            GemmPlan pl = gemm_plan_core(M, N, K, sms, a_kmajor, 0);
            pl.transpose_b = 1;
            pl.copy_b_bytes = (size_t(K) * size_t(transposed_ld(N)) * 4 + 255) / 256 * 256;
            pl.workspace_bytes += pl.copy_b_bytes;
            return pl;
        }
    }
    return gemm_plan_core(M, N, K, sms, a_kmajor, b_kmajor);
}

namespace {
GemmPlan gemm_plan_core(int64_t M, int64_t N, int64_t K, int sms, bool a_kmajor, int b_kmajor) {
    GemmPlan pl{};
    pl.transpose_a = 0;
    pl.copy_bytes = 0;
    pl.split_bytes = 0;
    const int64_t T = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int64_t nkt = (K + BK - 1) / BK;
    const int64_t nchunks = (K + kKChunk - 1) / kKChunk;
    pl.split = 0;
    pl.units_per_tile = 1;
    pl.kt_per_unit = int(nkt);
    pl.nchunks = int(nchunks);
    pl.workspace_bytes = 0;
    if (M == 0 || N == 0 || K == 0 || sms < 1) return pl;
    const double kt_step_s = 6.0e-6, hbm_bps = 6.0e12, launch_s = 5.0e-6;
    // An unsplit GEMM whose A is k-contiguous runs ~8% faster on a transposed
    // copy (row pairs, mma_group_mpair); take it where that gain, at ~48
    // TFLOP/s, exceeds the copy's launch and its read and write at HBM speed.
    auto consider_transpose = [&] {
        if (!a_kmajor) return;
        const double gain = 0.08 * 2.0 * double(M) * double(N) * double(K) / 48.0e12;
        const double cost = launch_s + 8.0 * double(M) * double(K) / hbm_bps;
        if (gain > cost) {
            pl.transpose_a = 1;
            pl.copy_bytes = pl.workspace_bytes = size_t(K) * size_t(transposed_ld(M)) * 4;
        }
    };
    // A split product may read A from a transposed copy too (the copy first in
    // the workspace, 256-byte rounded, the partials after it): from A itself
    // it runs the column-pair loop, or the scalar one when B is k-contiguous as
    // well (b_kmajor 1), ~8% and ~15% slower. Taken where that gain exceeds
    // the copy; b_kmajor < 0 (the two-product plans) never takes it.
    auto consider_split_copy = [&] {
        if (!a_kmajor || b_kmajor < 0) return;
        const double frac = b_kmajor ? 0.15 : 0.08;
        const double gain = frac * 2.0 * double(M) * double(N) * double(K) / 48.0e12;
        const double cost = launch_s + 8.0 * double(M) * double(K) / hbm_bps;
        if (gain > cost) {
            pl.transpose_a = 1;
            pl.copy_bytes = (size_t(K) * size_t(transposed_ld(M)) * 4 + 255) / 256 * 256;
            pl.workspace_bytes = pl.copy_bytes + pl.split_bytes;
        }
    };
    // enough tiles to fill every SM several times over: splitting cannot pay
    if (nchunks < 2 || T >= int64_t(sms) * 16) {
        consider_transpose();
        return pl;
    }
    double best = busiest_cta_steps(T, 1, nchunks, nkt, sms) * kt_step_s;
    for (int64_t S = 2; S <= nchunks; ++S) {
        const int64_t G = (nchunks + S - 1) / S;              // chunks a unit
        const int64_t S_eff = (nchunks + G - 1) / G;
        if (S_eff != S) continue;                             // same as a smaller S
        const double ws = double(nchunks) * double(T) * BM * BN * 4.0;
        const double cost = busiest_cta_steps(T, S_eff, G, nkt, sms) * kt_step_s +
                            (2.0 * ws + double(M) * double(N) * 4.0) / hbm_bps + launch_s;
        if (cost < 0.97 * best) {
            best = cost;
            pl.split = 1;
            pl.units_per_tile = int(S_eff);
            pl.kt_per_unit = int(G * TILES_PER_CHUNK);
            pl.split_bytes = pl.workspace_bytes = size_t(ws);
        }
    }
    // Unsplit head rows: where a split plan is chosen but the tiles fill the
    // SMs less than twice over, the first row blocks that make one round (at
    // most a tile an SM) run unsplit in a launch of their own, and only the
    // tiles after them are split by their own plan, so only their partials
    // cross HBM. Same bits: every output's chunks and their left-to-right sum
    // are the same whichever launch computes them.
    auto consider_head = [&] {
        const int64_t nt = (N + BN - 1) / BN, mt = (M + BM - 1) / BM;
        const int64_t mb1 = int64_t(sms) / nt;
        if (!pl.split || T >= 2 * int64_t(sms) || mb1 < 1 || mb1 >= mt) return;
        const int64_t M1 = mb1 * BM;
        const GemmPlan tail = gemm_plan(M - M1, N, K, sms, false, -1);
        const int64_t T2 = (mt - mb1) * nt;
        double tail_cost = launch_s;
        if (tail.split) {
            const int64_t G = tail.kt_per_unit / TILES_PER_CHUNK;
            tail_cost += busiest_cta_steps(T2, tail.units_per_tile, G, nkt, sms) * kt_step_s +
                         (2.0 * double(tail.split_bytes) + double(M - M1) * double(N) * 4.0) /
                             hbm_bps + launch_s;
        } else {
            tail_cost += busiest_cta_steps(T2, 1, nchunks, nkt, sms) * kt_step_s;
        }
        const double cost = double(nkt) * kt_step_s + launch_s + tail_cost;
        if (cost < 0.97 * best) {
            best = cost;
            pl.head_rows = M1;
            pl.split_bytes = pl.workspace_bytes = tail.workspace_bytes;
            if (!tail.split) pl.split = 0;
        }
    };
    consider_head();
    if (!pl.split && !pl.head_rows) consider_transpose();
    else consider_split_copy();
    return pl;
}
}  // namespace

// The plan launch_gemm runs with workspace_bytes at ws (16-byte aligned or
// null): the split keeps its partials and drops the copy when the workspace
// holds only the partials; with less, one unit a tile and no copy.
GemmPlan gemm_plan_for(const GemmArgs &a, int sms, const void *ws, size_t workspace_bytes) {
    GemmPlan pl = gemm_plan(a.M, a.N, a.K, sms, !a.transA, a.transB ? 1 : 0);
    const bool usable = ws != nullptr && reinterpret_cast<uintptr_t>(ws) % 16 == 0;
    if (pl.transpose_b && (!usable || workspace_bytes < pl.workspace_bytes))
        pl = gemm_plan_core(a.M, a.N, a.K, sms, !a.transA, a.transB ? 1 : 0);
    if ((pl.split || pl.head_rows) && pl.transpose_a &&
        (!usable || workspace_bytes < pl.workspace_bytes)) {
        pl.transpose_a = 0;
        pl.copy_bytes = 0;
        pl.workspace_bytes = pl.split_bytes;
    }
    if ((pl.split || pl.transpose_a || pl.head_rows) &&
        (!usable || workspace_bytes < pl.workspace_bytes)) {
        const int nchunks = pl.nchunks;
        pl = GemmPlan{};          // no usable workspace: one unit per tile
        pl.units_per_tile = 1;
        pl.kt_per_unit = int((a.K + BK - 1) / BK);
        pl.nchunks = nchunks;
    }
    return pl;
}

// The two products of a plan with head rows: rows [0, head_rows) and the rest.
void head_and_tail(const GemmArgs &a, int64_t head_rows, GemmArgs *h, GemmArgs *t) {
    *h = a;
    *t = a;
    h->M = head_rows;
    t->M = a.M - head_rows;
    t->A = a.transA ? a.A + head_rows : a.A + head_rows * a.lda;
    t->C = a.C + head_rows * a.ldc;
}

// The transA form of a over its K x M copy T (row stride transposed_ld(M)).
GemmArgs over_copy(const GemmArgs &a, const float *T) {
    GemmArgs t = a;
    t.A = T;
    t.lda = transposed_ld(a.M);
    t.transA = 1;
    return t;
}

int64_t gemm_launches(const GemmArgs &a, size_t workspace_bytes) {
    if (a.M == 0 || a.N == 0) return 0;
    if (a.K == 0) return 1;
    // any non-null aligned address stands for a caller workspace of that size
    const GemmPlan pl = gemm_plan_for(a, sm_count_current_device(),
                                      workspace_bytes ? reinterpret_cast<const void *>(256)
                                                      : nullptr,
                                      workspace_bytes);
    // as launch_gemm runs the plan
    if (pl.transpose_b) {
        GemmArgs t = a;
        t.transB = 0;
        t.ldb = transposed_ld(a.N);
        return 1 + gemm_launches(t, workspace_bytes - pl.copy_b_bytes);
    }
    if (pl.transpose_a)
        return 1 + gemm_launches(over_copy(a, a.A),
                                 pl.split || pl.head_rows ? workspace_bytes - pl.copy_bytes : 0);
    if (pl.head_rows) {
        GemmArgs h, t;
        head_and_tail(a, pl.head_rows, &h, &t);
        return gemm_launches(h, 0) + gemm_launches(t, workspace_bytes);
    }
    return 1 + int64_t(pl.split);
}

namespace {
// Kernel arguments and tensor maps of a non-batched product under plan pl
// (split partials, if any, go to W).
Prepared prepare(const GemmArgs &a, const GemmPlan &pl, void *W) {
    Prepared x{};
    KArgs &k = x.k;
    k.M = int(a.M); k.N = int(a.N); k.K = int(a.K);
    k.lda = a.lda; k.ldb = a.ldb; k.ldc = a.ldc;
    k.A = a.A; k.B = a.B; k.C = a.C;
    k.mt = int((a.M + BM - 1) / BM);
    k.nt = int((a.N + BN - 1) / BN);
    k.m_fast = a.M <= a.N;
    k.vec_store = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 4 == 0);
    k.split = pl.split;
    k.units_per_tile = pl.units_per_tile;
    k.kt_per_unit = pl.kt_per_unit;
    k.W = static_cast<float4 *>(pl.split ? W : nullptr);
    k.accumulate = a.accumulate;
    k.zcount = 1;
    k.zinner = 1;
    k.a_zb = k.a_zh = k.b_zb = k.b_zh = k.c_zb = k.c_zh = 0;
    k.causal = 0;
    k.live_tiles = k.mt * k.nt;
    k.tri = 0;
    k.tri_bad = nullptr;
    k.ctas0 = 0;
    // op(A) is k-contiguous when A is not transposed; op(B) when B is.
    x.a_km = !a.transA;
    x.b_km = a.transB != 0;
    x.tma = tma_ok(a.A, a.lda) && tma_ok(a.B, a.ldb);
    if (x.tma) {
        x.tma = x.a_km ? make_map(&x.ma, a.A, a.K, a.M, a.lda, true, BM)
                       : make_map(&x.ma, a.A, a.M, a.K, a.lda, false, BM);
        x.tma = x.tma && (x.b_km ? make_map(&x.mb, a.B, a.K, a.N, a.ldb, true, BN)
                                 : make_map(&x.mb, a.B, a.N, a.K, a.ldb, false, BN));
    }
    return x;
}

// T (K x M, row stride ldt) = A^T for A (M x K, row stride lda).
cudaError_t launch_transpose(const float *A, int64_t lda, int64_t M, int64_t K, float *T,
                             int64_t ldt, int sms, cudaStream_t s) {
    const int64_t tiles = ((M + kTrTile - 1) / kTrTile) * ((K + kTrTile - 1) / kTrTile);
    const unsigned blocks = unsigned(std::min<int64_t>(tiles, int64_t(sms) * 8));
    const int vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 4 == 0);
    return launch_dependent(transpose_kernel, dim3(blocks), dim3(256), 0, s, A, lda, int(M),
                            int(K), T, ldt, vec);
}

cudaError_t launch_chunk_sum(const Prepared &x, int nchunks, int sms, cudaStream_t s) {
    const KArgs &k = x.k;
    const int64_t slots = int64_t(k.mt) * k.nt * QUADS * THREADS;
    const int64_t blocks =
        std::max<int64_t>(1, std::min<int64_t>((slots + 255) / 256, int64_t(sms) * 8));
    return launch_dependent(chunk_sum_kernel, dim3(unsigned(blocks)), dim3(256), 0, s, k,
                            nchunks, int(x.a_km), int(x.b_km));
}
}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, void *workspace, size_t workspace_bytes,
                        cudaStream_t s) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.K == 0) {
        const int64_t total = a.M * a.N;
        const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
        fill_zero_kernel<<<unsigned(blocks), 256, 0, s>>>(a.C, a.ldc, a.M, a.N, a.accumulate);
        return cudaGetLastError();
    }
    const int sms = sm_count_current_device();
    const GemmPlan pl = gemm_plan_for(a, sms, workspace, workspace_bytes);
    if (pl.transpose_b) {
        // op(B) from the K x N copy of B (first in the workspace); the product
        // over it (transB 0) plans the rest of the workspace afresh
        float *TB = static_cast<float *>(workspace);
        const int64_t ldtb = transposed_ld(a.N);
        cudaError_t e = launch_transpose(a.B, a.ldb, a.N, a.K, TB, ldtb, sms, s);
        if (e != cudaSuccess) return e;
        GemmArgs t = a;
        t.B = TB;
        t.ldb = ldtb;
        t.transB = 0;
        return launch_gemm(t, static_cast<char *>(workspace) + pl.copy_b_bytes,
                           workspace_bytes - pl.copy_b_bytes, s);
    }
    if (pl.transpose_a) {
        // op(A) from the K x M copy: the transA form of the same product, its
        // split partials (if any) in the workspace after the copy
        float *T = static_cast<float *>(workspace);
        cudaError_t e = launch_transpose(a.A, a.lda, a.M, a.K, T, transposed_ld(a.M), sms, s);
        if (e != cudaSuccess) return e;
        const GemmArgs t = over_copy(a, T);
        if (!pl.split && !pl.head_rows) return launch_gemm(t, nullptr, 0, s);
        return launch_gemm(t, static_cast<char *>(workspace) + pl.copy_bytes,
                           workspace_bytes - pl.copy_bytes, s);
    }
    if (pl.head_rows) {
        // the head unsplit (no workspace), then the rest with its own plan
        GemmArgs h, t;
        head_and_tail(a, pl.head_rows, &h, &t);
        cudaError_t e = launch_gemm(h, nullptr, 0, s);
        if (e != cudaSuccess) return e;
        return launch_gemm(t, workspace, workspace_bytes, s);
    }
    const Prepared x = prepare(a, pl, workspace);
    cudaError_t e = launch_prepared(x, nullptr, s);
    if (e != cudaSuccess || !pl.split) return e;
    return launch_chunk_sum(x, pl.nchunks, sms, s);
}

// ---------------------------------------------------------------- two products, one launch
// Two independent products of the same layout can share one persistent grid:
// their work units are dealt out together, so the grid's last round is
// filled from both (a product alone leaves part of the 152 SMs idle when its
// units do not divide evenly). Both run unsplit, or both split K into groups
// of the same number of chunks; each product's units, chains, partials and
// chunk sums are exactly those of its own launch, so the bits are the same.
namespace {
constexpr double kKtStepS = 6.0e-6, kHbmBps = 6.0e12, kLaunchS = 5.0e-6;

// The k-tile steps of the busiest CTA when units with the given steps are
// dealt round-robin (unit u to CTA u mod grid) over min(units, sms) CTAs.
double busiest_of(const std::vector<int> &steps, int sms) {
    const int64_t n = int64_t(steps.size());
    const int64_t grid = std::min<int64_t>(n, sms);
    double worst = 0.0;
    for (int64_t b = 0; b < grid; ++b) {
        double t = 0.0;
        for (int64_t u = b; u < n; u += grid) t += steps[size_t(u)];
        worst = std::max(worst, t);
    }
    return worst;
}

// Appends a product's units: T tiles, each split into groups of G chunks
// (G >= nchunks: one unit over all of K), tiles running fastest.
void append_units(std::vector<int> &steps, int64_t T, int64_t nkt, int64_t nchunks, int64_t G) {
    const int64_t S = (nchunks + G - 1) / G;
    for (int64_t g = 0; g < S; ++g) {
        const int64_t kt0 = g * G * TILES_PER_CHUNK;
        const int st = int(std::min<int64_t>(nkt, kt0 + G * TILES_PER_CHUNK) - kt0);
        for (int64_t t = 0; t < T; ++t) steps.push_back(st);
    }
}

struct Shape {
    int64_t T, nkt, nchunks, cbytes;
};
Shape shape_of(const GemmArgs &a) {
    return {((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN), (a.K + BK - 1) / BK,
            (a.K + kKChunk - 1) / kKChunk, a.M * a.N * 4};
}

// Modelled time of a product alone under its own plan.
double alone_cost(const GemmArgs &a, const GemmPlan &pl, int sms) {
    const Shape h = shape_of(a);
    std::vector<int> steps;
    append_units(steps, h.T, h.nkt, h.nchunks,
                 pl.split ? pl.kt_per_unit / TILES_PER_CHUNK : h.nchunks);
    double c = busiest_of(steps, sms) * kKtStepS + kLaunchS;
    if (pl.split)
        c += (2.0 * double(pl.workspace_bytes) + double(h.cbytes)) / kHbmBps + kLaunchS;
    return c;
}
}  // namespace

// The CTAs of a two-product grid of `grid` CTAs are split: c0 for the
// first product's units, the rest for the second's, each set round-robin over
// its own units. Returns the k-tile steps of the busiest CTA for the best c0
// near the split that gives each product its share of the work.
double partition(const std::vector<int> &s0, const std::vector<int> &s1, int sms, int *c0_out,
                 int *grid_out) {
    const int64_t n0 = int64_t(s0.size()), n1 = int64_t(s1.size());
    const int grid = int(std::min<int64_t>(sms, n0 + n1));
    double w0 = 0.0, w1 = 0.0;
    for (int v : s0) w0 += v;
    for (int v : s1) w1 += v;
    const int mid = int(std::lround(double(grid) * w0 / (w0 + w1)));
    double best = 1e300;
    for (int c0 = std::max(1, mid - 8); c0 <= std::min(grid - 1, mid + 8); ++c0) {
        const int c1 = grid - c0;
        if (c0 > n0 || c1 > n1) continue;
        const double b = std::max(busiest_of(s0, c0), busiest_of(s1, c1));
        if (b < best) {
            best = b;
            *c0_out = c0;
        }
    }
    *grid_out = grid;
    return best;
}

PairPlan gemm_pair_plan(const GemmArgs &a0, const GemmArgs &a1, int sms) {
    PairPlan pp{};
    pp.pair = 0;
    pp.p0 = gemm_plan(a0.M, a0.N, a0.K, sms, !a0.transA);
    pp.p1 = gemm_plan(a1.M, a1.N, a1.K, sms, !a1.transA);
    pp.separate_bytes = std::max(pp.p0.workspace_bytes, pp.p1.workspace_bytes);
    pp.shared_transpose = 0;
    if (a0.M == 0 || a0.N == 0 || a0.K == 0 || a1.M == 0 || a1.N == 0 || a1.K == 0 ||
        sms < 2 || (a0.transA != 0) != (a1.transA != 0) ||
        (a0.transB != 0) != (a1.transB != 0))
        return pp;
    const Shape h0 = shape_of(a0), h1 = shape_of(a1);
    if (pp.p0.transpose_a || pp.p1.transpose_a) {
        // Products of one A (the gate and up projections of one input), each
        // of which would read a transposed copy of it: one copy serves both,
        // and their tiles share one grid.
        if (!(pp.p0.transpose_a && pp.p1.transpose_a && a0.A == a1.A && a0.lda == a1.lda &&
              a0.M == a1.M && a0.K == a1.K))
            return pp;
        const double copy = kLaunchS + 8.0 * double(a0.M) * double(a0.K) / kHbmBps;
        std::vector<int> s0, s1;
        append_units(s0, h0.T, h0.nkt, h0.nchunks, h0.nchunks);
        append_units(s1, h1.T, h1.nkt, h1.nchunks, h1.nchunks);
        const double separate = busiest_of(s0, sms) * kKtStepS + busiest_of(s1, sms) * kKtStepS +
                                2.0 * (copy + kLaunchS);
        int c0 = 1, grid = 2;
        const double paired = partition(s0, s1, sms, &c0, &grid) * kKtStepS + copy + kLaunchS;
        if (paired < 0.97 * separate) {
            pp.pair = 1;
            pp.split = 0;
            pp.shared_transpose = 1;
            pp.ctas0 = c0;
            pp.grid = grid;
            pp.p0 = GemmPlan{};
            pp.p0.units_per_tile = 1;
            pp.p0.kt_per_unit = int(h0.nkt);
            pp.p0.nchunks = int(h0.nchunks);
            pp.p1 = pp.p0;
            pp.p1.kt_per_unit = int(h1.nkt);
            pp.p1.nchunks = int(h1.nchunks);
            pp.ws0_bytes = 0;
            pp.workspace_bytes = size_t(a0.K) * size_t(transposed_ld(a0.M)) * 4;
        }
        return pp;
    }
    // Both unsplit, or both split K into groups of G chunks (one kernel
    // instance serves the grid; a common, fine G lets the partition balance).
    const double separate = alone_cost(a0, pp.p0, sms) + alone_cost(a1, pp.p1, sms);
    double best = 0.97 * separate;
    // G == 0: both unsplit; a few fine group sizes (coarse groups balance
    // worse, and each candidate costs the host a pass over the units)
    for (int64_t G : {int64_t(0), int64_t(1), int64_t(2), int64_t(3), int64_t(4)}) {
        const int64_t g0 = G ? G : h0.nchunks, g1 = G ? G : h1.nchunks;
        if (G && ((h0.nchunks + G - 1) / G < 2 || (h1.nchunks + G - 1) / G < 2)) continue;
        std::vector<int> s0, s1;
        append_units(s0, h0.T, h0.nkt, h0.nchunks, g0);
        append_units(s1, h1.T, h1.nkt, h1.nchunks, g1);
        int c0 = 1, grid = 2;
        double c = partition(s0, s1, sms, &c0, &grid) * kKtStepS + kLaunchS;
        const double ws = G ? double(h0.nchunks * h0.T + h1.nchunks * h1.T) * BM * BN * 4.0 : 0.0;
        if (G) c += (2.0 * ws + double(h0.cbytes + h1.cbytes)) / kHbmBps + 2.0 * kLaunchS;
        if (c < best) {
            best = c;
            pp.pair = 1;
            pp.split = G > 0;
            pp.ctas0 = c0;
            pp.grid = grid;
            auto set = [&](GemmPlan &pl, const Shape &h, int64_t g) {
                pl = GemmPlan{};
                pl.nchunks = int(h.nchunks);
                pl.split = G > 0;
                pl.units_per_tile = int((h.nchunks + g - 1) / g);
                pl.kt_per_unit = G ? int(g * TILES_PER_CHUNK) : int(h.nkt);
                pl.workspace_bytes = G ? size_t(h.nchunks * h.T) * BM * BN * 4 : 0;
            };
            set(pp.p0, h0, g0);
            set(pp.p1, h1, g1);
        }
    }
    if (!pp.pair) {
        pp.p0 = gemm_plan(a0.M, a0.N, a0.K, sms, !a0.transA);
        pp.p1 = gemm_plan(a1.M, a1.N, a1.K, sms, !a1.transA);
        return pp;
    }
    // the partials of the second product follow the first's, 256-byte aligned
    pp.ws0_bytes = (pp.p0.workspace_bytes + 255) / 256 * 256;
    pp.workspace_bytes = pp.split ? pp.ws0_bytes + pp.p1.workspace_bytes : 0;
    return pp;
}

cudaError_t launch_gemm_pair(const GemmArgs &a0, const GemmArgs &a1, void *workspace,
                             size_t workspace_bytes, cudaStream_t s) {
    const int sms = sm_count_current_device();
    const PairPlan pp = gemm_pair_plan(a0, a1, sms);
    const bool ws_ok = pp.workspace_bytes == 0 ||
                       (workspace != nullptr && workspace_bytes >= pp.workspace_bytes &&
                        reinterpret_cast<uintptr_t>(workspace) % 16 == 0);
    if (pp.pair && pp.shared_transpose && ws_ok && !a0.accumulate && !a1.accumulate) {
        // one transposed copy of the shared A, then both products read it
        float *T = static_cast<float *>(workspace);
        const int64_t ldt = transposed_ld(a0.M);
        cudaError_t e = launch_transpose(a0.A, a0.lda, a0.M, a0.K, T, ldt, sms, s);
        if (e != cudaSuccess) return e;
        GemmArgs t0 = a0, t1 = a1;
        t0.A = t1.A = T;
        t0.lda = t1.lda = ldt;
        t0.transA = t1.transA = 1;
        const Prepared x = prepare(t0, pp.p0, nullptr), y = prepare(t1, pp.p1, nullptr);
        if (x.tma == y.tma) return launch_prepared(x, &y, s, pp.ctas0, pp.grid);
        e = launch_prepared(x, nullptr, s);
        if (e != cudaSuccess) return e;
        return launch_prepared(y, nullptr, s);
    }
    if (pp.pair && !pp.shared_transpose && ws_ok && !a0.accumulate && !a1.accumulate) {
        const Prepared x = prepare(a0, pp.p0, workspace);
        const Prepared y =
            prepare(a1, pp.p1, static_cast<unsigned char *>(workspace) + pp.ws0_bytes);
        if (x.tma == y.tma && x.a_km == y.a_km && x.b_km == y.b_km) {
            cudaError_t e = launch_prepared(x, &y, s, pp.ctas0, pp.grid);
            if (e != cudaSuccess || !pp.split) return e;
            e = launch_chunk_sum(x, pp.p0.nchunks, sms, s);
            if (e != cudaSuccess) return e;
            return launch_chunk_sum(y, pp.p1.nchunks, sms, s);
        }
    }
    // one after the other (the workspace serves each in turn)
    cudaError_t e = launch_gemm(a0, workspace, workspace_bytes, s);
    if (e != cudaSuccess) return e;
    return launch_gemm(a1, workspace, workspace_bytes, s);
}

#endif  // DET_GEMM_PRIMARY

// The TMA row and column parts of an operand's per-product offsets
// zb * (z / inner) + zh * (z % inner) in a buffer of row stride ld (KArgs);
// false when a column part could carry into the next row or a part would not
// fit an int (the launch then stages by plain loads, which take the offsets
// as they are).
static bool split_offsets(int64_t zb, int64_t zh, int64_t ld, int64_t count, int64_t inner,
                          int *rb, int *cb, int *rh, int *ch) {
    const int64_t nzb = (count + inner - 1) / inner, nzh = std::min(count, inner);
    const int64_t r_b = zb / ld, c_b = zb % ld, r_h = zh / ld, c_h = zh % ld;
    const int64_t lim = int64_t(1) << 31;
    if ((nzb - 1) * c_b + (nzh - 1) * c_h >= ld) return false;
    if ((nzb - 1) * r_b + (nzh - 1) * r_h >= lim) return false;
    *rb = int(r_b); *cb = int(c_b); *rh = int(r_h); *ch = int(c_h);
    return true;
}

cudaError_t launch_gemm_batched(const GemmArgs &a, const GemmBatch &bt, cudaStream_t s) {
    if (bt.count == 0 || a.M == 0 || a.N == 0) return cudaSuccess;
    if (a.K == 0) {
        for (int64_t z = 0; z < bt.count; ++z) {
            const int64_t zb = z / bt.inner, zh = z % bt.inner;
            const int64_t total = a.M * a.N;
            const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 32);
            fill_zero_kernel<<<unsigned(blocks), 256, 0, s>>>(
                a.C + zb * bt.c_zb + zh * bt.c_zh, a.ldc, a.M, a.N, a.accumulate);
        }
        return cudaGetLastError();
    }
    Prepared x{};
    KArgs &k = x.k;
    k.M = int(a.M); k.N = int(a.N); k.K = int(a.K);
    k.lda = a.lda; k.ldb = a.ldb; k.ldc = a.ldc;
    k.A = a.A; k.B = a.B; k.C = a.C;
    k.mt = int((a.M + BM - 1) / BM);
    k.nt = int((a.N + BN - 1) / BN);
    k.m_fast = a.M <= a.N;
    k.split = 0;
    k.units_per_tile = 1;
    k.kt_per_unit = int((a.K + BK - 1) / BK);
    k.W = nullptr;
    k.accumulate = a.accumulate;
    k.zcount = int(bt.count);
    k.zinner = int(bt.inner);
    k.a_zb = bt.a_zb; k.a_zh = bt.a_zh;
    k.b_zb = bt.b_zb; k.b_zh = bt.b_zh;
    k.c_zb = bt.c_zb; k.c_zh = bt.c_zh;
    k.causal = bt.causal;
    // triangular skipping needs a square op(A) (every row tile then meets
    // some k in range) and the flag
    k.tri = (bt.tri && bt.tri_bad && a.M == a.K && !bt.causal) ? bt.tri : 0;
    k.tri_bad = k.tri ? bt.tri_bad : nullptr;
    int64_t live = int64_t(k.mt) * k.nt;
    if (bt.causal) {
        live = 0;
        for (int mb = 0; mb < k.mt; ++mb)
            live += std::min<int64_t>(k.nt, (int64_t(mb) * BM + BM - 1) / BN + 1);
    }
    k.live_tiles = int(live);
    k.ctas0 = 0;
    const bool off4 = bt.a_zb % 4 == 0 && bt.a_zh % 4 == 0 && bt.b_zb % 4 == 0 &&
                      bt.b_zh % 4 == 0;
    k.vec_store = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 4 == 0) &&
                  bt.c_zb % 4 == 0 && bt.c_zh % 4 == 0;
    x.a_km = !a.transA;
    x.b_km = a.transB != 0;
    // one map spans each whole buffer; a product's tile coordinates add its
    // offset's row and column, which TMA needs on a 16-byte boundary
    x.tma = off4 && tma_ok(a.A, a.lda) && tma_ok(a.B, a.ldb) &&
            bt.a_rows < (int64_t(1) << 31) && bt.b_rows < (int64_t(1) << 31) &&
            split_offsets(bt.a_zb, bt.a_zh, a.lda, bt.count, bt.inner, &k.a_rb, &k.a_cb,
                          &k.a_rh, &k.a_ch) &&
            split_offsets(bt.b_zb, bt.b_zh, a.ldb, bt.count, bt.inner, &k.b_rb, &k.b_cb,
                          &k.b_rh, &k.b_ch);
    if (x.tma) {
        x.tma = make_map(&x.ma, a.A, bt.a_cols, bt.a_rows, a.lda, x.a_km, BM) &&
                make_map(&x.mb, a.B, bt.b_cols, bt.b_rows, a.ldb, x.b_km, BN);
    }
    return launch_prepared(x, nullptr, s);
}

#if DET_GEMM_PRIMARY
cudaError_t launch_transpose_copy(const float *A, int64_t lda, int64_t M, int64_t K, float *T,
                                  int64_t ldt, cudaStream_t s) {
    if (M == 0 || K == 0) return cudaSuccess;
    return launch_transpose(A, lda, M, K, T, ldt, sm_count_current_device(), s);
}

// ---------------------------------------------------------------- no-allocation variant
// Some callers cannot allocate device memory at the moment they multiply: code
// running inside another framework's memory pool, where every allocation must
// go through that pool, or a latency-critical loop where cudaMalloc's implicit
// device synchronisation is not acceptable. For them detgemm_f32_noalloc runs
// the split-K GEMM with its chunk partials in this fixed, file-scope scratch
// array instead of a caller workspace. The array exists on every device that
// loads this library, for the life of the process.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;   // 64 MiB
static __device__ __align__(256) float4 g_static_scratch[kStaticScratchBytes / 16];

namespace {
std::mutex g_scratch_mu;
// Per device: the array's device address, and the unique id of the CUDA
// context it was looked up in. A device reset destroys that context and the
// module with it; the next context has another id, so the address is looked
// up again there.
void *g_scratch_ptr[64];
unsigned long long g_scratch_ctx[64];

typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_fns_once;

// The unique id of the calling thread's current context (0 if unavailable).
unsigned long long current_context_id() {
    std::call_once(g_ctx_fns_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current && g_ctx_get_id && g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx &&
        g_ctx_get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}
}  // namespace

// The device address of g_static_scratch on the current device. Looked up
// once per device and context (the host-side name of a __device__ array is
// not a device address), with that device current.
static cudaError_t static_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // 0 when no context is current yet in this thread (or the driver calls
    // are missing): the address is then looked up, and again on the next call
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

cudaError_t launch_gemm_noalloc(const GemmArgs &a, bool *too_big, cudaStream_t s) {
    *too_big = false;
    const GemmPlan pl = gemm_plan(a.M, a.N, a.K, sm_count_current_device(), !a.transA,
                                  a.transB ? 1 : 0);
    if (pl.split && pl.split_bytes > kStaticScratchBytes) {
        *too_big = true;
        return cudaSuccess;
    }
    // a transposed copy of A that does not fit is skipped: launch_gemm then
    // reads A in place (same bits, a little slower)
    void *scratch = nullptr;
    if (pl.split || pl.transpose_a || pl.transpose_b || pl.head_rows) {
        const cudaError_t e = static_scratch(&scratch);
        if (e != cudaSuccess) return e;
    }
    // every slot of the scratch that is read is written first by this call, so
    // nothing needs clearing between calls
    return launch_gemm(a, scratch, scratch ? kStaticScratchBytes : 0, s);
}

#endif  // DET_GEMM_PRIMARY

cudaError_t gemm_watchdog(unsigned int *code, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemm_watchdog, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear && *code) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_watchdog, &zero, sizeof(unsigned int));
    }
    return e;
}

#if !DET_GEMM_PRIMARY
}  // namespace DET_GEMM_SECONDARY_NS
#endif
}  // namespace det
