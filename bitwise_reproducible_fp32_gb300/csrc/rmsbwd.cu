// rmsbwd.cu -- RMSNorm backward for sm_103a: dx by rows, dgain by 256-row
// chunks of columns.
//
// What it computes (profile v1; the pages define the forward -- "MojoLearn
// 162M" model card, table "Compared with GPT-3 Small" -- and fix the reduction
// order and partitioning of every operation -- "mojolearn" PyPI page, section
// "What bitwise identity means, and why it is not the default"), per row with
// r the forward's inv_rms:
//   xhat_j = x_j r,  h_j = dy_j g_j;
//   dot = the 32-chain arrangement of the forward's sum of squares over
//         fmaf(h_j, xhat_j, .), folded by the xor butterfly 16..1;
//   dx_j = (h_j - xhat_j (dot / D)) r;
// and dgain_j, a contraction over the rows, in the GEMM's spelling: a chain
// of fmaf(dy_ij, xhat_ij, .) from +0 over each 256-row chunk in ascending
// row, the chunk partials added left to right.
//
// Design for GB300:
//  * dgain's parallelism is (chunk, column): 32 chunks x 768 columns at the
//    162M shape, each a 256-long dependent chain. A one-warp CTA takes one
//    chunk of 32 columns; TMA brings the chunk's x and dy as 64-row boxes
//    (8 KB each) through a ring of two slots, and lane j adds each box's rows
//    to column j's chain while the next box is in flight. At ~35 KB a CTA six
//    share an SM, which keeps ~200 KB of loads in flight per SM, what
//    saturating HBM takes. This kernel runs first; x and dy (50 MB at the
//    162M shape) stay in the 129 MB L2 for the next one.
//  * dx: a CTA's 8 rows of x and dy and the gain arrive by 1-D bulk copies
//    into shared memory on one mbarrier (again many bytes in flight for few
//    registers); then a warp a row in the forward kernel's layout (lane l
//    owns the float4 groups l, l + 32, ...): the dot, then dx, both from
//    shared memory, so x and dy are read once (from L2) and dx written once.
//    Its first CTAs also fold dgain's chunk partials left to right.
//  * Rows or strides that TMA or 16-byte copies cannot describe take the same
//    arithmetic with scalar loads.
#include <algorithm>

#include "det_internal.cuh"

namespace det {
namespace {

#ifndef DET_RMSBWD_COLS
#define DET_RMSBWD_COLS 32
#endif
#ifndef DET_RMSBWD_BOX_ROWS
#define DET_RMSBWD_BOX_ROWS 64
#endif
constexpr int kCols = DET_RMSBWD_COLS;           // columns of a chunk task, one a thread
constexpr int kBoxRows = DET_RMSBWD_BOX_ROWS;    // rows of a TMA box
constexpr int kRing = 2;                         // boxes in flight a CTA
constexpr unsigned kWatchdogRmsBwd = 4u;         // det_watchdog_status bit 2
constexpr size_t kBoxFloats = size_t(kBoxRows) * kCols;
constexpr size_t kColsSmem = 1024 + 2 * kRing * kBoxFloats * 4 + kKChunk * 4 + kRing * 8;
static_assert(kKChunk % kBoxRows == 0, "boxes tile the chunk");
static_assert(kCols % 32 == 0 && kCols <= 256, "whole warps; a TMA box is at most 256 wide");

__device__ unsigned int g_rmsbwd_watchdog;

struct ColArgs {
    int64_t rows, D, ldx, lddy;
    int64_t ncb;                 // column blocks
    const float *x, *dy, *inv;
    float *out;                  // dgain (one chunk) or partials [chunk][D]
};

__device__ __forceinline__ void issue_box(float *xs, float *ds, uint64_t *bar,
                                          const CUtensorMap *tmX, const CUtensorMap *tmD,
                                          int64_t j0, int64_t row0) {
    const uint32_t bb = smem_u32(bar);
    mbar_arrive_expect_tx(bb, 2u * kBoxRows * kCols * 4u);
    tma_load_2d(smem_u32(xs), tmX, int(j0), int(row0), bb);
    tma_load_2d(smem_u32(ds), tmD, int(j0), int(row0), bb);
}

// One CTA per (chunk, kCols-column block), a thread a column. The chunk's
// rows arrive as boxes of x and dy through a ring of two slots: while the
// threads add one box's rows to their columns' chains, the next box is in
// flight. Without TMA the CTA copies each box with coalesced scalar loads.
template <bool TMA>
__global__ void __launch_bounds__(kCols)
    rmsbwd_cols_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmD, const ColArgs a) {
    extern __shared__ unsigned char smem_raw[];
    float *xs = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *ds = xs + kRing * kBoxFloats;
    float *rs = ds + kRing * kBoxFloats;
    uint64_t *bar = reinterpret_cast<uint64_t *>(rs + kKChunk);
    // this grid is itself a programmatic dependent: once the previous grid
    // (the producer of x, dy or inv_rms) is complete, the dx kernel may start
    // (it reads x and dy at once, and waits for this grid only where it folds
    // the partials)
    grid_dependency_wait();
    allow_dependents();
    const int t = threadIdx.x;
    const int64_t c = int64_t(blockIdx.x) / a.ncb;
    const int64_t j0 = (int64_t(blockIdx.x) % a.ncb) * kCols;
    const int64_t i0 = c * kKChunk;
    const int nr = int(min(int64_t(kKChunk), a.rows - i0));
    const int nb = (nr + kBoxRows - 1) / kBoxRows;
    if (TMA && t == 0) {
        for (int k = 0; k < kRing; ++k) mbar_init(smem_u32(&bar[k]), 1);
        fence_mbar_init();
        for (int b = 0; b < kRing && b < nb; ++b)
            issue_box(xs + b * kBoxFloats, ds + b * kBoxFloats, &bar[b], &tmX, &tmD, j0,
                      i0 + b * kBoxRows);
    }
    for (int i = t; i < nr; i += kCols) rs[i] = a.inv[i0 + i];
    __syncthreads();

    // column j0 + t: fmaf chain over the chunk's rows, ascending
    float acc = 0.0f;
    bool ok = true;
    for (int b = 0; b < nb; ++b) {
        const int slot = b % kRing;
        float *xb = xs + slot * kBoxFloats, *db = ds + slot * kBoxFloats;
        const int e = min(nr - b * kBoxRows, kBoxRows);
        if (TMA) {
            ok = __syncthreads_and(
                mbar_wait_bounded(smem_u32(&bar[slot]), uint32_t(b / kRing) & 1u));
            if (!ok) break;
        } else {
            const int64_t j = j0 + t;
            for (int i = 0; i < e; ++i) {
                const int64_t row = i0 + b * kBoxRows + i;
                xb[i * kCols + t] = j < a.D ? a.x[row * a.ldx + j] : 0.0f;
                db[i * kCols + t] = j < a.D ? a.dy[row * a.lddy + j] : 0.0f;
            }
            __syncthreads();
        }
        const float *rb = rs + b * kBoxRows;
#pragma unroll 8
        for (int i = 0; i < e; ++i)
            acc = __fmaf_rn(db[i * kCols + t], __fmul_rn(xb[i * kCols + t], rb[i]), acc);
        __syncthreads();    // every thread is done with this slot
        if (TMA && t == 0 && b + kRing < nb) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_box(xb, db, &bar[slot], &tmX, &tmD, j0, i0 + (b + kRing) * kBoxRows);
        }
    }
    if (!ok) {
        // a box never landed: record it, and let the copies in flight finish
        // (or give up on them too) before the CTA's shared memory is released
        if (t == 0) {
            atomicOr(&g_rmsbwd_watchdog, kWatchdogRmsBwd);
            for (int k = 0; k < kRing; ++k) (void)mbar_wait_bounded(smem_u32(&bar[k]), 0);
            for (int k = 0; k < kRing; ++k) (void)mbar_wait_bounded(smem_u32(&bar[k]), 1);
        }
        __syncthreads();
        return;
    }
    const int64_t j = j0 + t;
    if (j < a.D) a.out[c * a.D + j] = acc;
}

struct RowArgs {
    int64_t rows, D, ldx, lddy, lddx;
    const float *x, *gain, *inv, *dy;
    float *dx;
    const float *partials;       // [nchunks][D], nchunks > 1
    float *dgain;
    int64_t nchunks;
};

constexpr int kRowWarps = 8;

__device__ __forceinline__ float butterfly32(float s) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// dgain_j = P_0 + P_1 + ... left to right, for the columns of this CTA.
__device__ __forceinline__ void fold_partials(const RowArgs &a) {
    if (a.nchunks <= 1) return;
    if (int64_t(blockIdx.x) * (kRowWarps * 32) >= a.D) return;
    // the partials are complete and visible once the column grid has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t j = int64_t(blockIdx.x) * (kRowWarps * 32) + threadIdx.x;
    if (j >= a.D) return;
    float t = a.partials[j];
    for (int64_t c = 1; c < a.nchunks; ++c) t = __fadd_rn(t, a.partials[c * a.D + j]);
    a.dgain[j] = t;
}

// Dense rows (strides == D) that are 16-byte aligned with D % 4 == 0: the
// CTA's 8 rows of x and of dy and the gain arrive by three bulk copies into
// shared memory on one mbarrier (few large copies: many small ones measured
// slow), so each SM keeps ~200 KB of loads in flight with few registers; then
// a warp a row: pass 1 the dot, pass 2 dx, both from shared memory, lane l
// taking the float4 groups l, l + 32, ...
__global__ void __launch_bounds__(kRowWarps * 32) rmsbwd_rows_bulk_kernel(const RowArgs a) {
    extern __shared__ unsigned char smem_raw[];
    float4 *gs = reinterpret_cast<float4 *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int ng = int(a.D >> 2);
    float4 *xs = gs + ng;                       // [kRowWarps][ng]
    float4 *dys = xs + size_t(kRowWarps) * ng;
    uint64_t *bar = reinterpret_cast<uint64_t *>(dys + size_t(kRowWarps) * ng);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r0 = int64_t(blockIdx.x) * kRowWarps;
    const int nrows = int(max(int64_t(0), min(int64_t(kRowWarps), a.rows - r0)));
    const uint32_t row_bytes = uint32_t(a.D) * 4u;
    if (threadIdx.x == 0 && nrows > 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(smem_u32(bar), row_bytes * uint32_t(2 * nrows + 1));
        // the CTA's rows are contiguous (row strides == D): one copy an array
        bulk_load(smem_u32(gs), a.gain, row_bytes, smem_u32(bar));
        bulk_load(smem_u32(xs), a.x + r0 * a.ldx, row_bytes * uint32_t(nrows), smem_u32(bar));
        bulk_load(smem_u32(dys), a.dy + r0 * a.lddy, row_bytes * uint32_t(nrows),
                  smem_u32(bar));
    }
    __syncthreads();
    if (nrows > 0) {
        const bool ok = __syncthreads_and(mbar_wait_bounded(smem_u32(bar), 0));
        if (!ok) {
            if (threadIdx.x == 0) atomicOr(&g_rmsbwd_watchdog, kWatchdogRmsBwd);
            return;
        }
        if (warp < nrows) {
            const int64_t row = r0 + warp;
            const float r = a.inv[row];
            const float4 *xr = xs + size_t(warp) * ng, *dr = dys + size_t(warp) * ng;
            float s = 0.0f;
            for (int g = lane; g < ng; g += 32) {
                const float4 xv = xr[g], dv = dr[g], gv = gs[g];
                s = __fmaf_rn(__fmul_rn(dv.x, gv.x), __fmul_rn(xv.x, r), s);
                s = __fmaf_rn(__fmul_rn(dv.y, gv.y), __fmul_rn(xv.y, r), s);
                s = __fmaf_rn(__fmul_rn(dv.z, gv.z), __fmul_rn(xv.z, r), s);
                s = __fmaf_rn(__fmul_rn(dv.w, gv.w), __fmul_rn(xv.w, r), s);
            }
            const float q = __fdiv_rn(butterfly32(s), float(a.D));
            float4 *o = reinterpret_cast<float4 *>(a.dx + row * a.lddx);
            for (int g = lane; g < ng; g += 32) {
                const float4 xv = xr[g], dv = dr[g], gv = gs[g];
                o[g] = make_float4(
                    __fmul_rn(__fsub_rn(__fmul_rn(dv.x, gv.x), __fmul_rn(__fmul_rn(xv.x, r), q)), r),
                    __fmul_rn(__fsub_rn(__fmul_rn(dv.y, gv.y), __fmul_rn(__fmul_rn(xv.y, r), q)), r),
                    __fmul_rn(__fsub_rn(__fmul_rn(dv.z, gv.z), __fmul_rn(__fmul_rn(xv.z, r), q)), r),
                    __fmul_rn(__fsub_rn(__fmul_rn(dv.w, gv.w), __fmul_rn(__fmul_rn(xv.w, r), q)), r));
            }
        }
    }
    fold_partials(a);
}

size_t rows_bulk_smem(int64_t D) { return 128 + size_t(2 * kRowWarps + 1) * size_t(D) * 4 + 8; }

// Any alignment and any D: the same operations with scalar loads, in two
// passes over the row (the dot, then dx). dx may equal dy: pass 2 reads dy_j
// before it writes dx_j.
__global__ void __launch_bounds__(kRowWarps * 32) rmsbwd_rows_kernel(const RowArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = int64_t(blockIdx.x) * kRowWarps + warp;
    if (row < a.rows) {
        const float *x = a.x + row * a.ldx;
        const float *dy = a.dy + row * a.lddy;
        float *dx = a.dx + row * a.lddx;
        const float r = a.inv[row];
        const int64_t ngroups = (a.D + 3) >> 2;
        float s = 0.0f;
        for (int64_t g = lane; g < ngroups; g += 32)
            for (int e = 0; e < 4; ++e) {
                const int64_t j = 4 * g + e;
                if (j < a.D)
                    s = __fmaf_rn(__fmul_rn(dy[j], a.gain[j]), __fmul_rn(x[j], r), s);
            }
        const float q = __fdiv_rn(butterfly32(s), float(a.D));
        for (int64_t g = lane; g < ngroups; g += 32)
            for (int e = 0; e < 4; ++e) {
                const int64_t j = 4 * g + e;
                if (j < a.D) {
                    const float h = __fmul_rn(dy[j], a.gain[j]);
                    dx[j] = __fmul_rn(__fsub_rn(h, __fmul_rn(__fmul_rn(x[j], r), q)), r);
                }
            }
    }
    fold_partials(a);
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

cudaError_t rmsbwd_watchdog(unsigned int *code, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_rmsbwd_watchdog, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_rmsbwd_watchdog, &z, sizeof(unsigned int));
}

size_t rmsnorm_bwd_workspace_bytes(int64_t rows, int64_t D) {
    const int64_t nchunks = (rows + kKChunk - 1) / kKChunk;
    return nchunks > 1 ? size_t(nchunks) * size_t(D) * 4 : 0;
}

cudaError_t launch_rmsnorm_bwd(int64_t rows, int64_t D, const float *x, int64_t ldx,
                               const float *gain, const float *inv_rms, const float *dy,
                               int64_t lddy, float *dx, int64_t lddx, float *dgain,
                               float *workspace, cudaStream_t s) {
    if (rows == 0) return cudaMemsetAsync(dgain, 0, size_t(D) * 4, s);   // +0: the empty sum
    const int64_t nchunks = (rows + kKChunk - 1) / kKChunk;
    const int64_t ncb = (D + kCols - 1) / kCols;
    if (nchunks * ncb >= (int64_t(1) << 31)) return cudaErrorInvalidValue;

    // 1. dgain's chunk partials (or dgain itself for a single chunk)
    const ColArgs ca{rows, D, ldx, lddy, ncb, x, dy, inv_rms, nchunks > 1 ? workspace : dgain};
    CUtensorMap mx{}, md{};
    const bool tma = tma_operand_ok(x, ldx) && tma_operand_ok(dy, lddy) &&
                     make_tensor_map_2d(&mx, x, D, rows, ldx, kCols, kBoxRows, false) &&
                     make_tensor_map_2d(&md, dy, D, rows, lddy, kCols, kBoxRows, false);
    auto ck = tma ? rmsbwd_cols_kernel<true> : rmsbwd_cols_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kColsSmem));
    if (e != cudaSuccess) return e;
    e = launch_dependent(ck, dim3(unsigned(nchunks * ncb)), dim3(kCols), kColsSmem, s, mx, md,
                         ca);
    if (e != cudaSuccess) return e;

    // 2. dx, and the left-to-right fold of the partials into dgain
    const RowArgs ra{rows, D, ldx, lddy, lddx, x, gain, inv_rms, dy, dx,
                     workspace, dgain, nchunks};
    int64_t blocks = (rows + kRowWarps - 1) / kRowWarps;
    if (nchunks > 1) blocks = std::max<int64_t>(blocks, (D + kRowWarps * 32 - 1) / (kRowWarps * 32));
    const dim3 grid{unsigned(blocks)}, block{unsigned(kRowWarps * 32)};
    const size_t bulk_smem = rows_bulk_smem(D);
    const bool bulk = D % 4 == 0 && bulk_smem <= 200 * 1024 && aligned16(x) && aligned16(dy) &&
                      aligned16(dx) && aligned16(gain) && ldx == D && lddy == D &&
                      lddx % 4 == 0;
    if (!bulk) {
        rmsbwd_rows_kernel<<<grid, block, 0, s>>>(ra);
        return cudaGetLastError();
    }
    e = cudaFuncSetAttribute(rmsbwd_rows_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(bulk_smem));
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent of the column kernel: its rows run
    // alongside the column chains, and the fold waits for them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = bulk_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, rmsbwd_rows_bulk_kernel, ra);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace det
