// gemm_n64.cu -- the fixed-order GEMM kernel with 64-wide CTA tiles, for the
// batched products whose N is a head's width (P V and the attention backward's
// dV, dQ, dK over 64-wide heads).
//
// Same arithmetic and bits as gemm.cu (every output's chunk chains are one
// thread's accumulator sequence, whatever the tile): the thread tile stays 16
// x 8, and a CTA of 2 x 2 warps covers 256 x 64, so every warp works on live
// columns where the 256 x 128 tile would leave half of them computing columns
// that are thrown away. Two such CTAs share an SM (eight warps, as one CTA of
// gemm.cu): their stages (2 x 40 KB each) fill the shared memory, so the
// running chunk totals (64 KB a CTA) live in Tensor Memory, 128 of its 512
// columns a CTA.
#define DET_GEMM_TN 8
#define DET_GEMM_WARPS_M 2
#define DET_GEMM_WARPS_N 2
#define DET_GEMM_CTAS_PER_SM 2
#define DET_GEMM_STAGES 2
#define DET_GEMM_TMEM 1
#define DET_GEMM_SECONDARY_NS n64
#include "gemm.cu"
