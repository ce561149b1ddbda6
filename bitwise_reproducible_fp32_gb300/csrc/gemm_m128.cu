// gemm_m128.cu -- the fixed-order GEMM kernel with 128 x 64 CTA tiles, for the
// triangular batched products of causal attention whose N is a head's width
// (P V, and the backward's dV, dQ and dK over 64-wide heads).
//
// Same arithmetic and bits as gemm.cu: the thread tile stays 16 x 8, and a CTA
// of 1 x 2 warps covers 128 x 64. In a triangular product the row blocks
// carry from one to seq / 256 chunks of work; with 256-row tiles the longest
// units (a whole row of chunks, at least 1/8 of the work of a head at seq
// 2048) bound the kernel while the mean load per CTA is well below them.
// Halving the tile height halves every unit, so the descending-work order
// (unit_of) evens the CTAs' loads. Four such CTAs share an SM (eight warps,
// as one CTA of gemm.cu); their stages (2 x 24 KB each) sit in shared memory
// and the running chunk totals (32 KB a CTA) in Tensor Memory, 128 of its 512
// columns a CTA.
#define DET_GEMM_TN 8
#define DET_GEMM_WARPS_M 1
#define DET_GEMM_WARPS_N 2
#define DET_GEMM_CTAS_PER_SM 4
#define DET_GEMM_STAGES 2
#define DET_GEMM_TMEM 1
#define DET_GEMM_SECONDARY_NS m128
#include "gemm.cu"
