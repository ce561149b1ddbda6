// gemm_n64.cu -- the fixed-order GEMM kernel with 64-wide CTA tiles, for the
// batched products whose N is a head's width (P V and the attention backward's
// dV, dQ, dK over 64-wide heads).
//
// Same arithmetic and bits as gemm.cu (every output's chunk chains are one
// thread's accumulator sequence, whatever the tile): only the thread tile
// changes, 16 x 4 instead of 16 x 8, so a 256 x 64 CTA tile keeps all eight
// warps on live columns where the 256 x 128 tile would leave half of them
// computing columns that are thrown away. The narrower tile loads 20 floats
// from shared memory a k for 64 FMAs (16 x 8: 24 for 128), so it runs closer
// to the shared-memory limit; three stages of 40 KB fit beside its 64 KB of
// running totals.
#define DET_GEMM_TN 4
#define DET_GEMM_STAGES 3
#define DET_GEMM_SECONDARY_NS n64
#include "gemm.cu"
