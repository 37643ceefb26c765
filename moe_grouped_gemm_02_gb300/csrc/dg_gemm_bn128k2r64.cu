// Instantiation of the FP8 GEMM kernel with a 128-column tile, two K-split MMA issuers and
// 64-row A stages (calls with at most 64 rows of A): 8 pipeline stages of 8 KB of A and 16 KB
// of B, so that a split-K CTA of the M = 64 decode shapes has its whole weight slice in flight.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG_AR(config_bn128_s8_k2_r64, 128, 8, 2, 1, 2, 64)
}  // namespace dg
