// Instantiation of the FP8 GEMM kernel with a 128-column tile, 5 pipeline stages and two MMA
// issuers splitting each stage's K steps into the two TMEM accumulators (the decode shapes).
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG_KS(config_bn128_s5_k2, 128, 5, 2, 1, 2)
}  // namespace dg
