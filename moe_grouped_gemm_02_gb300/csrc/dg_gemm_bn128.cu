// Instantiation of the FP8 GEMM kernel with a 128-column tile, 6 pipeline stages and 2
// TMEM accumulator buffer(s).  One configuration per file so that they compile in parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn128_s6_a2, 128, 6, 2, 1)
}  // namespace dg
