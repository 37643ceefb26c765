// Instantiation of the FP8 GEMM kernel with a 64-column tile, 8 pipeline stages and 2
// TMEM accumulator buffer(s).  One configuration per file so that they compile in parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn64_s8_a2, 64, 8, 2, 1)
}  // namespace dg
