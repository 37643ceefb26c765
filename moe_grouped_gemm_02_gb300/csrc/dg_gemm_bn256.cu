// Instantiation of the FP8 GEMM kernel with a 256-column tile, 4 pipeline stages and 1
// TMEM accumulator buffer(s).  One configuration per file so that they compile in parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn256_s4_a1, 256, 4, 1, 1)
}  // namespace dg
