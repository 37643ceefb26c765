// Instantiation of the FP8 GEMM kernel with a 192-column tile, 5 pipeline stages and 2
// TMEM accumulator buffer(s).  One configuration per file so that they compile in parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn192_s5_a2, 192, 5, 2, 1)
}  // namespace dg
