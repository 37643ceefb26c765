// Instantiation of the FP8 GEMM kernel with a 224-column tile, 4 pipeline stages and 2
// TMEM accumulator buffer(s).  One configuration per file so that they compile in parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn224_s4_a2, 224, 4, 2, 1)
}  // namespace dg
