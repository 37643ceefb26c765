// Instantiation of the FP8 GEMM kernel with a 256 x 208 tile (two 128-row halves), 3 pipeline
// stages and 1 TMEM accumulator buffer.  One configuration per file so that they compile in
// parallel.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn208_s3_m2, 208, 3, 1, 2)
}  // namespace dg
