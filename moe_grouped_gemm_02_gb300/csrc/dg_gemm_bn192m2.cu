// Instantiation of the FP8 GEMM kernel with 256 x 192 tiles (two 128-row halves sharing each
// B tile, one MMA issuer per half), 3 pipeline stages and one TMEM accumulator pair.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn192_s3_m2, 192, 3, 1, 2)
}  // namespace dg
