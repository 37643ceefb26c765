// Instantiation of the FP8 GEMM kernel with a 128-column tile, 4 pipeline stages and 2 TMEM
// accumulator buffers: the shallower ring leaves shared memory for the split-K receive buffer.
#include "dg_gemm_kernel.cuh"

namespace dg {
DG_DEFINE_CONFIG(config_bn128_s4_a2, 128, 4, 2, 1)
}  // namespace dg
