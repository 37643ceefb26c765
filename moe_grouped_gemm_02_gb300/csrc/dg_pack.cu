// Scale-factor pack: FP32 scales -> MN-major, TMA-aligned, packed UE8M0 words.
// (DeepGEMM README, "Interface / Notes": UE8M0 scales, four per int32, transposed and
// TMA-aligned; "Utilities": get_mn_major_tma_aligned_packed_ue8m0_tensor.  The
// DeepGEMM-Ascend article, "Cómo funciona", packs scale pairs along K in MN-major order.)
//
// Output word [g][kp][r], byte j = UE8M0 code of the scale of row r and K block 4*kp + j.
// One thread per output word, rows fastest: the stores of a warp are 128 contiguous bytes.
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {

// Smallest b in 0..254 with 2^(b-127) >= x; 0xFE above 2^127; 0xFF for x <= 0, NaN or Inf.
// Works on the FP32 bit pattern: a normal x = 2^(e-127) * (1 + m/2^23) has the power
// 2^(e-127) when m == 0 and needs one exponent step up otherwise; a subnormal
// x = m * 2^-149 is at most 2^-127 exactly when m <= 2^22.
__device__ __forceinline__ uint32_t ue8m0_code_ceil(float x) {
    const uint32_t bits = __float_as_uint(x);
    if (!(x > 0.0f) || bits >= 0x7F800000u) return 0xFFu;
    const uint32_t e = bits >> 23;
    const uint32_t m = bits & 0x7FFFFFu;
    if (e == 0) return m > (1u << 22) ? 1u : 0u;
    const uint32_t b = e + (m != 0u ? 1u : 0u);
    return b > 254u ? 254u : b;
}

__global__ void __launch_bounds__(256) pack_sf_kernel(const float* __restrict__ sf, int32_t* __restrict__ out,
                                                      int MN, int MNb, int Kb, int Kp, int mn_al, int gran_mn) {
    griddep_wait();   // with programmatic dependent launch: the inputs' producer has finished
    griddep_launch_dependents();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    const int kp = blockIdx.y;
    const int g = blockIdx.z;
    if (r >= mn_al) return;
    uint32_t w = 0;
    if (r < MN) {
        const float* src = sf + (static_cast<size_t>(g) * MNb + r / gran_mn) * Kb;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kb = 4 * kp + j;
            if (kb < Kb) w |= ue8m0_code_ceil(__ldg(src + kb)) << (8 * j);
        }
    }
    out[(static_cast<size_t>(g) * Kp + kp) * mn_al + r] = static_cast<int32_t>(w);
}

cudaError_t launch_pack_sf(const float* sf, int32_t* out, int G, int MN, int MNb, int Kb, int Kp,
                           int mn_al, int gran_mn, int pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((mn_al + 255) / 256, Kp, G);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, pack_sf_kernel, sf, out, MN, MNb, Kb, Kp, mn_al, gran_mn);
}

}  // namespace dg
