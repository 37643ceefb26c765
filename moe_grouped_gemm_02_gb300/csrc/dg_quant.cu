// Per-token 1x128 FP8 quantisation: BF16 activations -> E4M3 codes plus their scales, written
// straight into the packed UE8M0 layout the GEMMs read.
// (DeepGEMM README, "Interface / Notes": FP8 quantisation of the inputs is the caller's job, to
// be written separately or fused into the kernel that produces them; "Utilities": the scales
// are MN-major, TMA-aligned, four UE8M0 bytes per int32.)
//
// Scale of a 1x128 block: 2^e with e the smallest integer such that 448 * 2^e >= amax,
// clamped to [-127, 127]; e = 0 for an all-zero block.  Codes: round-to-nearest-even of
// x * 2^-e, which is at most 448 in magnitude, so nothing saturates.
//
// Work unit: one warp takes one row and one packed word (four K blocks, 512 elements, 1 KB of
// BF16).  Lane l loads the 8 elements at 256*i + 8*l for i = 0, 1, so lanes 0-15 hold blocks
// 0 and 2 of the word and lanes 16-31 blocks 1 and 3; each block's amax is a 16-lane
// butterfly.  A warp's code stores are 2 x 256 contiguous bytes; the eight warps of a CTA take
// eight consecutive rows of one word column, so their scale words are 32 contiguous bytes.
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {

// Exponent e of the block scale from amax's FP32 bit pattern (amax >= 0, finite).
// amax = 2^E * (1 + m/2^23) is covered by 448 * 2^e = 1.75 * 2^(e+8) at e = E - 8 when
// 1 + m/2^23 <= 1.75 (m <= 0x600000), else at e = E - 7.  A subnormal amax is below
// 2^-126, so its e is under -127 and clamps there.
__device__ __forceinline__ int block_scale_exponent(uint32_t amax_bits) {
    if (amax_bits == 0u) return 0;
    const int ef = static_cast<int>(amax_bits >> 23);
    if (ef == 0) return -127;
    const int e = ef - 127 - ((amax_bits & 0x7FFFFFu) <= 0x600000u ? 8 : 7);
    return max(-127, min(127, e));
}

// Two FP32 values -> two E4M3 codes (RNE, saturating to finite), `lo` in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Elementwise unsigned maximum of two pairs of 16-bit halves.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Elementwise BF16 product of two pairs, rounded to nearest even.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Byte permute: the bytes of {b, a} picked by `sel` (four 4-bit indices).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

constexpr int QUANT_WARPS = 8;

// The arithmetic works on BF16 pairs as they are loaded:
//  * the block amax is an unsigned maximum of the magnitude bits (sign cleared), two halves
//    at a time, and both of a lane's blocks travel through one 16-lane butterfly (block i in
//    half i);
//  * the scaling by 2^-e is one BF16 pair product.  2^-e is a BF16 normal for every e a
//    finite BF16 block can have (e in [-127, 120]) and BF16 has FP32's exponent range, so the
//    product is exact whenever it is a normal number; a product below the normal range is
//    under 2^-126 and rounds to a signed zero in E4M3 whichever way it was rounded before;
//  * the two products are widened to FP32 (exactly) for the E4M3 conversion.
__global__ void __launch_bounds__(32 * QUANT_WARPS)
    quantize_fp8_1x128_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                              int M, int K, int Kb, int Kp, int m_al, int row_groups) {
    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // blockIdx.x -> (g, kp, group of eight rows); rows fastest so neighbouring CTAs share a
    // scale-word column.
    const int rg = blockIdx.x % row_groups;
    const int kp = (blockIdx.x / row_groups) % Kp;
    const int g = blockIdx.x / (row_groups * Kp);
    const int r = rg * QUANT_WARPS + warp;
    if (r >= m_al) return;

    const size_t row = static_cast<size_t>(g) * M + r;
    uint4 v[2];
    bool valid[2];
    uint32_t mx[2];   // per block: the two 16-bit halves' maximum magnitudes
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int kb = 4 * kp + 2 * i + (lane >> 4);
        valid[i] = r < M && kb < Kb;
        v[i] = valid[i] ? __ldcs(reinterpret_cast<const uint4*>(x + row * K + 512 * kp + 256 * i + 8 * lane))
                        : make_uint4(0u, 0u, 0u, 0u);
        // |x| as BF16 magnitude bits; for finite values their integer order is the value order
        mx[i] = max_u16x2(max_u16x2(v[i].x & 0x7FFF7FFFu, v[i].y & 0x7FFF7FFFu),
                          max_u16x2(v[i].z & 0x7FFF7FFFu, v[i].w & 0x7FFF7FFFu));
    }
    // block 0's halves in the low 16 bits of both words, block 1's in the high ones
    uint32_t m = max_u16x2(prmt(mx[0], mx[1], 0x5410u), prmt(mx[0], mx[1], 0x7632u));
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, off));

    uint32_t codes = 0;   // this lane's two UE8M0 bytes: block 2i + (lane >> 4) in byte i
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t amax = i == 0 ? (m & 0xFFFFu) : (m >> 16);
        const int e = block_scale_exponent(amax << 16);
        if (valid[i]) codes |= static_cast<uint32_t>(e + 127) << (8 * i);
        // 2^-e as a BF16 pair (e <= 120 for BF16 inputs, as 448 * 2^120 exceeds the BF16
        // maximum, so 127 - e >= 7 and the exponent field is a normal one)
        const uint32_t s2 = static_cast<uint32_t>(127 - e) * 0x00800080u;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t y = mul_bf16x2(w[j], s2);
            c[j] = cvt_e4m3x2(__uint_as_float(y << 16), __uint_as_float(y & 0xFFFF0000u));
        }
        if (valid[i])
            *reinterpret_cast<uint2*>(q + row * K + 512 * kp + 256 * i + 8 * lane) =
                make_uint2(prmt(c[0], c[1], 0x5410u), prmt(c[2], c[3], 0x5410u));
    }

    // byte j of the word is block 4*kp + j: blocks 0 and 2 sit in lane 0, 1 and 3 in lane 16
    const uint32_t other = __shfl_sync(0xffffffffu, codes, 16);
    if (lane == 0) {
        const uint32_t word = (codes & 0xFFu) | ((other & 0xFFu) << 8) | ((codes & 0xFF00u) << 8) |
                              ((other & 0xFF00u) << 16);
        sf[(static_cast<size_t>(g) * Kp + kp) * m_al + r] = static_cast<int32_t>(word);
    }
}

cudaError_t launch_quantize_fp8_1x128(const void* x, void* q, int32_t* sf, int G, int M, int K, int pdl,
                                      cudaStream_t stream) {
    const int Kb = K / 128;
    const int Kp = (Kb + 3) / 4;
    const int m_al = (M + 3) / 4 * 4;
    const int row_groups = (m_al + QUANT_WARPS - 1) / QUANT_WARPS;
    const long long blocks = static_cast<long long>(row_groups) * Kp * G;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(32 * QUANT_WARPS, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quantize_fp8_1x128_kernel, static_cast<const uint16_t*>(x),
                              static_cast<uint8_t*>(q), sf, M, K, Kb, Kp, m_al, row_groups);
}

}  // namespace dg
