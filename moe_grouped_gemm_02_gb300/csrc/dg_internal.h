// Types shared between the host dispatcher and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dg {

enum : int { MODE_DENSE = 0, MODE_CONTIGUOUS = 1, MODE_MASKED = 2, MODE_K_GROUPED = 3 };

// Timeout sites recorded in the device error word (bits 8..15), DG_ERR_TIMEOUT in bits 0..7.
enum : int { SITE_EMPTY = 1, SITE_FULL = 2, SITE_TMEM_EMPTY = 3, SITE_TMEM_FULL = 4, SITE_SF_EMPTY = 5, SITE_RED_EMPTY = 6, SITE_RED_FULL = 7,
             SITE_SF_READY = 8, SITE_SF_FULL = 9, SITE_RED_UNIT = 10 };

struct GemmArgs {
    int rows;           // rows of A and D per group: M (dense), M_sum (contiguous), max_m (masked),
                        // M (K-grouped)
    int N, K;           // K: the whole K extent (K-grouped: the sum over the groups)
    int mode;           // MODE_*
    int groups;         // groups of A and D (masked and K-grouped: G; otherwise 1)
    int b_groups;       // groups of B (dense: 1; contiguous and masked: G)
    int num_m_blocks;   // ceil(rows / 128)
    int num_n_blocks;   // ceil(N / BN)
    int kblocks;        // K / 128
    int raster_n;       // n-blocks per raster band (dense and contiguous)
    int num_units;      // tiles to compute (dense and contiguous); masked counts on the device
    int split;          // CTAs (a thread-block cluster) sharing one tile's K range: 1, 2, 4 or 8
    int num_m_units;    // m-tiles: 128-row blocks, or 256-row pairs of them when MH = 2
    int a_mn;           // 1: A is stored MN-major ([K, rows], rows contiguous)
    int b_mn;           // 1: B is stored MN-major ([K, N], N contiguous)
    int out_f32;        // 1: D is FP32; 0: BF16
    int b_fp4;          // 1: B is E2M1, unpacked by TMA into 16-byte units of 16 values
    const int32_t* m_indices;
    const int32_t* masked_m;
    const int32_t* ks;  // K-grouped: K rows of each group (multiples of 128)
    const float* c;     // FP32 C added to the accumulators (out_f32 only; may alias d), or null
    void* d;            // BF16 bit patterns or FP32
    int* err;           // device error word
    unsigned long long timeout_ns;
    int debug_drop_stage;   // test hook: the producer skips this stage's loads (-1: never)
    int pdl;                // launch with programmatic dependent launch
    int tma_store;          // the epilogue writes D through its tensor map (else plain stores)
    int prefetch_b;         // before its dependency wait, each CTA prefetches its first tile's B slice
                            // into L2 (weights that fit in L2 many times over)
    int d_evict_first;      // D is larger than L2: its TMA stores carry an L2 evict-first hint so that
                            // they do not push the operand tiles still being re-read out of L2
    int c_reduce;           // FP32 C is D itself and D goes out through its tensor map: the epilogue's
                            // boxes are added to D in place by TMA reductions (no C loads)
};

// Shared-memory ints after the barriers: the masked-mode m-unit prefix sums (G + 1) or the
// K-grouped K-block and scale-row prefix sums (2 (G + 1)).
__host__ __device__ inline int extra_smem_ints(int mode, int groups) {
    return mode == MODE_MASKED ? groups + 1 : (mode == MODE_K_GROUPED ? 2 * (groups + 1) : 0);
}

// maps: A, B, scales of A, scales of B, D (32 x 32-byte boxes), D (BF16: 64-column x 32-row
// boxes in the 128-byte swizzle, for whole-tile stores from the idle operand ring)
using GemmLaunchFn = cudaError_t (*)(const CUtensorMap* maps, const GemmArgs& args, int grid,
                                     cudaStream_t stream);

struct KernelConfig {
    int bn;             // N tile (columns of D per tile)
    int stages;         // shared-memory pipeline depth
    int acc;            // TMEM accumulator buffers
    int mh;             // 128-row halves per tile (2: one B tile serves 256 rows)
    int ks;             // MMA issuers splitting each stage's K steps (2: both accumulators serve one tile)
    int a_rows;         // A rows loaded per 128-row half: 128, or 64 (calls with at most 64 rows of A)
    const char* name;
    size_t (*smem_bytes)(int extra_ints, int split, int tma_store);
    GemmLaunchFn launch;
    cudaError_t (*prepare)(int max_smem);   // per-device one-time kernel attribute setup
    int (*max_clusters)(int split, size_t smem);   // co-resident clusters of `split` CTAs
};

// One per instantiation translation unit.
const KernelConfig& config_bn256_s4_a1();
const KernelConfig& config_bn224_s4_a2();
const KernelConfig& config_bn192_s5_a2();
const KernelConfig& config_bn128_s6_a2();
const KernelConfig& config_bn128_s4_a2();
const KernelConfig& config_bn64_s8_a2();
const KernelConfig& config_bn32_s8_a2();
const KernelConfig& config_bn224_s3_m2();
const KernelConfig& config_bn192_s3_m2();
const KernelConfig& config_bn208_s3_m2();
const KernelConfig& config_bn128_s5_k2();
const KernelConfig& config_bn192_s5_k2();
const KernelConfig& config_bn128_s8_k2_r64();

cudaError_t launch_pack_sf(const float* sf, int32_t* out, int G, int MN, int MNb, int Kb, int Kp,
                           int mn_al, int gran_mn, int pdl, cudaStream_t stream);
cudaError_t launch_pack_sf_k_grouped(const float* sf, int32_t* out, const int32_t* ks, int G, int MN, int mn_al,
                                     int kb_total, int pdl, cudaStream_t stream);
cudaError_t launch_quantize_fp8_1x128(const void* x, void* q, int32_t* sf, int G, int M, int K, int pdl,
                                      cudaStream_t stream);

}  // namespace dg
