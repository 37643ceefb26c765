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

// Per-row scales of more than 256 rows (gran_mn = 1, the activations' scales packed every step): the pack is a
// transpose, [row][K block] floats to [word][row] words.  Each CTA stages a tile of PACK_ROWS
// rows x PACK_WORDS words (32 K blocks) through shared memory: a warp loads one row's 32
// scales per instruction (128 contiguous bytes), each becomes one UE8M0 byte of a row-major
// byte tile, then the words go out along the rows (coalesced).  Tile rows are padded to an odd
// number of words, so the word reads of consecutive rows fall in distinct banks.
constexpr int PACK_ROWS = 64;
constexpr int PACK_WORDS = 8;
constexpr int PACK_STRIDE = PACK_WORDS + 1;   // words per tile row

__global__ void __launch_bounds__(256) pack_sf_rows_kernel(const float* __restrict__ sf, int32_t* __restrict__ out,
                                                           int MN, int Kb, int Kp, int mn_al) {
    __shared__ uint32_t tile[PACK_ROWS * PACK_STRIDE];
    griddep_wait();
    griddep_launch_dependents();
    const int r0 = blockIdx.x * PACK_ROWS;
    const int kp0 = blockIdx.y * PACK_WORDS;
    const int g = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint8_t* bytes = reinterpret_cast<uint8_t*>(tile);
    const int kb = 4 * kp0 + lane;
    // warp w takes rows w, w + 8, ...: one 32-scale row segment per load, all in flight at once
#pragma unroll
    for (int r = warp; r < PACK_ROWS; r += 8) {
        const int row = r0 + r;
        uint32_t code = 0u;
        if (row < MN && kb < Kb) code = ue8m0_code_ceil(__ldg(sf + (static_cast<size_t>(g) * MN + row) * Kb + kb));
        bytes[r * 4 * PACK_STRIDE + lane] = static_cast<uint8_t>(code);
    }
    __syncthreads();
    // word kp of row r: bytes 4kp..4kp+3 of the row (little-endian: K block 4kp in byte 0)
    for (int i = threadIdx.x; i < PACK_ROWS * PACK_WORDS; i += blockDim.x) {
        const int w = i / PACK_ROWS, r = i - w * PACK_ROWS;
        if (kp0 + w < Kp && r0 + r < mn_al)
            out[(static_cast<size_t>(g) * Kp + kp0 + w) * mn_al + r0 + r] = static_cast<int32_t>(tile[r * PACK_STRIDE + w]);
    }
}

cudaError_t launch_pack_sf(const float* sf, int32_t* out, int G, int MN, int MNb, int Kb, int Kp,
                           int mn_al, int gran_mn, int pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    // (a few hundred rows leave the tiled kernel with too few CTAs to hide the load latency:
    // there one thread per word, Kp CTAs per 256 rows, is faster)
    if (gran_mn == 1 && MN > 256) {
        cfg.gridDim = dim3((mn_al + PACK_ROWS - 1) / PACK_ROWS, (Kp + PACK_WORDS - 1) / PACK_WORDS, G);
        return cudaLaunchKernelEx(&cfg, pack_sf_rows_kernel, sf, out, MN, Kb, Kp, mn_al);
    }
    cfg.gridDim = dim3((mn_al + 255) / 256, Kp, G);
    return cudaLaunchKernelEx(&cfg, pack_sf_kernel, sf, out, MN, MNb, Kb, Kp, mn_al, gran_mn);
}

// K-grouped pack: FP32 scales sf [sum_g Kb_g][MN] (one per K block of 128 rows and per column
// of an MN-major operand) -> int32 [sum_g ceil(Kb_g / 4)][mn_al], each group packed on its own
// (its first K block starts a new word).  (README "News" 2025.05.14 and API list:
// get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor.)  The group sizes are read on the
// device: every CTA first forms the prefix sums of the groups' K blocks and word rows in shared
// memory, then each thread fills one word; threads past the last group's rows write nothing.
__global__ void __launch_bounds__(256) pack_sf_k_grouped_kernel(const float* __restrict__ sf, int32_t* __restrict__ out,
                                                                const int32_t* __restrict__ ks, int G, int MN,
                                                                int mn_al, int kb_total) {
    extern __shared__ int pk[];          // [0, G]: first K block of each group; [G+1, 2G+1]: first word row
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int per = (G + 255) / 256;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    // clip the groups to the call's K extent (a broken contract still reads only sf's rows)
    auto kb_raw = [&](int g) { return max(__ldg(ks + g), 0) / 128; };
    int run_kb = 0, run_kp = 0;
    for (int g = g0; g < g1; ++g) {
        run_kb += kb_raw(g);
        run_kp += (kb_raw(g) + 3) / 4;
    }
    int* scan = pk + 2 * (G + 1);       // 2 x 256 ints of scratch
    scan[tid] = run_kb;
    scan[256 + tid] = run_kp;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {   // inclusive Hillis-Steele scan, 8 steps
        const int a = tid >= off ? scan[tid - off] : 0;
        const int b = tid >= off ? scan[256 + tid - off] : 0;
        __syncthreads();
        scan[tid] += a;
        scan[256 + tid] += b;
        __syncthreads();
    }
    int acc_kb = scan[tid] - run_kb, acc_kp = scan[256 + tid] - run_kp;
    for (int g = g0; g < g1; ++g) {
        pk[g] = acc_kb;
        pk[G + 1 + g] = acc_kp;
        acc_kb += kb_raw(g);
        acc_kp += (kb_raw(g) + 3) / 4;
    }
    if (tid == 255) {
        pk[G] = scan[255];
        pk[2 * G + 1] = scan[511];
    }
    __syncthreads();

    const int r = blockIdx.x * blockDim.x + tid;
    const int w = blockIdx.y;
    if (r >= mn_al || w >= pk[2 * G + 1]) return;
    int lo = 0, hi = G - 1;                      // the group whose word rows hold w
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pk[G + 1 + mid] <= w) lo = mid; else hi = mid - 1;
    }
    const int kb0 = pk[lo];
    const int kbn = min(pk[lo + 1], kb_total) - min(kb0, kb_total);
    const int j = w - pk[G + 1 + lo];
    uint32_t word = 0;
    if (r < MN) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kb = 4 * j + i;
            if (kb < kbn) word |= ue8m0_code_ceil(__ldg(sf + static_cast<size_t>(kb0 + kb) * MN + r)) << (8 * i);
        }
    }
    out[static_cast<size_t>(w) * mn_al + r] = static_cast<int32_t>(word);
}

cudaError_t launch_pack_sf_k_grouped(const float* sf, int32_t* out, const int32_t* ks, int G, int MN, int mn_al,
                                     int kb_total, int pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((mn_al + 255) / 256, kb_total / 4 + G, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(2 * (G + 1) + 512) * sizeof(int);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, pack_sf_k_grouped_kernel, sf, out, ks, G, MN, mn_al, kb_total);
}

}  // namespace dg
