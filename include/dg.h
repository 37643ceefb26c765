/*
 * dg.h -- C ABI of the GB300 (sm_103a) FP8 block-scaled GEMM library.
 *
 * The operations are those of DeepGEMM as its README describes them:
 *   "Interface / Notes"                 D = A @ B^T on FP8 (E4M3) operands with fine-grained
 *                                       scale factors; on SM100-class GPUs the scale factors
 *                                       are UE8M0, four packed into one int32, in a transposed
 *                                       (MN-major), TMA-aligned tensor; FP8 quantization is the
 *                                       caller's job.
 *   "Grouped GEMM (contiguous layout)"  only M is grouped; the tokens of all experts are
 *                                       concatenated, each expert segment aligned to the GEMM M
 *                                       block (get_mk_alignment_for_contiguous_layout).
 *   "Grouped GEMM (masked layout)"      for CUDA-graph decode where the host does not know the
 *                                       per-expert token counts: a device mask gives the valid
 *                                       rows of every group and only those are computed.
 *   "Utilities"                         get_tma_aligned_size, set_num_sms / get_num_sms,
 *                                       get_mn_major_tma_aligned_packed_ue8m0_tensor.
 * The DeepGEMM article (2048ai.net, section 4.2) gives the older argument order
 * (lhs, rhs, lhs_scale, rhs_scale, M, N, K) and the BF16 output; the calls below keep it.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer is a DEVICE pointer owned by the caller.  The library allocates and frees
 *    no memory in any of these calls.
 *  - All tensors are dense and row-major (last dimension contiguous) with the shapes given.
 *  - Every pointer must be 16-byte aligned (TMA requirement), else DG_ERR_ALIGNMENT.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL means the
 *    legacy default stream).  They never synchronize, except in validation mode (the
 *    environment variable DG_VALIDATE=1), where the device-side contracts below are read
 *    back and checked first.
 *  - Argument checks happen on the host before anything is launched; a failing check
 *    returns an error code and launches nothing.  Launch failures return DG_ERR_CUDA.
 *  - Scale factors ("SF") are packed UE8M0 words: word [kp][r] of an SF tensor holds in
 *    byte j (bits 8j..8j+7) the scale of row r for K block 4*kp + j (K blocks are 128
 *    wide), as a UE8M0 byte (value 2^(b-127)).  The row extent is padded to
 *    dg_get_tma_aligned_size(rows, 4) words.  Kp = ceil((K/128) / 4).
 *  - FP8 operands are E4M3 ("fn") bytes; D is BF16 (round-to-nearest-even of the FP32
 *    accumulator).
 *  - The environment variable DG_PRINT_CONFIGS=1 prints the kernel configuration chosen
 *    for each call to stderr; DG_NUM_SMS=n caps the SMs used (as dg_set_num_sms).
 *    DG_FORCE_CONFIG=<configuration name> / DG_FORCE_SPLIT=<1..8> pin the kernel plan
 *    (tuning and tests; the planner itself splits K over 1, 2, 4 or 8 CTAs);
 *    DG_TIMEOUT_MS sets the bound on each in-kernel barrier wait (default 4000) and
 *    DG_DEBUG_DROP_LOAD=n makes the GEMM skip its n-th load stage, so that a wait runs out:
 *    a test hook for the timeout path (dg_check_device_error then reports DG_ERR_TIMEOUT).
 *    Two performance switches, neither of which changes a result: DG_PREFETCH_B=0 / 1 turns
 *    off / forces the L2 prefetch of a dense GEMM's weight tiles before it waits for the
 *    previous kernel (by default on for weights of at most 64 MB whose grid leaves half the
 *    SMs idle); DG_D_EVICT_FIRST=0 stores an output larger than the L2 without the
 *    evict-first cache hint (by default the hint is on for outputs above 128 MB).
 */
#ifndef DG_H
#define DG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum value            */
    DG_ERR_SHAPE = 2,              /* K % 128 != 0, N % 8 != 0, M_sum % 128 != 0, too large  */
    DG_ERR_ALIGNMENT = 3,          /* a pointer is not 16-byte aligned                       */
    DG_ERR_UNSUPPORTED_DEVICE = 4, /* the current device is not compute capability 10.3     */
    DG_ERR_CUDA = 5,               /* a CUDA runtime or driver call failed                   */
    DG_ERR_TIMEOUT = 6,            /* a kernel gave up waiting on one of its barriers        */
    DG_ERR_CONTRACT = 7            /* validation mode found a bad m_indices / masked_m entry */
} dg_status;

/*
 * Dense GEMM, NT layout:  D[m, n] = bf16( sum_k A[m,k] * sa(m, k/128) * B[n,k] * sb(n, k/128) )
 * (README "Interface / Notes": fp8_gemm_nt; article section 4.2: gemm_fp8_fp8_bf16_nt).
 *
 *   a    E4M3  [M, K]              activations ("lhs")
 *   sfa  int32 [Kp][al4(M)]        packed UE8M0 scales of A, one per row and 1x128 block
 *   b    E4M3  [N, K]              weights ("rhs"), stored N-major (the "T" of NT)
 *   sfb  int32 [Kp][al4(N)]        packed UE8M0 scales of B, one word per row of B
 *                                  (a 128x128 block scale broadcast to its rows by
 *                                  dg_pack_sf_ue8m0 with gran_mn = 128)
 *   d    BF16  [M, N]              output, fully overwritten
 * Requires M >= 0 (M == 0 is a no-op), N > 0 with N % 8 == 0, K > 0 with K % 128 == 0.
 */
dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         void* d, int M, int N, int K, void* stream);

/*
 * M-grouped GEMM, contiguous layout (README "Grouped GEMM (contiguous layout)";
 * article section 5.1, "contiguous grouping" for training and prefill).
 *
 *   a          E4M3  [M_sum, K]           tokens of all experts, concatenated
 *   sfa        int32 [Kp][al4(M_sum)]     packed scales of A
 *   b          E4M3  [G, N, K]            one weight matrix per expert
 *   sfb        int32 [G][Kp][al4(N)]      packed scales of every expert's B
 *   d          BF16  [M_sum, N]           output, fully overwritten
 *   m_indices  int32 [M_sum]              expert of every row, -1 on padding rows
 * Row m with e = m_indices[m] in [0, G) is  A[m] @ B[e]^T; rows with m_indices[m] == -1 are
 * written as +0.0.  Contract (device data, checked only in validation mode): every expert's
 * rows are contiguous and start at a multiple of 128
 * (dg_get_mk_alignment_for_contiguous_layout()); inside a 128-row block all rows that are not
 * -1 share one expert.  A block whose first row is -1 is written as zeros.  Entries >= G are
 * treated like -1.  Requires M_sum % 128 == 0 (M_sum == 0 is a no-op), G > 0, N and K as for
 * the dense call.
 */
dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, void* d, const int32_t* m_indices,
                                              int M_sum, int N, int K, int G, void* stream);

/*
 * M-grouped GEMM, masked layout (README "Grouped GEMM (masked layout)"; article section 5.1,
 * "masked grouping" for inference with CUDA graphs).
 *
 *   a         E4M3  [G, max_m, K]         group g's rows at a[g]
 *   sfa       int32 [G][Kp][al4(max_m)]   packed scales of A, per group
 *   b         E4M3  [G, N, K]
 *   sfb       int32 [G][Kp][al4(N)]
 *   d         BF16  [G, max_m, N]
 *   masked_m  int32 [G]                   valid rows of every group, read on the device
 * For every g, rows m < masked_m[g] of d[g] are A[g][m] @ B[g]^T; every other row of d is
 * left untouched.  Because the counts are read on the device, the call launches the same
 * work whatever they are and can be captured in a CUDA graph.  Contract (checked only in
 * validation mode): 0 <= masked_m[g] <= max_m; values outside are clamped to that range.
 * Requires G > 0 and G <= 4096, max_m >= 0 (0 is a no-op), N and K as for the dense call.
 */
dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b,
                                          const int32_t* sfb, void* d, const int32_t* masked_m,
                                          int G, int max_m, int N, int K, void* stream);

/*
 * FP8 x FP4: E4M3 activations times E2M1 weights, BF16 out (README "News" 2026.04.16: FP8xFP4
 * GEMM; the DeepGEMM-Ascend article's FP8xFP4 row: FP4 as the weight format halves its memory).
 * Same arguments, layouts, scales and semantics as dg_fp8_gemm_nt and the two M-grouped calls,
 * except that B holds E2M1 codes packed two per byte:
 *   b   uint8 [N][K/2] (dense) or [G][N][K/2] (grouped): K element 2i of a row in the low
 *       nibble of byte i, element 2i + 1 in the high nibble; E2M1 = sign, 2 exponent bits
 *       (bias 1), 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
 *   sfb packed UE8M0 words exactly as for the FP8 calls: one word per row of B and group of
 *       four 1x128 K blocks (per-row scales, or 128x128 block scales broadcast by
 *       dg_pack_sf_ue8m0 with gran_mn = 128)
 * b must be 32-byte aligned.  The weights cross HBM at half the FP8 bytes; in shared memory
 * and in the tensor cores they take the FP8 path's footprint and rate.
 */
dg_status dg_fp8_fp4_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, void* d, int M,
                             int N, int K, void* stream);
dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                                  const int32_t* sfb, void* d, const int32_t* m_indices, int M_sum,
                                                  int N, int K, int G, void* stream);
dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* masked_m, int G, int max_m, int N, int K,
                                              void* stream);

/* Storage layouts of the operands of dg_fp8_gemm (README "Interface / Notes": the SM100 kernels
 * take the NT, TN, NN and TT layouts).  The first letter is A's, the second B's:
 *   A 'n': [M, K], K contiguous        A 't': [K, M], M contiguous (MN-major)
 *   B 't': [N, K], K contiguous        B 'n': [K, N], N contiguous (MN-major)  */
enum { DG_LAYOUT_NT = 0, DG_LAYOUT_NN = 1, DG_LAYOUT_TN = 2, DG_LAYOUT_TT = 3 };

/*
 * D = C + A @ B^T in any of the four layouts, BF16 or FP32 out (README "Interface / Notes":
 * fp8_gemm_{nt, nn, tn, tt} compute D = C + A @ B.T).
 *
 *   a, b      E4M3, stored as `layout` says (see DG_LAYOUT_*)
 *   sfa, sfb  packed UE8M0 scales exactly as for dg_fp8_gemm_nt: word [kp][m] covers row m of
 *             D's rows and K blocks 4kp..4kp+3, word [kp][n] column n (the layout of the
 *             operands does not change the scales' layout)
 *   c         FP32 [M, N] or NULL; only with out_f32 = 1.  c may equal d (in-place
 *             accumulation): each element of C is read before the same element of D is written
 *   d         BF16 [M, N] (out_f32 = 0) or FP32 [M, N] (out_f32 = 1)
 * Requires what dg_fp8_gemm_nt requires, plus M % 16 == 0 when A is MN-major and N % 16 == 0
 * when B is MN-major (16-byte row pitch); c, when given, 16-byte aligned.
 * C is added to the FP32 accumulator before the final rounding.  layout = DG_LAYOUT_NT with
 * out_f32 = 0 and c = NULL is dg_fp8_gemm_nt.
 */
dg_status dg_fp8_gemm(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const float* c,
                      void* d, int M, int N, int K, int layout, int out_f32, void* stream);

/*
 * K-grouped GEMM of MoE weight gradients (README "News" 2025.05.14 and the API list:
 * k_grouped_fp8_gemm_tn_contiguous): for every group g,
 *     D[g] = C[g] + A_g^T B_g,   A_g = rows koff[g] .. koff[g] + ks[g] of A, same for B,
 * koff the exclusive prefix sum of ks.  Both operands are MN-major (the 't' A and 'n' B of
 * the TN layout): the groups are consecutive row ranges of the shared K (token) dimension.
 *
 *   a     e4m3  [sum_K][M]   M contiguous
 *   b     e4m3  [sum_K][N]   N contiguous
 *   sfa   int32 [sum_g ceil(ks[g]/512)][al4(M)]   per-group packed scales of A's 1x128 K blocks
 *   sfb   int32 [sum_g ceil(ks[g]/512)][al4(N)]   the same for B (dg_pack_sf_ue8m0_k_grouped)
 *   c     float [G][M][N] or NULL (may equal d)
 *   d     float [G][M][N]
 *   ks    int32 [G], device memory: K rows per group, each a multiple of 128, summing to sum_K
 *         (read on the device, so the call can be captured in a CUDA graph; checked only under
 *         DG_VALIDATE=1, which returns DG_ERR_CONTRACT)
 * A group with ks[g] = 0 gives D[g] = C[g] (zeros without C).  Requires G in 1..4096,
 * M % 16 == 0, N % 16 == 0, sum_K % 128 == 0, 16-byte aligned pointers.  Group sizes summing
 * past sum_K are clipped there (only rows of a and b below sum_K are read).
 */
dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              const float* c, float* d, const int32_t* ks, int G, int M, int N,
                                              int sum_K, void* stream);

/*
 * Per-group scale pack for the K-grouped GEMM (README API list:
 * get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor).
 *
 *   sf   float [sum_K / 128][MN]           one scale per 128-row K block and per column
 *   out  int32 [sum_g ceil(ks[g]/512)][al4(MN)]
 *   ks   int32 [G], device memory, as for dg_k_grouped_fp8_gemm_tn_contiguous
 * Group g's word row kpoff[g] + j, byte i holds the UE8M0 code (the rounding-up rule of
 * dg_pack_sf_ue8m0) of the scale of the group's K block 4j + i, 0 past its last block; no
 * word spans two groups.  Padding columns [MN, al4(MN)) are 0.  Requires sum_K % 128 == 0 and
 * sum_K / 512 + G <= 65535.
 */
dg_status dg_pack_sf_ue8m0_k_grouped(const float* sf, int32_t* out, const int32_t* ks, int G, int MN, int sum_K,
                                     void* stream);

/*
 * Scale-factor pack: FP32 scales -> MN-major, TMA-aligned, packed UE8M0
 * (README "Interface / Notes" and "Utilities": get_mn_major_tma_aligned_packed_ue8m0_tensor;
 * the DeepGEMM-Ascend article, "Cómo funciona", packs scales along K in MN-major order).
 *
 *   sf   float [G][ceil(MN/gran_mn)][Kb]     row-major, Kb = K / gran_k
 *   out  int32 [G][Kp][al4(MN)]              Kp = ceil(Kb/4); fully overwritten
 * Word [g][kp][r] byte j = UE8M0 code of sf[g][r / gran_mn][4*kp + j] (0 when 4*kp+j >= Kb);
 * words of the padding rows r in [MN, al4(MN)) are 0.  gran_mn is 1 (per-row 1x128 scales of
 * A) or 128 (128x128 block scales of B, broadcast to every row); gran_k must be 128.
 * UE8M0 code of a float x: the smallest b in 0..254 with 2^(b-127) >= x (a scale that is not
 * a power of two rounds up), 0xFE when x > 2^127, 0xFF when x is zero, negative, NaN or Inf.
 * Requires G > 0, MN >= 0 (0 is a no-op), K > 0 with K % 128 == 0.
 */
dg_status dg_pack_sf_ue8m0(const float* sf, int32_t* out, int G, int MN, int K, int gran_mn,
                           int gran_k, void* stream);

/*
 * Per-token 1x128 FP8 quantisation of BF16 activations, writing the packed scales directly
 * (README "Interface / Notes": FP8 quantisation of the inputs is left to the caller, to be
 * implemented separately or fused into the kernel that produces them).
 *
 *   x   bf16  [G][M][K]          row-major, finite values (a NaN or Inf gives unspecified codes)
 *   q   e4m3  [G][M][K]          row-major; fully overwritten
 *   sf  int32 [G][Kp][al4(M)]    packed UE8M0 scales in the A-operand layout of the GEMMs;
 *                                fully overwritten, padding rows [M, al4(M)) and bytes of
 *                                K blocks >= Kb are 0
 * For each row and 1x128 block: amax = max |x|; e = the smallest integer with
 * 448 * 2^e >= amax, clamped to [-127, 127], and 0 when amax = 0; the scale byte is e + 127
 * and the codes are round-to-nearest-even of x * 2^-e (|x * 2^-e| <= 448: no saturation).
 * G = 1 with M = M_sum quantises a contiguous-layout A; G groups of max_m rows a masked one.
 * Requires G > 0, M >= 0 (0 is a no-op), K > 0 with K % 128 == 0, 16-byte aligned pointers.
 * Asynchronous on `stream`; buffers are the caller's; nothing is allocated.
 */
dg_status dg_quantize_fp8_1x128(const void* x, void* q, int32_t* sf, int G, int M, int K, void* stream);

/* Row alignment of expert segments in the contiguous layout (the GEMM M block): 128.
 * (README "Grouped GEMM (contiguous layout)": get_mk_alignment_for_contiguous_layout.) */
int dg_get_mk_alignment_for_contiguous_layout(void);

/* mn rounded up so that mn elements of elem_bytes bytes span a multiple of 16 bytes;
 * -1 when elem_bytes is not 1, 2, 4, 8 or 16 or mn < 0.  (README "Utilities".) */
int dg_get_tma_aligned_size(int mn, int elem_bytes);

/* Caps the number of SMs the persistent kernels use (0 = all SMs).  Process-wide.
 * (README "Utilities": set_num_sms / get_num_sms.) */
void dg_set_num_sms(int n);
/* The SM count the next call on the current device will use. */
int dg_get_num_sms(void);

/* Programmatic dependent launch (README "Utilities": set_pdl).  When enabled (the default;
 * the environment variable DG_PDL=0 disables it), every kernel of this library is launched so
 * that its set-up (barrier initialisation, tensor-memory allocation) may overlap the end of the
 * previous kernel in the stream; each kernel waits for that kernel to complete before it reads
 * any global memory, so results never depend on the setting.  Process-wide. */
void dg_set_pdl(int enable);
int dg_get_pdl(void);

/* A static description of a status code. */
const char* dg_status_string(dg_status s);

/*
 * Reads and clears the device-side error word that the GEMM kernels set when a barrier wait
 * times out (about 4 s; it never happens in a correct run).  There is one word per device,
 * shared by every stream of the process on that device, so the call first waits for all work
 * on the current device (`stream` first, then the whole device): a timeout raised by a kernel
 * on another stream is reported too, to whichever caller checks first.  Returns
 * DG_ERR_TIMEOUT if any kernel on the device timed out since the last check, DG_ERR_CUDA if
 * the synchronization failed, DG_OK otherwise.  With DG_PRINT_CONFIGS=1 the word is printed
 * with the wait site that gave up (its bits 8..15).  Not part of the pages' API: a debugging
 * aid.
 */
dg_status dg_check_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
