"""CPU oracle for the FP8 block-scaled GEMM family.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The library (the CUDA kernels behind the C ABI) never calls it,
and it shares no code with the library: no kernels, headers, tables, helpers or
constants.

What it computes is the plain definition of each operation, slow and in
float64, so that it can be checked against the pages by eye:

  * E4M3 decode (closed form of the 8-bit "fn" format) and UE8M0 decode
    (2**(b - 127)): the DeepGEMM README, "Interface / Notes", which names E4M3
    operands and UE8M0 scale factors (linking the PTX "alternate floating point
    data formats" section).
  * the scale-factor pack: four UE8M0 bytes per int32, MN-major, MN extent
    padded to 16 bytes (README "Interface / Notes": "4 UE8M0 packed into one
    torch.int", transposed, TMA-aligned; README "Utilities":
    get_mn_major_tma_aligned_packed_ue8m0_tensor, get_tma_aligned_size; the
    DeepGEMM-Ascend news article, "Cómo funciona", packs scale pairs along K in
    MN-major order).
  * D = A @ B^T with fine-grained scales (README "Interface / Notes": fp8_gemm_nt
    computes D = C + A @ B.T; the article's §四.2 gemm_fp8_fp8_bf16_nt takes lhs,
    rhs, lhs_scale, rhs_scale and returns BF16).
  * the M-grouped contiguous and masked layouts (README "Grouped GEMM
    (contiguous layout)" and "Grouped GEMM (masked layout)"; the article's §五.1
    layout table).
  * the NT/NN/TN/TT storage layouts and D = C + A @ B.T with FP32 C and D
    (README "Interface / Notes": SM100 supports all four layouts).
  * the K-grouped GEMM of MoE weight gradients and its per-group scale pack
    (README "News" 2025.05.14 and API list: k_grouped_fp8_gemm_tn_contiguous,
    get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor).
  * per-token 1x128 FP8 quantisation writing packed scales (README "Interface /
    Notes": quantisation is left to the caller, to be fused into a producer).
  * FP8 x FP4: E4M3 activations times E2M1 weights (README "News" 2026.04.16;
    the DeepGEMM-Ascend article's FP8xFP4 row and its note on FP4 weights).

Readings where the pages are silent (each listed in the design notes):
  P2  byte j of packed word kp holds K block 4*kp + j (little-endian).
  P3  B's 128x128 scales are broadcast to one packed word per row of B.
  P4  MN padded to a multiple of 4 int32 (16 bytes) with zero words.
  P5  a scale that is not a power of two rounds UP to the next one; below
      2**-127 gives byte 0x00, above 2**127 gives 0xFE; zero, negative, NaN or
      Inf gives 0xFF.  This convention is parity UNPINNED by the pages.
  P7  the exact sum is rounded once to BF16, round-to-nearest-even.
  P8  contiguous-layout padding rows (m_indices == -1) come out as +0.0.
  P9  masked-layout rows at or past masked_m[g] keep whatever D held before.
  P18 C is added to the exact product sum and the result rounded once (to FP32
      or BF16); the GPU adds C to its FP32 accumulator, one more rounding.
  P19 K-grouped scales: one FP32 scale per 128-row K block and per column of the
      MN-major operand ([sum Kb][MN]), packed per group so that no packed word
      spans two groups; every ks[g] is a multiple of 128.
  P20 FP4 weights: E2M1 codes packed two per byte, element 2i in the low nibble;
      their scales are the same packed UE8M0 1x128 words as FP8 B's (one per row
      and 128-wide K block) -- the pages fix neither the nibble order nor the
      FP4 scale granularity.
  P1  (per-token quantisation) the scale of a 1x128 block is 2**e with e the smallest integer
      such that 448 * 2**e >= amax, clamped to [-127, 127], 0 for an all-zero block.
"""
from .reference import (  # noqa: F401
    e4m3_decode_table, e4m3_decode, ue8m0_decode, ue8m0_encode, tma_aligned_size,
    pack_sf_ue8m0, unpack_sf_ue8m0, bf16_round_bits, bf16_bits_to_float,
    fp8_gemm_nt, fp8_gemm_nt_unrounded, m_grouped_fp8_gemm_nt_contiguous,
    m_grouped_fp8_gemm_nt_masked, e4m3_encode_rne, block_scale_exponent, quantize_fp8_1x128,
    f32_round, fp8_gemm, k_group_offsets, pack_sf_ue8m0_k_grouped, k_grouped_fp8_gemm_tn_contiguous,
    e2m1_decode_table, fp4_unpack, fp8_fp4_gemm_nt_unrounded, fp8_fp4_gemm_nt,
    m_grouped_fp8_fp4_gemm_nt_contiguous, m_grouped_fp8_fp4_gemm_nt_masked,
)
