"""Seeded synthetic inputs for the FP8 block-scaled GEMM family.

This module is shared by the tests, the benchmark and the smoke check. It holds
input generation only: random numbers, the test-side FP8 quantization recipe
and the MoE routing layouts. It holds none of the GEMM's arithmetic (no E4M3 or
UE8M0 decoding, no scale-factor packing, no products or sums), and it imports
neither the CUDA library nor the oracle.

Quantization is the caller's job in the DeepGEMM design ("Interface / Notes" of
the DeepGEMM README: FP8 casting is left to the user, to be fused into an
earlier kernel), so the recipe below is test scaffolding, not part of the
library. The recipe: one power-of-two scale per 1x128 block of an activation
row (A) and per 128x128 block of a weight matrix (B); the scale is 2**e with e
the smallest integer such that 448 * 2**e >= amax of the block (448 is the
largest finite E4M3 value), e clamped to [-127, 127] and e = 0 for an all-zero
block; the block divided by its scale is rounded to E4M3 with
round-to-nearest-even by torch's float8_e4m3fn cast.

Workload recipes (shapes from the DeepGEMM article's H800 tables and the MoE
layout section of the README):
  dense        A, B ~ N(0, 1)
  decode       A ~ N(0, 1) with 1 % of elements (uniform, without replacement)
               multiplied by 20; B ~ N(0, 0.02**2)
  prefill      A ~ N(0, 1), B ~ N(0, 0.02**2)
  contiguous   per-expert token counts ~ Multinomial(T, uniform over G);
               each expert segment padded to a multiple of 128 rows; padding
               rows of A hold the E4M3 NaN code 0x7F (they must not leak into
               the result) and m_indices = -1 there
  masked       masked_m[g] ~ U{1..max_m}
Every tensor draws from its own PCG64 stream, derived from (seed, stream id).
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0
BLOCK = 128          # scale-factor granularity along K, and along N for B
NAN_CODE = 0x7F      # E4M3 NaN bit pattern, used to poison padding rows

# Stream ids, one per tensor role, so that changing one tensor's shape does not
# shift the random numbers of another.
_STREAM = {"a": 1, "b": 2, "outlier": 3, "counts": 4, "masked_m": 5, "perm": 6,
           "d_fill": 7, "sf": 8, "act": 9}


def rng(seed: int, role: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM[role], sub])))


def normal(shape, seed: int, role: str, std: float = 1.0, sub: int = 0) -> np.ndarray:
    x = rng(seed, role, sub).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def add_outliers(x: np.ndarray, seed: int, frac: float = 0.01, factor: float = 20.0, sub: int = 0) -> np.ndarray:
    """Multiply `frac` of the elements (uniform, without replacement) by `factor`."""
    flat = x.reshape(-1)
    n = int(round(frac * flat.size))
    if n:
        idx = rng(seed, "outlier", sub).choice(flat.size, size=n, replace=False)
        flat[idx] *= np.float32(factor)
    return x


def _scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with 448 * 2**e >= amax, clamped to [-127, 127]; 0 where amax == 0.

    Computed without dividing by 448.  With amax = f * 2**fe (f in [0.5, 1)) and
    448 = 0.875 * 2**9:  448 * 2**(fe-9) = 0.875 * 2**fe >= amax  iff  f <= 0.875,
    while 448 * 2**(fe-10) < 0.5 * 2**fe <= amax always.  So e = fe - 9, plus one
    when f > 0.875.  Both comparisons are exact.
    """
    a = amax.astype(np.float64)
    f, fe = np.frexp(a)
    e = fe.astype(np.int64) - 9 + (f > 0.875)
    e = np.clip(e, -127, 127)
    e = np.where(a == 0, 0, e)
    return e.astype(np.int64)


def _to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round float32 values (already within +-448) to E4M3 codes, RNE, via torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def quantize_1x128(x: np.ndarray):
    """Per-row 1x128 block quantization of x[..., R, K] (K % 128 == 0).

    Returns (codes uint8 [..., R, K], sf float32 [..., R, K/128]) with sf exact powers of two.
    """
    *lead, R, K = x.shape
    assert K % BLOCK == 0
    xb = x.reshape(*lead, R, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=-1)
    e = _scale_exponent(amax)
    scaled = (xb * np.ldexp(np.float32(1.0), -e)[..., None].astype(np.float32)).astype(np.float32)
    q = _to_e4m3_codes(scaled.reshape(*lead, R, K))
    sf = np.ldexp(np.float32(1.0), e).astype(np.float32)
    return q, sf


def quantize_128x128(x: np.ndarray):
    """128x128 block quantization of x[..., N, K] (K % 128 == 0; the last row block may be short).

    Returns (codes uint8 [..., N, K], sf float32 [..., ceil(N/128), K/128]).
    """
    *lead, N, K = x.shape
    assert K % BLOCK == 0
    Nb = -(-N // BLOCK)
    pad = Nb * BLOCK - N
    xp = np.pad(x, [(0, 0)] * len(lead) + [(0, pad), (0, 0)]) if pad else x
    xb = xp.reshape(*lead, Nb, BLOCK, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=(-3, -1))                     # [..., Nb, Kb]
    e = _scale_exponent(amax)
    mult = np.ldexp(np.float32(1.0), -e).astype(np.float32)  # [..., Nb, Kb]
    scaled = (xb * mult[..., :, None, :, None]).astype(np.float32)
    q = _to_e4m3_codes(scaled.reshape(*lead, Nb * BLOCK, K))
    if pad:
        q = np.ascontiguousarray(q[..., :N, :])
    sf = np.ldexp(np.float32(1.0), e).astype(np.float32)
    return q, sf


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

def make_dense(M: int, N: int, K: int, seed: int = 0, a_outliers: bool = False, b_std: float = 1.0) -> dict:
    a = normal((M, K), seed, "a")
    if a_outliers:
        add_outliers(a, seed)
    b = normal((N, K), seed, "b", std=b_std)
    a_q, a_sf = quantize_1x128(a)
    b_q, b_sf = quantize_128x128(b)
    return dict(kind="dense", M=M, N=N, K=K, a=a_q, sfa=a_sf, b=b_q, sfb=b_sf)


def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def contiguous_layout(counts) -> np.ndarray:
    """m_indices for per-expert token counts: each expert's rows contiguous, starting at a
    multiple of 128, valid rows first and -1 up to the next multiple of 128; experts with
    zero tokens have no rows."""
    parts = []
    for e, c in enumerate(counts):
        c = int(c)
        if c == 0:
            continue
        seg = np.full(align_up(c, BLOCK), -1, dtype=np.int32)
        seg[:c] = e
        parts.append(seg)
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int32)


def make_contiguous(G: int, N: int, K: int, tokens: int, seed: int = 0, counts=None,
                    b_std: float = 0.02, a_outliers: bool = False) -> dict:
    if counts is None:
        counts = rng(seed, "counts").multinomial(tokens, [1.0 / G] * G)
    counts = np.asarray(counts, dtype=np.int64)
    m_indices = contiguous_layout(counts)
    M_sum = int(m_indices.size)
    a = normal((M_sum, K), seed, "a")
    if a_outliers:
        add_outliers(a, seed)
    valid = m_indices >= 0
    a[~valid] = 0.0
    a_q, a_sf = quantize_1x128(a)
    a_q[~valid] = NAN_CODE
    b = normal((G, N, K), seed, "b", std=b_std)
    b_q, b_sf = quantize_128x128(b)
    return dict(kind="contiguous", G=G, M_sum=M_sum, N=N, K=K, counts=counts, m_indices=m_indices,
                a=a_q, sfa=a_sf, b=b_q, sfb=b_sf)


def make_masked(G: int, max_m: int, N: int, K: int, seed: int = 0, masked_m=None,
                b_std: float = 0.02) -> dict:
    if masked_m is None:
        masked_m = rng(seed, "masked_m").integers(1, max_m + 1, size=G)
    masked_m = np.asarray(masked_m, dtype=np.int32)
    a = normal((G, max_m, K), seed, "a")
    b = normal((G, N, K), seed, "b", std=b_std)
    a_q, a_sf = quantize_1x128(a)
    b_q, b_sf = quantize_128x128(b)
    return dict(kind="masked", G=G, max_m=max_m, N=N, K=K, masked_m=masked_m,
                a=a_q, sfa=a_sf, b=b_q, sfb=b_sf)


def make_k_grouped(M: int, N: int, ks, seed: int = 0, a_outliers: bool = True) -> dict:
    """Inputs of the K-grouped (weight-gradient) GEMM: a [sum K, M] and b [sum K, N], both
    MN-major, N(0,1) (a with 1% outliers x20), quantized per group in blocks of 128 K rows by
    1 column: sfa [sum K / 128, M], sfb [sum K / 128, N] (FP32 powers of two)."""
    ks = np.asarray(ks, dtype=np.int64)
    assert np.all(ks % BLOCK == 0)
    K = int(ks.sum())
    a = normal((K, M), seed, "a")
    if a_outliers:
        add_outliers(a, seed)
    b = normal((K, N), seed, "b")
    # each K block of 128 rows lies inside one group (ks are multiples of 128), so quantising
    # the transposed operands in 1x128 blocks along K is the per-group quantisation
    a_q, a_sf = quantize_1x128(np.ascontiguousarray(a.T))
    b_q, b_sf = quantize_1x128(np.ascontiguousarray(b.T))
    return dict(kind="k_grouped", G=int(ks.size), M=M, N=N, K=K, ks=ks.astype(np.int32),
                a=np.ascontiguousarray(a_q.T), sfa=np.ascontiguousarray(a_sf.T),
                b=np.ascontiguousarray(b_q.T), sfb=np.ascontiguousarray(b_sf.T))


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def quantize_fp4_1x128(x: np.ndarray):
    """Per-row 1x128 block quantisation of x[..., R, K] to E2M1, packed two per byte (element
    2i in the low nibble).  Scale 2**e with e the smallest integer such that 6 * 2**e >= amax
    (0 for an all-zero block); codes round x / 2**e to the nearest E2M1 value, ties to the
    code with an even mantissa bit.  Returns (packed uint8 [..., R, K/2], sf float32 [..., R, K/128])."""
    *lead, R, K = x.shape
    xb = np.asarray(x, dtype=np.float64).reshape(*lead, R, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=-1)
    f, fe = np.frexp(amax)                      # amax = f * 2**fe, f in [0.5, 1)
    e = fe.astype(np.int64) - 3 + (f > 0.75)    # 6 * 2**(fe-3) = 0.75 * 2**fe
    e = np.where(amax == 0, 0, np.clip(e, -127, 127))
    y = np.abs(xb) / np.ldexp(1.0, e)[..., None]
    hi = np.minimum(np.searchsorted(_E2M1_GRID, y, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    d_hi, d_lo = _E2M1_GRID[hi] - y, y - _E2M1_GRID[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)) | (d_hi == 0)
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(xb) & (code > 0), code | 8, code).reshape(*lead, R, K).astype(np.uint8)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, np.ldexp(np.float32(1.0), e).astype(np.float32)


def with_fp4_b(w: dict, seed: int, b_std: float = 0.02) -> dict:
    """The same workload with FP4 weights: B [..., N, K] redrawn (same stream) and quantized
    to E2M1 with per-row 1x128 scales (sfb [..., N, K/128]); b_fp4 holds the packed bytes."""
    shape = w["b"].shape
    b = normal(shape, seed, "b", std=b_std)
    packed, sf = quantize_fp4_1x128(b)
    return dict(w, b_fp4=packed, sfb_fp4=sf)


SENTINEL_BF16 = 0x7FA5   # a NaN pattern used to pre-fill D where rows must stay untouched


# The five workloads, by name.  Sizes from the DeepGEMM article's H800 tables.
def make_activations(G: int, M: int, K: int, seed: int = 0, wide: bool = False) -> np.ndarray:
    """BF16 activations [G, M, K] as uint16 bit patterns: N(0,1) with 1% outliers x20.

    wide=True stresses the scale range: every row gets its own magnitude 2**U{-120..110},
    every fifth 1x128 block is zero, and some rows hold BF16 subnormals and values two
    hundred binades below their block's maximum.
    """
    x = add_outliers(normal((G, M, K), seed, "act"), seed, sub=9)
    if wide:
        r = rng(seed, "act", 1)
        x *= np.ldexp(np.float32(1.0), r.integers(-120, 111, size=(G, M, 1)))
        xb = x.reshape(G, M, K // BLOCK, BLOCK)
        xb[:, :, ::5, :] = 0.0
        if M > 2:
            x[:, 1, :] = np.ldexp(np.float32(1.0), -130) * r.integers(-7, 8, size=(G, K))   # subnormals
            x[:, 2, :] = np.ldexp(normal((G, K), seed, "act", sub=2), r.integers(-126, 101, size=(G, K)))
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


DECODE_SHAPES = [(64, 2112, 7168), (128, 24576, 1536), (128, 7168, 2048), (64, 4096, 7168)]
PREFILL_SHAPE = (4096, 7168, 16384)
CONTIGUOUS = dict(G=4, N=4096, K=7168, tokens=32768)
MASKED = dict(G=4, max_m=256, N=7168, K=2048)
SMALL_DENSE = (128, 512, 1024)
