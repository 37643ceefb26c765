"""Plain float64 definitions of the FP8 block-scaled GEMM family (test infrastructure).

See the package docstring for the passages each function follows and for the
readings taken where the pages are silent.  Nothing here is tuned: every
function is the definition written out, with numpy's matmul as the one library
step (used only where the result is exact, see `_block_products`).
"""
from __future__ import annotations

import math

import numpy as np

BLOCK_K = 128        # scale granularity along K (1x128 for A, 128x128 for B)


# ---------------------------------------------------------------------------
# Formats (README "Interface / Notes": E4M3 operands, UE8M0 scale factors)
# ---------------------------------------------------------------------------

def _e4m3_value(code: int) -> float:
    """The 8-bit E4M3 ("fn") value of one code: sign, 4 exponent bits (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal, (m/8) * 2**-6.  Exponent field 15 with mantissa 7 is NaN
    (the format has no infinity); all other codes are normal, (1 + m/8) * 2**(e - 7).
    """
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e4m3_decode_table() -> np.ndarray:
    """float64[256]: the value of every E4M3 code."""
    return np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


_E4M3 = e4m3_decode_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def ue8m0_decode(b) -> np.ndarray:
    """UE8M0 byte -> 2**(b - 127); 0xFF is NaN."""
    b = np.asarray(b, dtype=np.int64)
    out = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, out)


def ue8m0_encode(x) -> np.ndarray:
    """Float scales -> UE8M0 bytes (reading P5), elementwise.

    The byte is the smallest b in 0..254 with 2**(b - 127) >= x, or 0xFE when x > 2**127.
    Zero, negative, NaN and infinite x give 0xFF.  With x = f * 2**fe (f in [0.5, 1)):
    x is the power 2**(fe - 1) when f == 0.5, otherwise the next power up is 2**fe.
    """
    x = np.asarray(x, dtype=np.float64)
    bad = ~(x > 0.0) | np.isinf(x)
    f, fe = np.frexp(np.where(bad, 1.0, x))
    b = fe.astype(np.int64) + 127 - (f == 0.5)
    b = np.clip(b, 0, 0xFE)
    return np.where(bad, 0xFF, b).astype(np.uint8)


def tma_aligned_size(mn: int, elem_bytes: int = 4) -> int:
    """MN rounded up so that one MN-major row of the scale tensor spans a multiple of 16 bytes
    (README "Utilities": get_tma_aligned_size)."""
    per = 16 // elem_bytes
    return (mn + per - 1) // per * per


# ---------------------------------------------------------------------------
# Scale-factor pack (README "Interface / Notes" and "Utilities"; Ascend article, "Cómo funciona")
# ---------------------------------------------------------------------------

def pack_sf_ue8m0(sf: np.ndarray, mn: int, gran_mn: int) -> np.ndarray:
    """float sf[G][ceil(mn/gran_mn)][Kb] -> int32 [G][ceil(Kb/4)][tma_aligned_size(mn)].

    Word [g][kp][r] holds, in byte j (bits 8j..8j+7), the UE8M0 code of the scale covering
    row r and K block 4*kp + j: sf[g][r // gran_mn][4*kp + j].  Bytes for K blocks past Kb,
    and whole words for rows r >= mn, are zero.
    """
    sf = np.asarray(sf, dtype=np.float32)
    if sf.ndim == 2:
        sf = sf[None]
    G, MNb, Kb = sf.shape
    assert MNb == (mn + gran_mn - 1) // gran_mn
    Kp = (Kb + 3) // 4
    codes = ue8m0_encode(sf)                                  # [G, MNb, Kb]
    per_row = codes[:, np.arange(mn) // gran_mn, :]           # [G, mn, Kb]: scale of row r
    padded = np.zeros((G, mn, 4 * Kp), dtype=np.uint32)       # K blocks past Kb stay 0
    padded[:, :, :Kb] = per_row
    bytes4 = padded.reshape(G, mn, Kp, 4)
    words = (bytes4[..., 0] | (bytes4[..., 1] << 8) | (bytes4[..., 2] << 16)
             | (bytes4[..., 3] << 24))                        # [G, mn, Kp]
    out = np.zeros((G, Kp, tma_aligned_size(mn, 4)), dtype=np.uint32)
    out[:, :, :mn] = words.transpose(0, 2, 1)                 # MN-major; rows >= mn stay 0
    return out.view(np.int32)


def unpack_sf_ue8m0(packed: np.ndarray, mn: int, kb_count: int) -> np.ndarray:
    """int32 [G][Kp][al4(mn)] -> uint8 codes [G][mn][Kb]: the inverse view of the pack."""
    p = np.asarray(packed).view(np.uint32)
    if p.ndim == 2:
        p = p[None]
    G, Kp, _ = p.shape
    codes = np.zeros((G, mn, kb_count), dtype=np.uint8)
    for kb in range(kb_count):
        kp, j = divmod(kb, 4)
        codes[:, :, kb] = (p[:, kp, :mn] >> (8 * j)) & 0xFF
    return codes


# ---------------------------------------------------------------------------
# BF16 rounding (reading P7)
# ---------------------------------------------------------------------------

def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> BF16 bit patterns (uint16), one round-to-nearest-even step.

    BF16 has 8 significant bits and FP32's exponent range: normal binades 2**-126 ..
    2**127, subnormal spacing 2**-133.  The quantum of x is 2**(max(E, -126) - 7) with E
    the binade exponent of x; x / quantum is exact, np.rint rounds it half-to-even, and the
    product is exactly representable in BF16 (hence in float32, whose top 16 bits it is).
    Results of magnitude >= 2**128 are infinities.  NaN maps to 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    nan = np.isnan(x)
    _, fe = np.frexp(np.where(nan, 0.0, x))           # |x| in [2**(fe-1), 2**fe)
    E = fe.astype(np.int64) - 1
    q_exp = np.maximum(E, -126) - 7
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.rint(np.ldexp(np.where(nan, 0.0, x), -q_exp))
        y = np.ldexp(r, q_exp)
    inf = np.abs(y) >= 2.0 ** 128
    y32 = np.where(inf, 0.0, y).astype(np.float32)   # exact: y is a BF16 value
    bits = (y32.view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(inf, np.where(y > 0, 0x7F80, 0xFF80), bits).astype(np.uint16)
    bits = np.where(nan, 0x7FC0, bits).astype(np.uint16)
    out[...] = bits
    return out


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# GEMMs (README "Interface / Notes", "Grouped GEMM (contiguous / masked layout)")
# ---------------------------------------------------------------------------

def _block_products(a_codes: np.ndarray, b_codes: np.ndarray, kb: int) -> np.ndarray:
    """sum_{k in block kb} e4m3(A[m,k]) * e4m3(B[n,k]) for all m, n, exactly.

    Every E4M3 value is an integer multiple of 2**-9 below 2**9, so each product is a
    multiple of 2**-18 below 2**18 and a 128-term sum needs fewer than 43 bits: float64
    holds it exactly in any summation order, which is why a library matmul may be used.
    """
    ks = slice(kb * BLOCK_K, (kb + 1) * BLOCK_K)
    a = e4m3_decode(a_codes[:, ks])
    b = e4m3_decode(b_codes[:, ks])
    return a @ b.T


def fp8_gemm_nt_unrounded(a_codes, sfa_packed, b_codes, sfb_packed) -> np.ndarray:
    """float64 D[m, n] = sum_kb 2**(sa(m,kb)-127) * 2**(sb(n,kb)-127) * sum_{k in kb} a*b.

    a_codes uint8 [M, K], b_codes uint8 [N, K]; sfa_packed int32 [Kp][al4(M)] and
    sfb_packed int32 [Kp][al4(N)] are packed UE8M0 words (one per row).  The K blocks are
    added in ascending order; each block's sum is exact (see `_block_products`).
    """
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    b_codes = np.asarray(b_codes, dtype=np.uint8)
    M, K = a_codes.shape
    N = b_codes.shape[0]
    assert K % BLOCK_K == 0 and b_codes.shape[1] == K
    Kb = K // BLOCK_K
    sa = unpack_sf_ue8m0(sfa_packed, M, Kb)[0]        # [M, Kb] codes
    sb = unpack_sf_ue8m0(sfb_packed, N, Kb)[0]        # [N, Kb]
    d = np.zeros((M, N), dtype=np.float64)
    for kb in range(Kb):
        scale = ue8m0_decode(sa[:, kb])[:, None] * ue8m0_decode(sb[:, kb])[None, :]
        d += scale * _block_products(a_codes, b_codes, kb)
    return d


def fp8_gemm_nt(a_codes, sfa_packed, b_codes, sfb_packed) -> np.ndarray:
    """BF16 bits [M, N] of D = A @ B^T (dense; the definition above, rounded once)."""
    return bf16_round_bits(fp8_gemm_nt_unrounded(a_codes, sfa_packed, b_codes, sfb_packed))


def m_grouped_fp8_gemm_nt_contiguous(a_codes, sfa_packed, b_codes, sfb_packed, m_indices,
                                     rows=None) -> np.ndarray:
    """BF16 bits [M_sum, N] of the contiguous-layout grouped GEMM.

    Row m with e = m_indices[m] >= 0 is the dense row A[m] @ B[e]^T with A's scales and
    expert e's scales; rows with m_indices[m] == -1 are +0.0 (reading P8).
    a_codes [M_sum, K]; sfa_packed [Kp][al4(M_sum)]; b_codes [G, N, K];
    sfb_packed [G][Kp][al4(N)].  `rows` restricts the computation to a subset of rows
    (the result then has len(rows) rows, in that order).
    """
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    m_indices = np.asarray(m_indices, dtype=np.int64)
    M_sum, K = a_codes.shape
    G, N, _ = b_codes.shape
    Kb = K // BLOCK_K
    rows = np.arange(M_sum) if rows is None else np.asarray(rows, dtype=np.int64)
    sa_all = unpack_sf_ue8m0(sfa_packed, M_sum, Kb)[0]
    out = np.zeros((rows.size, N), dtype=np.uint16)
    for e in range(G):
        sel = np.nonzero(m_indices[rows] == e)[0]
        if sel.size == 0:
            continue
        r = rows[sel]
        sub_sfa = _repack_rows(sa_all[r])
        out[sel] = fp8_gemm_nt(a_codes[r], sub_sfa, b_codes[e], sfb_packed[e])
    return out


def m_grouped_fp8_gemm_nt_masked(a_codes, sfa_packed, b_codes, sfb_packed, masked_m,
                                 d_prior) -> np.ndarray:
    """BF16 bits [G, max_m, N] of the masked-layout grouped GEMM.

    For every group g, rows m < masked_m[g] are the dense rows A[g][m] @ B[g]^T; all other
    rows keep the bits of d_prior (reading P9).
    """
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    G, max_m, K = a_codes.shape
    out = np.array(d_prior, dtype=np.uint16, copy=True)
    Kb = K // BLOCK_K
    for g in range(G):
        m = int(masked_m[g])
        if m <= 0:
            continue
        sa = unpack_sf_ue8m0(sfa_packed[g], max_m, Kb)[0][:m]
        out[g, :m] = fp8_gemm_nt(a_codes[g, :m], _repack_rows(sa), b_codes[g], sfb_packed[g])
    return out


def _repack_rows(codes_rows: np.ndarray) -> np.ndarray:
    """uint8 codes [R, Kb] -> packed int32 [Kp][al4(R)] (the pack layout, for a row subset)."""
    R, Kb = codes_rows.shape
    Kp = (Kb + 3) // 4
    out = np.zeros((Kp, tma_aligned_size(R, 4)), dtype=np.uint32)
    for kb in range(Kb):
        kp, j = divmod(kb, 4)
        out[kp, :R] |= codes_rows[:, kb].astype(np.uint32) << (8 * j)
    return out.view(np.int32)


# ---------------------------------------------------------------------------
# Per-token 1x128 quantisation (README "Interface / Notes": FP8 casting is the caller's job,
# to be fused into an earlier kernel; this is the operation such a kernel performs)
# ---------------------------------------------------------------------------

_POS_CODES = np.arange(0x7F)                 # codes 0x00..0x7E: the non-negative finite values
_POS_VALUES = _E4M3[:0x7F]                   # increasing


def e4m3_encode_rne(v: np.ndarray) -> np.ndarray:
    """float64 values with |v| <= 448 -> E4M3 codes, round to nearest, ties to the even code.

    The nearest of the 127 non-negative finite values is found by search; on a tie the code
    whose mantissa bit 0 is clear wins.  The sign bit is the sign of v (so -0.0 -> 0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    assert np.all(a <= 448.0), "values beyond the E4M3 range"
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    exact = d_hi == 0
    pick_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def block_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with 448 * 2**e >= amax, clamped to [-127, 127]; 0 when amax == 0.

    Found by walking e from the frexp exponent of amax (448 * 2**e is exact in float64).
    """
    a = np.asarray(amax, dtype=np.float64)
    _, fe = np.frexp(a)
    e = fe.astype(np.int64) - 10                               # 448 * 2**(fe-10) < 2**(fe-1) <= a
    for _ in range(3):                                         # at most two steps up
        e = np.where(np.ldexp(448.0, e) < a, e + 1, e)
    e = np.clip(e, -127, 127)
    return np.where(a == 0, 0, e).astype(np.int64)


def quantize_fp8_1x128(x: np.ndarray):
    """x [M, K] (any float dtype, finite) -> (E4M3 codes [M, K], packed UE8M0 int32 [Kp][al4(M)]).

    Per 1x128 block of a row: e = block_scale_exponent(amax), codes = RNE(x / 2**e).
    """
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    assert K % BLOCK_K == 0
    xb = x.reshape(M, K // BLOCK_K, BLOCK_K)
    e = block_scale_exponent(np.abs(xb).max(axis=-1))          # [M, Kb]
    scaled = xb / np.ldexp(1.0, e)[..., None]                  # exact: division by a power of two
    codes = e4m3_encode_rne(scaled).reshape(M, K)
    packed = pack_sf_ue8m0(np.ldexp(1.0, e).astype(np.float32), M, 1)[0]
    return codes, packed


# ---------------------------------------------------------------------------
# Memory layouts and FP32 accumulation (README "Interface / Notes": the SM100 kernels take
# the NT, TN, NN and TT layouts and compute D = C + A @ B.T)
# ---------------------------------------------------------------------------

def f32_round(x: np.ndarray) -> np.ndarray:
    """float64 -> float32, one round-to-nearest-even step (numpy's conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def _k_major(codes: np.ndarray, stored_mn_major: bool) -> np.ndarray:
    """An operand as [rows, K] codes: an MN-major operand is stored [K, rows]."""
    codes = np.asarray(codes, dtype=np.uint8)
    return np.ascontiguousarray(codes.T) if stored_mn_major else codes


def fp8_gemm(a_codes, sfa_packed, b_codes, sfb_packed, layout: str = "nt", c=None, out: str = "bf16"):
    """D = C + A @ B^T for the four storage layouts, rounded once to BF16 bits or FP32.

    layout[0] is A's letter: 'n' = stored [M, K] (K contiguous), 't' = stored [K, M].
    layout[1] is B's letter: 't' = stored [N, K] (K contiguous), 'n' = stored [K, N].
    The scale tensors do not depend on the layout: word [kp][r] of sfa covers row m = r of
    D's rows, of sfb row n = r.  c (optional) is FP32 [M, N], added exactly before rounding.
    """
    assert layout in ("nt", "nn", "tn", "tt") and out in ("bf16", "f32")
    a = _k_major(a_codes, layout[0] == "t")
    b = _k_major(b_codes, layout[1] == "n")
    d = fp8_gemm_nt_unrounded(a, sfa_packed, b, sfb_packed)
    if c is not None:
        d = d + np.asarray(c, dtype=np.float32).astype(np.float64)
    return bf16_round_bits(d) if out == "bf16" else f32_round(d)


# ---------------------------------------------------------------------------
# K-grouped GEMM for MoE weight gradients (README "News" 2025.05.14 and the API list:
# k_grouped_fp8_gemm_tn_contiguous, get_k_grouped_mn_major_tma_aligned_packed_ue8m0_tensor)
# ---------------------------------------------------------------------------

def k_group_offsets(ks):
    """Per group: first K row, first K block and first packed-word row (exclusive prefix sums
    of ks, ks / 128 and ceil(ks / 512)); each ks[g] is a multiple of 128."""
    ks = np.asarray(ks, dtype=np.int64)
    assert np.all(ks >= 0) and np.all(ks % BLOCK_K == 0)
    kb = ks // BLOCK_K
    kp = (kb + 3) // 4
    excl = lambda v: np.concatenate([[0], np.cumsum(v)[:-1]]).astype(np.int64)
    return excl(ks), excl(kb), excl(kp)


def pack_sf_ue8m0_k_grouped(sf: np.ndarray, mn: int, ks) -> np.ndarray:
    """float sf [sum_g ks[g]/128][mn] (one scale per K block and row, MN contiguous) ->
    int32 [sum_g ceil(ks[g]/512)][al4(mn)].

    Each group is packed on its own: word row kpoff[g] + j, byte i holds the UE8M0 code of
    the scale of the group's K block 4j + i (0 past the group's last block); rows >= mn are 0.
    """
    sf = np.asarray(sf, dtype=np.float32)
    ks = np.asarray(ks, dtype=np.int64)
    _, kboff, _ = k_group_offsets(ks)
    parts = []
    for g in range(ks.size):
        kb_g = int(ks[g]) // BLOCK_K
        if kb_g == 0:
            continue
        per_row = sf[kboff[g]:kboff[g] + kb_g, :mn].T                 # [mn, Kb_g]
        parts.append(pack_sf_ue8m0(per_row[None], mn, 1)[0])
    if not parts:
        return np.zeros((0, tma_aligned_size(mn, 4)), dtype=np.int32)
    return np.concatenate(parts, axis=0)


def k_grouped_fp8_gemm_tn_contiguous(a_codes, sfa_packed, b_codes, sfb_packed, ks, c=None) -> np.ndarray:
    """FP32 [G, M, N]: D[g] = C[g] + sum over the K rows k of group g of A[k, :]^T B[k, :].

    a_codes [sum K, M] and b_codes [sum K, N] are MN-major (the 't' A and 'n' B layouts);
    group g owns K rows koff[g] .. koff[g] + ks[g].  sfa_packed [sum Kp_g][al4(M)] and
    sfb_packed [sum Kp_g][al4(N)] hold per-row scales of 1x128 K blocks, packed per group
    (`pack_sf_ue8m0_k_grouped`).  A group with ks[g] = 0 gives D[g] = C[g] (0 without C).
    """
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    b_codes = np.asarray(b_codes, dtype=np.uint8)
    ks = np.asarray(ks, dtype=np.int64)
    M, N = a_codes.shape[1], b_codes.shape[1]
    koff, _, kpoff = k_group_offsets(ks)
    out = np.zeros((ks.size, M, N), dtype=np.float32)
    for g in range(ks.size):
        d = np.zeros((M, N), dtype=np.float64)
        if ks[g] > 0:
            rows = slice(koff[g], koff[g] + ks[g])
            kp = (int(ks[g]) // BLOCK_K + 3) // 4
            words = slice(kpoff[g], kpoff[g] + kp)
            d = fp8_gemm_nt_unrounded(a_codes[rows].T, sfa_packed[words], b_codes[rows].T, sfb_packed[words])
        if c is not None:
            d = d + np.asarray(c[g], dtype=np.float32).astype(np.float64)
        out[g] = f32_round(d)
    return out


# ---------------------------------------------------------------------------
# FP8 x FP4 (README "News" 2026.04.16: FP8xFP4 GEMM; the DeepGEMM-Ascend article: FP4 as the
# weight format, mixed with FP8 activations)
# ---------------------------------------------------------------------------

def _e2m1_value(code: int) -> float:
    """The 4-bit E2M1 value of one code: sign, 2 exponent bits (bias 1), 1 mantissa bit.

    Exponent field 0 is subnormal, (m/2) * 2**0; otherwise (1 + m/2) * 2**(e - 1).  Every
    code is finite: the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6.
    """
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    mag = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


_E2M1 = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_decode_table() -> np.ndarray:
    """float64[16]: the value of every E2M1 code."""
    return _E2M1.copy()


def fp4_unpack(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> E2M1 codes uint8 [..., K]: element 2i is the low nibble of byte i,
    element 2i + 1 the high nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def _fp4_block_products(a_codes, b_codes4, kb):
    """sum_{k in block kb} e4m3(A[m,k]) * e2m1(B[n,k]), exactly: the products are multiples of
    2**-10 below 2688, so 128-term sums need fewer than 32 bits and float64 holds them in any
    order."""
    ks = slice(kb * BLOCK_K, (kb + 1) * BLOCK_K)
    return e4m3_decode(a_codes[:, ks]) @ _E2M1[b_codes4[:, ks]].T


def fp8_fp4_gemm_nt_unrounded(a_codes, sfa_packed, b_packed, sfb_packed) -> np.ndarray:
    """float64 D = A @ B^T with A E4M3 [M, K] and B E2M1 packed two per byte [N, K/2]; scales as
    for fp8_gemm_nt_unrounded (packed UE8M0, one word per row, 1x128 K blocks)."""
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    b4 = fp4_unpack(b_packed)
    M, K = a_codes.shape
    N = b4.shape[0]
    assert K % BLOCK_K == 0 and b4.shape[1] == K
    Kb = K // BLOCK_K
    sa = unpack_sf_ue8m0(sfa_packed, M, Kb)[0]
    sb = unpack_sf_ue8m0(sfb_packed, N, Kb)[0]
    d = np.zeros((M, N), dtype=np.float64)
    for kb in range(Kb):
        scale = ue8m0_decode(sa[:, kb])[:, None] * ue8m0_decode(sb[:, kb])[None, :]
        d += scale * _fp4_block_products(a_codes, b4, kb)
    return d


def fp8_fp4_gemm_nt(a_codes, sfa_packed, b_packed, sfb_packed) -> np.ndarray:
    """BF16 bits [M, N] of D = A @ B^T, FP8 A and FP4 B, rounded once."""
    return bf16_round_bits(fp8_fp4_gemm_nt_unrounded(a_codes, sfa_packed, b_packed, sfb_packed))


def m_grouped_fp8_fp4_gemm_nt_contiguous(a_codes, sfa_packed, b_packed, sfb_packed, m_indices, rows=None):
    """The contiguous-layout grouped GEMM with FP4 experts b_packed [G, N, K/2]: row m with
    e = m_indices[m] >= 0 is A[m] @ B[e]^T, rows with -1 are +0.0."""
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    m_indices = np.asarray(m_indices, dtype=np.int64)
    M_sum, K = a_codes.shape
    G, N, _ = b_packed.shape
    Kb = K // BLOCK_K
    rows = np.arange(M_sum) if rows is None else np.asarray(rows, dtype=np.int64)
    sa_all = unpack_sf_ue8m0(sfa_packed, M_sum, Kb)[0]
    out = np.zeros((rows.size, N), dtype=np.uint16)
    for e in range(G):
        sel = np.nonzero(m_indices[rows] == e)[0]
        if sel.size:
            r = rows[sel]
            out[sel] = fp8_fp4_gemm_nt(a_codes[r], _repack_rows(sa_all[r]), b_packed[e], sfb_packed[e])
    return out


def m_grouped_fp8_fp4_gemm_nt_masked(a_codes, sfa_packed, b_packed, sfb_packed, masked_m, d_prior):
    """The masked-layout grouped GEMM with FP4 experts: rows m < masked_m[g] of group g are
    A[g][m] @ B[g]^T, every other row keeps d_prior's bits."""
    a_codes = np.asarray(a_codes, dtype=np.uint8)
    G, max_m, K = a_codes.shape
    out = np.array(d_prior, dtype=np.uint16, copy=True)
    Kb = K // BLOCK_K
    for g in range(G):
        m = int(masked_m[g])
        if m > 0:
            sa = unpack_sf_ue8m0(sfa_packed[g], max_m, Kb)[0][:m]
            out[g, :m] = fp8_fp4_gemm_nt(a_codes[g, :m], _repack_rows(sa), b_packed[g], sfb_packed[g])
    return out
