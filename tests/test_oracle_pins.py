"""Pins for the CPU oracle: each check fixes a fact from the pages or from mathematics,
computed by a route that does not go through the oracle's own code.

Formats (DeepGEMM README, "Interface / Notes"): E4M3 operands, UE8M0 scale factors
packed four per int32, MN-major, TMA-aligned.  GEMM (same section): D = A @ B^T.
Grouped layouts: README "Grouped GEMM (contiguous layout)" / "(masked layout)".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import reference as R

# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------


def test_e4m3_spot_values():
    t = oracle.e4m3_decode_table()
    assert t[0x00] == 0.0 and not math.copysign(1, t[0x00]) < 0
    assert t[0x80] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert t[0x01] == 2.0 ** -9                       # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9                   # largest subnormal
    assert t[0x08] == 2.0 ** -6                       # smallest normal
    assert t[0x38] == 1.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0     # largest finite
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])


def test_e4m3_table_structure():
    t = oracle.e4m3_decode_table()
    finite = t[np.isfinite(t)]
    assert finite.size == 254                          # 256 codes minus two NaNs
    assert np.unique(finite).size == 253               # +0 and -0 are one value
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                    # codes 0x00..0x7E increase
    assert np.array_equal(t[0x80:0xFF], -t[:0x7F])     # sign bit negates


def test_e4m3_table_matches_torch_decoder():
    # torch's float8_e4m3fn decode is an independent implementation of the same format
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = oracle.e4m3_decode_table()
    both_nan = np.isnan(ref) & np.isnan(t)
    assert np.all(both_nan | (ref == t))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(t[~both_nan]))

# ---------------------------------------------------------------------------
# UE8M0
# ---------------------------------------------------------------------------


def test_ue8m0_decode():
    b = np.arange(256)
    v = oracle.ue8m0_decode(b)
    assert v[127] == 1.0 and v[0] == 2.0 ** -127 and v[254] == 2.0 ** 127
    assert math.isnan(v[255])
    for k in range(255):
        assert v[k] == Fraction(2) ** (k - 127)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
        ref = ref.to(torch.float64).numpy()
        assert np.array_equal(ref[:255], v[:255])


def _encode_by_search(x: float) -> int:
    """Brute force: walk all 255 finite codes, take the first whose value is >= x."""
    if not (x > 0) or math.isinf(x):
        return 0xFF
    xf = Fraction(x)
    for b in range(255):
        if Fraction(2) ** (b - 127) >= xf:
            return b
    return 0xFE


def test_ue8m0_encode_against_search():
    vals = []
    for k in range(-150, 131):
        p = np.float32(2.0 ** k) if -149 <= k <= 127 else None
        if p is None:
            continue
        vals += [p, np.nextafter(p, np.float32(np.inf)), np.nextafter(p, np.float32(0))]
    rs = np.random.default_rng(7)
    vals += list((rs.standard_normal(300) * 10.0 ** rs.integers(-30, 30, 300)).astype(np.float32))
    vals += [np.float32(0), np.float32(-0.0), np.float32(np.nan), np.float32(np.inf),
             np.float32(-np.inf), np.float32(3.4e38)]
    vals = np.array(vals, dtype=np.float32)
    got = oracle.ue8m0_encode(vals)
    want = np.array([_encode_by_search(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_ue8m0_roundtrip_on_powers():
    k = np.arange(-127, 128)
    x = np.ldexp(1.0, k).astype(np.float32)           # exact in float32 (subnormals incl.)
    codes = oracle.ue8m0_encode(x)
    assert np.array_equal(oracle.ue8m0_decode(codes), x.astype(np.float64))

# ---------------------------------------------------------------------------
# Pack
# ---------------------------------------------------------------------------


def _load_pack_cases(golden_dir):
    cases, cur = [], None
    with open(os.path.join(golden_dir, "pack_sf_ue8m0.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = dict(name=tok[1], G=int(tok[2]), MN=int(tok[3]), gran=int(tok[4]),
                           Kb=int(tok[5]), sf=[], words=[])
                cases.append(cur)
            elif tok[0] == "sf:":
                cur["sf"].append([float(v) for v in tok[1:]])
            elif tok[0] == "word":
                cur["words"].append((int(tok[1]), int(tok[2]), int(tok[3]), int(tok[4], 16)))
            elif tok[0] == "wordrange":
                g, kp, r0, r1, w = int(tok[1]), int(tok[2]), int(tok[3]), int(tok[4]), int(tok[5], 16)
                cur["words"] += [(g, kp, r, w) for r in range(r0, r1 + 1)]
    return cases


def test_pack_golden(golden_dir):
    cases = _load_pack_cases(golden_dir)
    assert {c["name"] for c in cases} == {"rows_a", "blocks_b", "rounding"}
    for c in cases:
        MNb = -(-c["MN"] // c["gran"])
        sf = np.array(c["sf"], dtype=np.float32).reshape(c["G"], MNb, c["Kb"])
        out = oracle.pack_sf_ue8m0(sf, c["MN"], c["gran"]).view(np.uint32)
        Kp = -(-c["Kb"] // 4)
        al = oracle.tma_aligned_size(c["MN"])
        assert out.shape == (c["G"], Kp, al), c["name"]
        seen = np.zeros(out.shape, dtype=bool)
        for g, kp, r, w in c["words"]:
            assert out[g, kp, r] == w, (c["name"], g, kp, r, hex(int(out[g, kp, r])), hex(w))
            seen[g, kp, r] = True
        assert seen.all(), c["name"]                   # the fixture lists every word


def test_tma_aligned_size():
    assert [oracle.tma_aligned_size(n) for n in (1, 4, 5, 130, 2112, 33152)] == [4, 4, 8, 132, 2112, 33152]
    assert oracle.tma_aligned_size(3, 1) == 16 and oracle.tma_aligned_size(9, 2) == 16


def test_pack_unpack_roundtrip_random():
    rs = np.random.default_rng(3)
    for G, MN, gran, Kb in [(1, 1, 1, 1), (2, 7, 1, 5), (3, 257, 128, 9), (1, 130, 1, 8)]:
        MNb = -(-MN // gran)
        e = rs.integers(-127, 128, size=(G, MNb, Kb))
        sf = np.ldexp(1.0, e).astype(np.float32)
        packed = oracle.pack_sf_ue8m0(sf, MN, gran)
        codes = oracle.unpack_sf_ue8m0(packed, MN, Kb)
        per_row = (e + 127)[:, np.arange(MN) // gran, :]
        assert np.array_equal(codes, per_row.astype(np.uint8))
        al = oracle.tma_aligned_size(MN)
        assert np.all(packed[:, :, MN:al] == 0)
        if Kb % 4:
            top = packed[:, -1, :MN].view(np.uint32) >> (8 * (Kb % 4))
            assert np.all(top == 0)

# ---------------------------------------------------------------------------
# BF16 rounding
# ---------------------------------------------------------------------------


def test_bf16_round_matches_torch_on_float32_inputs():
    # For float32-representable inputs, one RNE step from float64 equals torch's float32->bf16.
    rs = np.random.default_rng(11)
    x = (rs.standard_normal(20000) * 10.0 ** rs.integers(-40, 38, 20000)).astype(np.float32)
    # ties and near-ties: values with the low 16 bits set to 0x8000, 0x7FFF, 0x8001
    base = rs.integers(0, 2 ** 31, 3000, dtype=np.uint32) & 0x7F7F0000
    ties = np.concatenate([base | 0x8000, base | 0x18000, base | 0x7FFF, base | 0x8001]).view(np.float32)
    sub = np.array([1e-40, -3e-39, 1.2e-38, 9.2e-41], dtype=np.float32)
    x = np.concatenate([x, ties, -ties, sub])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_single_step_not_double():
    # 1 + 2**-8 is halfway between 1.0 and 1 + 2**-7: ties to even -> 1.0
    assert oracle.bf16_round_bits(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    # 1 + 3*2**-8 is halfway between 1 + 2**-7 (odd) and 1 + 2**-6 (even)
    assert oracle.bf16_round_bits(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above the tie: a float32 detour would lose the 2**-40 and round down
    assert oracle.bf16_round_bits(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert oracle.bf16_round_bits(np.array([-(1 + 2.0 ** -8 + 2.0 ** -40)]))[0] == 0xBF81
    # overflow and specials
    assert oracle.bf16_round_bits(np.array([2.0 ** 128]))[0] == 0x7F80
    assert oracle.bf16_round_bits(np.array([-(2.0 ** 129)]))[0] == 0xFF80
    big = (2 - 2.0 ** -8) * 2.0 ** 127                   # rounds up to 2**128 -> inf
    assert oracle.bf16_round_bits(np.array([big]))[0] == 0x7F80
    assert oracle.bf16_round_bits(np.array([0.0]))[0] == 0x0000
    assert oracle.bf16_round_bits(np.array([-0.0]))[0] == 0x8000
    assert oracle.bf16_round_bits(np.array([2.0 ** -133]))[0] == 0x0001   # smallest subnormal
    assert oracle.bf16_round_bits(np.array([2.0 ** -134]))[0] == 0x0000   # tie to even (0)
    assert oracle.bf16_round_bits(np.array([3 * 2.0 ** -134]))[0] == 0x0002


# ---------------------------------------------------------------------------
# GEMM: brute force in exact rational arithmetic
# ---------------------------------------------------------------------------

def _torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_exact(q: Fraction) -> int:
    """BF16 bits of an exact rational, round half to even, via integer arithmetic."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                                             # now 2**e <= a < 2**(e+1)
    qe = max(e, -126) - 7                                  # quantum exponent
    n = a / Fraction(2) ** qe
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = Fraction(fl) * Fraction(2) ** qe
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = int(np.array([float(v)], dtype=np.float32).view(np.uint32)[0] >> 16)
    return sign | bits


def _random_codes(rs, shape):
    c = rs.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38                           # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (3, 5, 256), (8, 8, 512), (2, 7, 384)])
def test_gemm_bruteforce_exact(M, N, K):
    rs = np.random.default_rng(M * 100 + N * 10 + K)
    Kb = K // 128
    a = _random_codes(rs, (M, K))
    b = _random_codes(rs, (N, K))
    ea = rs.integers(-20, 21, size=(M, Kb))
    eb = rs.integers(-20, 21, size=(N, Kb))
    sfa = oracle.pack_sf_ue8m0(np.ldexp(1.0, ea).astype(np.float32), M, 1)
    sfb = oracle.pack_sf_ue8m0(np.ldexp(1.0, eb).astype(np.float32), N, 1)
    got_f = oracle.fp8_gemm_nt_unrounded(a, sfa, b, sfb)
    got = oracle.fp8_gemm_nt(a, sfa, b, sfb)
    da, db = _torch_decode(a), _torch_decode(b)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            absum = Fraction(0)
            for k in range(K):
                kb = k // 128
                t = Fraction(da[m, k]) * Fraction(db[n, k]) * Fraction(2) ** int(ea[m, kb] + eb[n, kb])
                exact += t
                absum += abs(t)
            # float64 rounding happens only when the Kb block sums are added
            assert abs(Fraction(got_f[m, n]) - exact) <= absum * Kb * Fraction(2) ** -52
            assert got[m, n] == _bf16_exact(exact)


def test_gemm_bruteforce_single_block_exact():
    # With one K block the float64 result is exact, so it must equal the rational sum.
    rs = np.random.default_rng(5)
    a = _random_codes(rs, (4, 128))
    b = _random_codes(rs, (6, 128))
    sfa = oracle.pack_sf_ue8m0(np.full((4, 1), 2.0 ** -3, np.float32), 4, 1)
    sfb = oracle.pack_sf_ue8m0(np.full((1, 1), 2.0 ** 5, np.float32), 6, 128)
    got = oracle.fp8_gemm_nt_unrounded(a, sfa, b, sfb)
    da, db = _torch_decode(a), _torch_decode(b)
    for m in range(4):
        for n in range(6):
            exact = sum(Fraction(da[m, k]) * Fraction(db[n, k]) for k in range(128)) * 4
            assert Fraction(got[m, n]) == exact


# ---------------------------------------------------------------------------
# GEMM: identity, permutation, scale invariance, negation
# ---------------------------------------------------------------------------

def _unit_sf(rows, Kb, gran=1):
    return oracle.pack_sf_ue8m0(np.ones((-(-rows // gran), Kb), np.float32), rows, gran)


def test_gemm_identity_and_permutation():
    rs = np.random.default_rng(9)
    M, K = 6, 256
    a = _random_codes(rs, (M, K))
    ea = rs.integers(-10, 11, size=(M, 2))
    sfa = oracle.pack_sf_ue8m0(np.ldexp(1.0, ea).astype(np.float32), M, 1)
    deq = _torch_decode(a) * np.ldexp(1.0, np.repeat(ea, 128, axis=1))
    eye = np.zeros((K, K), np.uint8)
    eye[np.arange(K), np.arange(K)] = 0x38
    d = oracle.fp8_gemm_nt(a, sfa, eye, _unit_sf(K, 2, 128))
    want = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    val = oracle.bf16_bits_to_float
    # E4M3 * 2**e is exact in BF16 (compared as values: a -0 input sums with +0 products to +0)
    assert np.array_equal(val(d), val(want))
    perm = rs.permutation(K)
    P = np.zeros((K, K), np.uint8)
    P[np.arange(K), perm] = 0x38                       # row n of B selects column perm[n]
    dp = oracle.fp8_gemm_nt(a, sfa, P, _unit_sf(K, 2, 128))
    assert np.array_equal(val(dp), val(want[:, perm]))


def test_gemm_power_of_two_scale_invariance_and_negation():
    rs = np.random.default_rng(13)
    M, N, K = 16, 24, 512
    Kb = K // 128
    a = _random_codes(rs, (M, K))
    b = _random_codes(rs, (N, K))
    ea = rs.integers(-8, 9, size=(M, Kb))
    eb = rs.integers(-8, 9, size=(-(-N // 128), Kb))
    sf = lambda e, mn, g: oracle.pack_sf_ue8m0(np.ldexp(1.0, e).astype(np.float32), mn, g)
    base = oracle.fp8_gemm_nt_unrounded(a, sf(ea, M, 1), b, sf(eb, N, 128))
    d0 = oracle.bf16_round_bits(base)
    for k in (-5, 3, 17):
        dk = oracle.fp8_gemm_nt(a, sf(ea + k, M, 1), b, sf(eb, N, 128))
        assert np.array_equal(dk, oracle.bf16_round_bits(base * 2.0 ** k))
        dkb = oracle.fp8_gemm_nt(a, sf(ea, M, 1), b, sf(eb + k, N, 128))
        assert np.array_equal(dkb, dk)
    dk0 = oracle.fp8_gemm_nt(a, sf(ea + 4, M, 1), b, sf(eb - 4, N, 128))
    assert np.array_equal(dk0, d0)
    neg = oracle.fp8_gemm_nt(a ^ 0x80, sf(ea, M, 1), b, sf(eb, N, 128))
    assert np.array_equal(oracle.bf16_bits_to_float(neg), -oracle.bf16_bits_to_float(d0))


def test_gemm_k_block_scales_are_per_block():
    # Only K block 1 gets a large A scale: the result must change by exactly that block's share.
    rs = np.random.default_rng(17)
    a = _random_codes(rs, (3, 384))
    b = _random_codes(rs, (5, 384))
    e0 = np.zeros((3, 3), np.int64)
    e1 = e0.copy(); e1[:, 1] = 6
    sf = lambda e: oracle.pack_sf_ue8m0(np.ldexp(1.0, e).astype(np.float32), 3, 1)
    sfb = _unit_sf(5, 3, 128)
    d0 = oracle.fp8_gemm_nt_unrounded(a, sf(e0), b, sfb)
    d1 = oracle.fp8_gemm_nt_unrounded(a, sf(e1), b, sfb)
    blk1 = _torch_decode(a)[:, 128:256] @ _torch_decode(b)[:, 128:256].T
    assert np.allclose(d1 - d0, 63 * blk1, rtol=0, atol=1e-9 * np.abs(d1).max())


# ---------------------------------------------------------------------------
# Grouped layouts equal concatenated dense GEMMs
# ---------------------------------------------------------------------------

def _grouped_problem(rs, G, N, K, counts):
    from synth import contiguous_layout
    m_idx = contiguous_layout(counts)
    M_sum = m_idx.size
    Kb = K // 128
    a = _random_codes(rs, (M_sum, K))
    a[m_idx < 0] = 0x7F                                # NaN codes in padding rows
    b = _random_codes(rs, (G, N, K))
    ea = rs.integers(-6, 7, size=(M_sum, Kb))
    eb = rs.integers(-6, 7, size=(G, -(-N // 128), Kb))
    sfa = oracle.pack_sf_ue8m0(np.ldexp(1.0, ea).astype(np.float32), M_sum, 1)[0]
    sfb = oracle.pack_sf_ue8m0(np.ldexp(1.0, eb).astype(np.float32), N, 128)
    return m_idx, a, b, sfa, sfb, ea


def test_contiguous_equals_dense_per_expert():
    rs = np.random.default_rng(19)
    G, N, K = 3, 40, 256
    counts = [130, 0, 5]
    m_idx, a, b, sfa, sfb, ea = _grouped_problem(rs, G, N, K, counts)
    assert m_idx.size == 256 + 128
    d = oracle.m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_idx)
    assert np.all(d[m_idx < 0] == 0)                   # padding rows are +0.0
    for e in range(G):
        rows = np.nonzero(m_idx == e)[0]
        if rows.size == 0:
            continue
        sub_sfa = oracle.pack_sf_ue8m0(np.ldexp(1.0, ea[rows]).astype(np.float32), rows.size, 1)[0]
        dense = oracle.fp8_gemm_nt(a[rows], sub_sfa, b[e], sfb[e])
        assert np.array_equal(d[rows], dense)
    sample = np.array([0, 129, 256, 260])
    assert np.array_equal(oracle.m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_idx, rows=sample),
                          d[sample])


def test_contiguous_single_group_no_padding_equals_dense():
    rs = np.random.default_rng(23)
    m_idx, a, b, sfa, sfb, _ = _grouped_problem(rs, 1, 24, 384, [256])
    d = oracle.m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_idx)
    assert np.array_equal(d, oracle.fp8_gemm_nt(a, sfa, b[0], sfb[0]))


def test_masked_equals_dense_and_keeps_prior_rows():
    rs = np.random.default_rng(29)
    G, max_m, N, K = 3, 20, 16, 256
    a = _random_codes(rs, (G, max_m, K))
    b = _random_codes(rs, (G, N, K))
    ea = rs.integers(-6, 7, size=(G, max_m, 2))
    sfa = oracle.pack_sf_ue8m0(np.ldexp(1.0, ea).astype(np.float32), max_m, 1)
    sfb = oracle.pack_sf_ue8m0(np.ones((G, 1, 2), np.float32), N, 128)
    masked_m = np.array([0, 20, 7], np.int32)
    prior = np.full((G, max_m, N), 0x7FA5, np.uint16)
    d = oracle.m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, masked_m, prior)
    for g in range(G):
        m = masked_m[g]
        assert np.all(d[g, m:] == 0x7FA5)
        if m:
            dense = oracle.fp8_gemm_nt(a[g, :m], oracle.pack_sf_ue8m0(
                np.ldexp(1.0, ea[g, :m]).astype(np.float32), int(m), 1)[0], b[g], sfb[g])
            assert np.array_equal(d[g, :m], dense)


# ---------------------------------------------------------------------------
# Per-token quantisation
# ---------------------------------------------------------------------------

def test_e4m3_encode_matches_torch_cast_on_float32():
    # torch's float32 -> float8_e4m3fn cast is an independent RNE implementation
    rs = np.random.default_rng(21)
    v = (rs.uniform(-448, 448, 20000) * 2.0 ** rs.integers(-14, 1, 20000)).astype(np.float32)
    mids = (oracle.e4m3_decode_table()[:0x7E] + oracle.e4m3_decode_table()[1:0x7F]) / 2
    v = np.concatenate([v, mids.astype(np.float32), -mids.astype(np.float32),
                        np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -10])])
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_rne(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_block_scale_exponent_definition():
    amax = np.array([448.0, 448.0 * (1 + 2.0 ** -52), 448.0 * 2 ** -3, 1.0, 0.0, 2.0 ** -140, 3.0e38, 224.0, 225.0])
    e = oracle.block_scale_exponent(amax)
    for a, ei in zip(amax, e):
        if a == 0:
            assert ei == 0
            continue
        if -127 < ei < 127:
            assert 448.0 * 2.0 ** int(ei) >= a and 448.0 * 2.0 ** (int(ei) - 1) < a
    assert list(e[:4]) == [0, 1, -3, -8] and e[5] == -127 and e[7] == -1 and e[8] == 0


def test_quantize_round_trip_and_bounds():
    rs = np.random.default_rng(22)
    x = rs.standard_normal((5, 384)) * 10.0 ** rs.integers(-3, 4, (5, 1))
    x[2, 128:256] = 0.0                                      # an all-zero block
    codes, packed = oracle.quantize_fp8_1x128(x)
    e = oracle.unpack_sf_ue8m0(packed, 5, 3)[0].astype(np.int64) - 127
    deq = oracle.e4m3_decode(codes).reshape(5, 3, 128) * np.ldexp(1.0, e)[..., None]
    xb = x.reshape(5, 3, 128)
    err = np.abs(deq - xb)
    # within half an E4M3 ulp of the scaled value (3 mantissa bits, subnormal below 2**-6)
    scaled = np.abs(xb) / np.ldexp(1.0, e)[..., None]
    E = np.floor(np.log2(np.maximum(scaled, 2.0 ** -30)))
    half_ulp = np.ldexp(1.0, (np.maximum(E, -6) - 4).astype(np.int64)) * np.ldexp(1.0, e)[..., None]
    assert np.all(err <= half_ulp)
    assert e[2, 1] == 0 and np.all(codes[2, 128:256] == 0)
    amax_q = np.abs(oracle.e4m3_decode(codes)).reshape(5, 3, 128).max(-1)
    assert np.all((amax_q[e != 0] >= 224) & (amax_q[e != 0] <= 448))


def test_quantize_agrees_with_the_input_generator_on_bf16_activations():
    # The input generator quantises with frexp and torch's cast; the oracle with a search over
    # the E4M3 table and an exponent walk.  On BF16 inputs both must give the same bytes.
    import synth
    x = synth.make_activations(1, 6, 1280, seed=4, wide=True)[0]
    xf = oracle.bf16_bits_to_float(x)
    codes, packed = oracle.quantize_fp8_1x128(xf)
    s_codes, s_sf = synth.quantize_1x128(xf.astype(np.float32))
    assert np.array_equal(codes, s_codes)
    assert np.array_equal(packed, oracle.pack_sf_ue8m0(s_sf, 6, 1)[0])


# ---------------------------------------------------------------------------
# Layouts, FP32 accumulation, K-grouped GEMM: brute force on tiny inputs, from the FP32 scales
# (not the packed words) and with torch's E4M3 decode, one product at a time.
# ---------------------------------------------------------------------------

def _finite_codes(rs, shape):
    c = rs.integers(0, 256, size=shape).astype(np.uint8)
    return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)      # no NaN codes


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("layout", ["nt", "nn", "tn", "tt"])
def test_fp8_gemm_layouts_and_accumulation_brute_force(layout):
    rs = np.random.default_rng(31)
    M, N, K = 3, 5, 256
    a = _finite_codes(rs, (M, K))                      # logical A[m, k]
    b = _finite_codes(rs, (N, K))                      # logical B[n, k]
    sa = np.ldexp(np.float32(1), rs.integers(-6, 7, (M, 2))).astype(np.float32)
    sb = np.ldexp(np.float32(1), rs.integers(-6, 7, (N, 2))).astype(np.float32)
    c = rs.standard_normal((M, N)).astype(np.float32)
    a_st = a if layout[0] == "n" else np.ascontiguousarray(a.T)
    b_st = b if layout[1] == "t" else np.ascontiguousarray(b.T)
    got = oracle.fp8_gemm(a_st, oracle.pack_sf_ue8m0(sa, M, 1)[0], b_st, oracle.pack_sf_ue8m0(sb, N, 1)[0],
                          layout=layout, c=c, out="f32")
    av, bv = _dec(a), _dec(b)
    for m in range(M):
        for n in range(N):
            terms = [float(c[m, n])]
            for k in range(K):
                terms.append(av[m, k] * bv[n, k] * float(sa[m, k // 128]) * float(sb[n, k // 128]))
            assert got[m, n] == np.float32(math.fsum(terms)), (layout, m, n)


def test_k_grouped_pack_brute_force():
    rs = np.random.default_rng(32)
    ks = [128, 0, 640, 384, 512]
    mn = 6
    kb_total = sum(ks) // 128
    sf = np.ldexp(np.float32(1), rs.integers(-20, 21, (kb_total, mn))).astype(np.float32)
    packed = oracle.pack_sf_ue8m0_k_grouped(sf, mn, ks).view(np.uint32)
    assert packed.shape == (1 + 0 + 2 + 1 + 1, 8)
    row = 0
    blk = 0
    for kg in ks:
        nb = kg // 128
        for w in range((nb + 3) // 4):
            for r in range(8):
                for i in range(4):
                    byte = (int(packed[row + w, r]) >> (8 * i)) & 0xFF
                    j = 4 * w + i
                    if r >= mn or j >= nb:
                        assert byte == 0
                    else:
                        assert byte == math.frexp(float(sf[blk + j, r]))[1] - 1 + 127
        row += (nb + 3) // 4
        blk += nb


def test_k_grouped_gemm_brute_force():
    rs = np.random.default_rng(33)
    ks = [128, 0, 256]
    M, N = 3, 4
    Kt = sum(ks)
    a = _finite_codes(rs, (Kt, M))                     # MN-major: [K, M]
    b = _finite_codes(rs, (Kt, N))
    sa = np.ldexp(np.float32(1), rs.integers(-5, 6, (Kt // 128, M))).astype(np.float32)
    sb = np.ldexp(np.float32(1), rs.integers(-5, 6, (Kt // 128, N))).astype(np.float32)
    c = rs.standard_normal((len(ks), M, N)).astype(np.float32)
    got = oracle.k_grouped_fp8_gemm_tn_contiguous(a, oracle.pack_sf_ue8m0_k_grouped(sa, M, ks), b,
                                                  oracle.pack_sf_ue8m0_k_grouped(sb, N, ks), ks, c=c)
    av, bv = _dec(a), _dec(b)
    k0 = 0
    for g, kg in enumerate(ks):
        for m in range(M):
            for n in range(N):
                terms = [float(c[g, m, n])]
                for k in range(k0, k0 + kg):
                    terms.append(av[k, m] * bv[k, n] * float(sa[k // 128, m]) * float(sb[k // 128, n]))
                assert got[g, m, n] == np.float32(math.fsum(terms)), (g, m, n)
        k0 += kg
    no_c = oracle.k_grouped_fp8_gemm_tn_contiguous(a, oracle.pack_sf_ue8m0_k_grouped(sa, M, ks), b,
                                                   oracle.pack_sf_ue8m0_k_grouped(sb, N, ks), ks)
    assert np.all(no_c[1] == 0) and no_c[1].tobytes() == np.zeros((M, N), np.float32).tobytes()


# ---------------------------------------------------------------------------
# FP8 x FP4
# ---------------------------------------------------------------------------

def test_e2m1_table_is_the_format():
    # E2M1 (the 4-bit MX element format): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 the sign
    t = oracle.e2m1_decode_table()
    assert list(t[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(t[8:], -t[:8]) and np.signbit(t[8])
    # every value times 2 is an integer and the spacing doubles per binade
    assert np.all((t[:8] * 2) == np.round(t[:8] * 2))


def test_fp4_unpack_nibble_order():
    p = np.array([[0x21, 0xF0]], np.uint8)
    assert oracle.fp4_unpack(p).tolist() == [[1, 2, 0, 15]]


def test_fp8_fp4_gemm_brute_force():
    rs = np.random.default_rng(41)
    M, N, K = 3, 4, 256
    a = _finite_codes(rs, (M, K))
    b4 = rs.integers(0, 16, size=(N, K)).astype(np.uint8)
    packed = (b4[:, 0::2] | (b4[:, 1::2] << 4)).astype(np.uint8)
    sa = np.ldexp(np.float32(1), rs.integers(-6, 7, (M, 2))).astype(np.float32)
    sb = np.ldexp(np.float32(1), rs.integers(-6, 7, (N, 2))).astype(np.float32)
    got = oracle.fp8_fp4_gemm_nt_unrounded(a, oracle.pack_sf_ue8m0(sa, M, 1)[0], packed,
                                           oracle.pack_sf_ue8m0(sb, N, 1)[0])
    av = _dec(a)
    # E2M1 by its definition, one code at a time
    def e2m1(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        v = m * 0.5 if e == 0 else (1 + m * 0.5) * 2.0 ** (e - 1)
        return -v if s else v
    for m in range(M):
        for n in range(N):
            terms = [av[m, k] * e2m1(int(b4[n, k])) * float(sa[m, k // 128]) * float(sb[n, k // 128])
                     for k in range(K)]
            assert got[m, n] == math.fsum(terms)
