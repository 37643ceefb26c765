"""The synthetic-input recipe's invariants, and planted mistakes that the oracle pins must catch.

The planted mistakes are made in the oracle, on the CPU, through monkeypatching; each
one is a plausible slip (a dropped term, a wrong sign, a transposed operand, a wrong
byte order, a wrong row broadcast) and at least one pin must fail under it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import reference as R
import tests.test_oracle_pins as pins


def _deq(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("shape", [(3, 256), (2, 5, 384)])
def test_quantize_1x128_invariants(shape):
    x = synth.normal(shape, 0, "a")
    synth.add_outliers(x, 0)
    q, sf = synth.quantize_1x128(x)
    assert q.dtype == np.uint8 and sf.shape == shape[:-1] + (shape[-1] // 128,)
    e = np.log2(sf.astype(np.float64))
    assert np.array_equal(e, np.round(e))                  # powers of two
    qd = _deq(q).reshape(*shape[:-1], -1, 128)
    amax_q = np.abs(qd).max(-1)
    # smallest exponent: the scaled amax is in (224, 448]; RNE can land it on the grid point 224
    assert np.all((amax_q >= 224) & (amax_q <= 448))
    xb = x.reshape(*shape[:-1], -1, 128).astype(np.float64)
    scaled = xb / sf[..., None]
    err = np.abs(qd - scaled)
    # half an E4M3 ulp of the scaled value: ulp = 2**(max(E,-6) - 3)
    E = np.floor(np.log2(np.maximum(np.abs(scaled), 2.0 ** -30)))
    ulp = np.ldexp(1.0, (np.maximum(E, -6) - 3).astype(np.int64))
    assert np.all(err <= ulp / 2)


def test_quantize_128x128_invariants_with_tail():
    x = synth.normal((200, 256), 1, "b", std=0.02)
    q, sf = synth.quantize_128x128(x)
    assert sf.shape == (2, 2)
    qd = _deq(q)
    for i in range(2):
        for kb in range(2):
            blk = qd[i * 128:(i + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.abs(blk).max()
            assert 224 <= amax <= 448
            xs = x[i * 128:(i + 1) * 128, kb * 128:(kb + 1) * 128] / sf[i, kb]
            assert np.all(np.abs(blk - xs) <= np.maximum(np.abs(xs) * 2.0 ** -4, 2.0 ** -10))


def test_quantize_exponent_boundaries():
    # amax exactly 448 * 2**e takes e; a hair above takes e + 1; zero block takes 0
    for e in (-10, 0, 3):
        x = np.zeros((1, 128), np.float32)
        x[0, 5] = 448.0 * 2.0 ** e
        _, sf = synth.quantize_1x128(x)
        assert sf[0, 0] == 2.0 ** e
        x[0, 5] = np.nextafter(np.float32(448.0 * 2.0 ** e), np.float32(np.inf))
        _, sf = synth.quantize_1x128(x)
        assert sf[0, 0] == 2.0 ** (e + 1)
    _, sf = synth.quantize_1x128(np.zeros((1, 128), np.float32))
    assert sf[0, 0] == 1.0


def test_contiguous_layout():
    m = synth.contiguous_layout([130, 0, 5, 128])
    assert m.size == 256 + 128 + 128
    assert np.all(m[:130] == 0) and np.all(m[130:256] == -1)
    assert np.all(m[256:261] == 2) and np.all(m[261:384] == -1)
    assert np.all(m[384:] == 3)


def test_workloads_are_seeded():
    a = synth.make_masked(2, 8, 16, 256, seed=4)
    b = synth.make_masked(2, 8, 16, 256, seed=4)
    assert np.array_equal(a["a"], b["a"]) and np.array_equal(a["masked_m"], b["masked_m"])
    c = synth.make_contiguous(3, 16, 128, 300, seed=2)
    assert c["m_indices"].size == c["M_sum"] and c["M_sum"] % 128 == 0
    assert np.all(c["a"][c["m_indices"] < 0] == synth.NAN_CODE)
    assert int(c["counts"].sum()) == 300


# ---------------------------------------------------------------------------
# Planted mistakes
# ---------------------------------------------------------------------------

def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_mutation_dropped_term(monkeypatch):
    orig = R._block_products

    def dropped(a, b, kb):
        a2 = a.copy()
        a2[:, kb * 128 + 127] = 0                          # last element of each block ignored
        return orig(a2, b, kb)
    monkeypatch.setattr(R, "_block_products", dropped)
    _fails(pins.test_gemm_bruteforce_exact, 3, 5, 256)


def test_mutation_dropped_k_block(monkeypatch):
    orig = R.fp8_gemm_nt_unrounded

    def short(a, sfa, b, sfb):
        return orig(a[:, :-128], sfa, b[:, :-128], sfb) if a.shape[1] > 128 else orig(a, sfa, b, sfb)
    monkeypatch.setattr(R, "fp8_gemm_nt_unrounded", short)
    _fails(pins.test_gemm_bruteforce_exact, 8, 8, 512)


def test_mutation_wrong_sign(monkeypatch):
    t = R._E4M3.copy()
    t[0xB8] = 1.0                                          # -1.0 decoded as +1.0
    monkeypatch.setattr(R, "_E4M3", t)
    monkeypatch.setattr(oracle, "e4m3_decode_table", lambda: t.copy())
    _fails(pins.test_e4m3_table_matches_torch_decoder)
    _fails(pins.test_gemm_bruteforce_exact, 8, 8, 512)


def test_mutation_transposed_operand(monkeypatch):
    def transposed(a_codes, b_codes, kb):
        # B read as [K, N] instead of [N, K] (shapes agree for the square B of the pin)
        ks = slice(kb * 128, (kb + 1) * 128)
        bt = np.ascontiguousarray(b_codes.T)
        return R.e4m3_decode(a_codes[:, ks]) @ R.e4m3_decode(bt[:, ks]).T
    monkeypatch.setattr(R, "_block_products", transposed)
    _fails(pins.test_gemm_identity_and_permutation)


def test_mutation_pack_byte_order(monkeypatch, golden_dir):
    orig = R.ue8m0_encode

    def swapped_pack(sf, mn, gran_mn):
        out = orig_pack(sf, mn, gran_mn).view(np.uint32)
        return out.byteswap().view(np.int32)
    orig_pack = R.pack_sf_ue8m0
    monkeypatch.setattr(oracle, "pack_sf_ue8m0", swapped_pack)
    _fails(pins.test_pack_golden, golden_dir)
    assert R.ue8m0_encode is orig


def test_mutation_block_row_broadcast(monkeypatch, golden_dir):
    orig_pack = R.pack_sf_ue8m0

    def per_block_not_per_row(sf, mn, gran_mn):
        # wrong reading: one word per 128-row block instead of one per row
        return orig_pack(sf, -(-mn // gran_mn), 1) if gran_mn > 1 else orig_pack(sf, mn, gran_mn)
    monkeypatch.setattr(oracle, "pack_sf_ue8m0", per_block_not_per_row)
    _fails(pins.test_pack_golden, golden_dir)


def test_mutation_double_rounding(monkeypatch):
    def via_float32(x):
        x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
        return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    monkeypatch.setattr(oracle, "bf16_round_bits", via_float32)
    _fails(pins.test_bf16_round_single_step_not_double)


def test_mutation_padding_not_zeroed(monkeypatch):
    orig = R.m_grouped_fp8_gemm_nt_contiguous

    def leaky(a, sfa, b, sfb, m_idx, rows=None):
        out = orig(a, sfa, b, sfb, m_idx, rows)
        sel = np.arange(len(m_idx)) if rows is None else np.asarray(rows)
        out[np.asarray(m_idx)[sel] < 0] = 0x7FC0           # NaN leaks from padding rows
        return out
    monkeypatch.setattr(oracle, "m_grouped_fp8_gemm_nt_contiguous", leaky)
    _fails(pins.test_contiguous_equals_dense_per_expert)


# ---------------------------------------------------------------------------
# Planted mistakes in the layout, K-grouped, FP8 x FP4 and quantisation parts of the oracle
# ---------------------------------------------------------------------------

def _fails_any(fn, *args):
    """A pin catches the mistake by failing an assertion or by refusing the data outright."""
    with pytest.raises((AssertionError, ValueError, IndexError)):
        fn(*args)


def test_mutation_layout_transpose_dropped(monkeypatch):
    monkeypatch.setattr(R, "_k_major", lambda codes, stored_mn_major: np.asarray(codes, dtype=np.uint8))
    _fails_any(pins.test_fp8_gemm_layouts_and_accumulation_brute_force, "tn")
    _fails_any(pins.test_fp8_gemm_layouts_and_accumulation_brute_force, "nn")


def test_mutation_c_subtracted(monkeypatch):
    orig = R.fp8_gemm

    def minus_c(a, sfa, b, sfb, layout="nt", c=None, out="bf16"):
        return orig(a, sfa, b, sfb, layout, None if c is None else -np.asarray(c), out)
    monkeypatch.setattr(oracle, "fp8_gemm", minus_c)
    _fails(pins.test_fp8_gemm_layouts_and_accumulation_brute_force, "nt")


def test_mutation_f32_out_rounded_to_bf16(monkeypatch):
    def via_bf16(x):
        return R.bf16_bits_to_float(R.bf16_round_bits(x)).astype(np.float32)
    monkeypatch.setattr(R, "f32_round", via_bf16)
    _fails(pins.test_fp8_gemm_layouts_and_accumulation_brute_force, "nt")
    _fails(pins.test_k_grouped_gemm_brute_force)


def test_mutation_k_group_offsets_inclusive(monkeypatch):
    orig = R.k_group_offsets

    def inclusive(ks):
        koff, kboff, kpoff = orig(ks)
        ks = np.asarray(ks, dtype=np.int64)
        return koff + ks, kboff, kpoff                     # groups start at their own end
    monkeypatch.setattr(R, "k_group_offsets", inclusive)
    _fails_any(pins.test_k_grouped_gemm_brute_force)


def test_mutation_k_grouped_pack_spans_groups(monkeypatch):
    def one_pack(sf, mn, ks):
        # wrong reading: the groups' K blocks packed as one run, words spanning group boundaries
        return R.pack_sf_ue8m0(np.asarray(sf, np.float32)[:, :mn].T[None], mn, 1)[0]
    monkeypatch.setattr(oracle, "pack_sf_ue8m0_k_grouped", one_pack)
    _fails_any(pins.test_k_grouped_pack_brute_force)


def test_mutation_e2m1_bias(monkeypatch):
    t = R._E2M1 * 2.0                                      # exponent bias 0 instead of 1
    monkeypatch.setattr(R, "_E2M1", t)
    monkeypatch.setattr(oracle, "e2m1_decode_table", lambda: t.copy())
    _fails(pins.test_e2m1_table_is_the_format)
    _fails(pins.test_fp8_fp4_gemm_brute_force)


def test_mutation_fp4_nibble_order(monkeypatch):
    def swapped(packed):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0xF
        return out
    monkeypatch.setattr(R, "fp4_unpack", swapped)
    monkeypatch.setattr(oracle, "fp4_unpack", swapped)
    _fails(pins.test_fp4_unpack_nibble_order)
    _fails(pins.test_fp8_fp4_gemm_brute_force)


def test_mutation_quantiser_ties_away(monkeypatch):
    orig = R.e4m3_encode_rne

    def ties_away(v):
        v = np.asarray(v, dtype=np.float64)
        # nudge every value a hair away from zero, which turns ties into round-half-away
        return orig(np.where(np.abs(v) < 448, v * (1 + 2.0 ** -40), v))
    monkeypatch.setattr(oracle, "e4m3_encode_rne", ties_away)
    _fails(pins.test_e4m3_encode_matches_torch_cast_on_float32)


def test_mutation_quantiser_exponent_boundary(monkeypatch):
    orig = R.block_scale_exponent

    def strict(amax):
        e = orig(amax)
        a = np.asarray(amax, dtype=np.float64)
        return np.where(np.ldexp(448.0, e) == a, e + 1, e)   # 448 * 2**e == amax wrongly bumped
    monkeypatch.setattr(oracle, "block_scale_exponent", strict)
    _fails(pins.test_block_scale_exponent_definition)
