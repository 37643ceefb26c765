"""GPU GEMM parity against the oracle, element by element, through the C ABI.

Floating-point results: within the stated tolerance (tests/_parity.py).  Padding rows of the
contiguous layout: bit-exact +0.0.  Rows the masked layout must not touch: bit-exact
sentinel.  Power-of-two scale changes and negation: bit-exact on the GPU too, since scaling
every product by 2**k and flipping signs commute exactly with FP32 accumulation and with
the final rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu

SENT = synth.SENTINEL_BF16


def _pack(sf, mn, gran):
    return oracle.pack_sf_ue8m0(sf, mn, gran)


def run_dense(w, sfa=None, sfb=None):
    M, N, K = w["M"], w["N"], w["K"]
    sfa = _pack(w["sfa"], M, 1)[0] if sfa is None else sfa
    sfb = _pack(w["sfb"], N, 128)[0] if sfb is None else sfb
    d = torch.full((M, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    return bits(d), sfa, sfb


@pytest.mark.parametrize("M,N,K", [
    (128, 512, 1024),     # the small dense workload
    (1, 256, 128),        # one row, one K block
    (64, 2112, 512),      # N tail of 64 (2112 = 16.5 * 128) and a half-empty M block
    (200, 96, 640),       # ragged M tail, Kb = 5 (a partly filled packed word)
    (384, 40, 256),       # N = 40: not a multiple of 32
    (129, 8, 384),        # the smallest N; one row in the second M block
    (256, 4096, 1024),    # many tiles per CTA
])
def test_dense_parity(M, N, K):
    w = synth.make_dense(M, N, K, seed=M + N + K)
    got, sfa, sfb = run_dense(w)
    want = oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb)
    assert_within_tolerance(got, want, f"dense {M}x{N}x{K}")


def test_dense_outliers_and_small_weights():
    w = synth.make_dense(128, 1024, 2048, seed=3, a_outliers=True, b_std=0.02)
    got, sfa, sfb = run_dense(w)
    assert_within_tolerance(got, oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb), "decode-like")


def test_dense_scale_invariance_and_negation_bit_exact():
    w = synth.make_dense(256, 512, 1024, seed=11)
    base, sfa, sfb = run_dense(w)
    for k in (-3, 5):
        sfa_k = _pack(w["sfa"] * np.float32(2.0 ** k), w["M"], 1)[0]
        got_k, _, _ = run_dense(w, sfa=sfa_k, sfb=sfb)
        want_k = oracle.bf16_round_bits(oracle.bf16_bits_to_float(base) * 2.0 ** k)
        assert np.array_equal(got_k, want_k)
        sfb_k = _pack(w["sfb"] * np.float32(2.0 ** k), w["N"], 128)[0]
        got_kb, _, _ = run_dense(w, sfa=sfa, sfb=sfb_k)
        assert np.array_equal(got_kb, got_k)
    neg = dict(w, a=w["a"] ^ np.uint8(0x80))
    got_n, _, _ = run_dense(neg, sfa=sfa, sfb=sfb)
    assert np.array_equal(oracle.bf16_bits_to_float(got_n), -oracle.bf16_bits_to_float(base))


def test_dense_identity_exact():
    # B = identity (E4M3 1.0 on the diagonal), unit B scales: D = dequantised A, exactly.
    M, K = 256, 512
    w = synth.make_dense(M, K, K, seed=2)
    eye = np.zeros((K, K), np.uint8)
    eye[np.arange(K), np.arange(K)] = 0x38
    w = dict(w, b=eye, sfb=np.ones((K // 128, K // 128), np.float32))
    got, sfa, sfb = run_dense(w)
    want = oracle.fp8_gemm_nt(w["a"], sfa, eye, sfb)
    assert np.array_equal(oracle.bf16_bits_to_float(got), oracle.bf16_bits_to_float(want))


def test_pack_then_gemm_pipeline():
    # GPU pack feeding the GPU GEMM equals the GEMM on oracle-packed scales, bit for bit.
    w = synth.make_dense(192, 256, 1536, seed=21)
    ref_bits, sfa, sfb = run_dense(w)
    sfa_d = torch.empty(dg.packed_sf_shape(None, 192, 1536), dtype=torch.int32, device="cuda")
    sfb_d = torch.empty(dg.packed_sf_shape(None, 256, 1536), dtype=torch.int32, device="cuda")
    dg.dg_pack_sf_ue8m0(to_dev(w["sfa"]), sfa_d, 192, 1)
    dg.dg_pack_sf_ue8m0(to_dev(w["sfb"]), sfb_d, 256, 128)
    d = torch.empty((192, 256), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), sfa_d, to_dev(w["b"]), sfb_d, d)
    assert np.array_equal(bits(d), ref_bits)


# ---------------------------------------------------------------------------
# Contiguous layout
# ---------------------------------------------------------------------------

def run_contiguous(w):
    G, N, K, M_sum = w["G"], w["N"], w["K"], w["M_sum"]
    sfa = _pack(w["sfa"], M_sum, 1)[0]
    sfb = _pack(w["sfb"], N, 128)
    d = torch.full((M_sum, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_contiguous(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d,
                                          to_dev(w["m_indices"]))
    dg.dg_check_device_error()
    return bits(d), sfa, sfb


@pytest.mark.parametrize("G,N,K,counts", [
    (4, 512, 1024, [130, 0, 5, 256]),     # an empty expert, ragged segments
    (1, 256, 512, [384]),                 # one expert, no padding
    (3, 2112, 256, [1, 127, 129]),        # N tail, single-row expert
    (8, 96, 384, [17, 300, 0, 0, 128, 1, 64, 255]),
])
def test_contiguous_parity(G, N, K, counts):
    w = synth.make_contiguous(G, N, K, tokens=0, seed=G + N, counts=counts)
    got, sfa, sfb = run_contiguous(w)
    m_idx = w["m_indices"]
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(w["a"], sfa, w["b"], sfb, m_idx)
    valid = m_idx >= 0
    assert np.all(got[~valid] == 0), "padding rows must be +0.0"
    assert_within_tolerance(got[valid], want[valid], f"contiguous G={G}")


def test_contiguous_trailing_padding_blocks():
    # Whole 128-row blocks of -1 after the last expert are written as zeros.
    w = synth.make_contiguous(2, 256, 512, tokens=0, seed=5, counts=[100, 40])
    extra = 256
    w["m_indices"] = np.concatenate([w["m_indices"], np.full(extra, -1, np.int32)])
    w["a"] = np.concatenate([w["a"], np.full((extra, w["K"]), 0x7F, np.uint8)])
    w["sfa"] = np.concatenate([w["sfa"], np.ones((extra, w["K"] // 128), np.float32)])
    w["M_sum"] += extra
    got, sfa, sfb = run_contiguous(w)
    valid = w["m_indices"] >= 0
    assert np.all(got[~valid] == 0)
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(w["a"], sfa, w["b"], sfb, w["m_indices"])
    assert_within_tolerance(got[valid], want[valid], "trailing padding")


# ---------------------------------------------------------------------------
# Masked layout
# ---------------------------------------------------------------------------

def run_masked(w):
    G, max_m, N, K = w["G"], w["max_m"], w["N"], w["K"]
    sfa = _pack(w["sfa"], max_m, 1)
    sfb = _pack(w["sfb"], N, 128)
    d = torch.full((G, max_m, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_masked(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d,
                                      to_dev(w["masked_m"]))
    dg.dg_check_device_error()
    return bits(d), sfa, sfb


@pytest.mark.parametrize("G,max_m,N,K,masked_m", [
    (4, 256, 512, 1024, [0, 1, 255, 256]),
    (3, 200, 256, 512, [127, 128, 129]),
    (5, 64, 2112, 256, [64, 0, 0, 33, 1]),
    (2, 256, 96, 384, [0, 0]),                # nothing to compute: all rows untouched
])
def test_masked_parity(G, max_m, N, K, masked_m):
    w = synth.make_masked(G, max_m, N, K, seed=G + max_m, masked_m=masked_m)
    got, sfa, sfb = run_masked(w)
    prior = np.full((G, max_m, N), SENT, np.uint16)
    want = oracle.m_grouped_fp8_gemm_nt_masked(w["a"], sfa, w["b"], sfb, w["masked_m"], prior)
    rows = np.arange(max_m)[None, :] < np.asarray(masked_m)[:, None]
    assert np.array_equal(got[~rows], want[~rows]), "rows past masked_m must stay untouched"
    assert_within_tolerance(got[rows], want[rows], f"masked {masked_m}")


@pytest.mark.parametrize("pdl", [False, True])
def test_programmatic_dependent_launch_setting(pdl):
    # Results must not depend on whether kernels may start before the previous one finished:
    # a kernel writing the inputs runs right before the GEMM on the same stream.
    prev = dg.dg_get_pdl()
    dg.dg_set_pdl(pdl)
    try:
        w = synth.make_dense(256, 1024, 1536, seed=41)
        sfa = oracle.pack_sf_ue8m0(w["sfa"], 256, 1)[0]
        sfb = oracle.pack_sf_ue8m0(w["sfb"], 1024, 128)[0]
        a = torch.zeros((256, 1536), dtype=torch.uint8, device="cuda")
        src = to_dev(w["a"])
        d = torch.empty((256, 1024), dtype=torch.int16, device="cuda")
        a.copy_(src)                                   # produces A immediately before the GEMM
        dg.dg_fp8_gemm_nt(a, to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
        dg.dg_check_device_error()
        assert dg.dg_get_pdl() == pdl
        assert_within_tolerance(bits(d), oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb), f"pdl={pdl}")
    finally:
        dg.dg_set_pdl(prev)
