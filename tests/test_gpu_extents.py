"""GPU parity at the extremes of the extents: many K blocks, many column tiles, many groups.

Each case drives one index of the kernels far past the bench's shapes: a K of 65536 (512
K blocks per output tile, 128 packed scale words per row), N = 131136 (1025 column tiles of
128, an N tail of 64), 4096 masked groups (the library's maximum: the device-side prefix over
the groups is at its largest), a contiguous call over 256 experts, many of them empty, a
K-grouped call over 64 ragged or empty groups, and E2M1 weights over 256 K blocks.  Results are checked element by element against the oracle; rows the layouts must not
touch are checked bit-exactly.
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


def _dense(M, N, K, seed):
    w = synth.make_dense(M, N, K, seed=seed, a_outliers=True, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    d = torch.full((M, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    return bits(d), oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb)


@pytest.mark.parametrize("split", [None, 8])
def test_long_k(split, monkeypatch):
    # 512 K blocks: the split-K ranges (when forced) still hold 64 blocks each.
    if split:
        monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    got, want = _dense(128, 256, 65536, seed=81)
    assert_within_tolerance(got, want, f"K = 65536, split {split}")


def test_wide_n():
    # 1025 column tiles of 128 for one 64-row block; the last tile holds 64 columns.
    got, want = _dense(64, 131136, 256, seed=82)
    assert_within_tolerance(got, want, "N = 131136")


def test_most_masked_groups():
    G, max_m, N, K = 4096, 8, 128, 128
    masked_m = synth.rng(83, "masked_m").integers(0, max_m + 1, size=G).astype(np.int32)
    m = synth.make_masked(G, max_m, N, K, seed=83, masked_m=masked_m)
    msfa = oracle.pack_sf_ue8m0(m["sfa"], max_m, 1)
    msfb = oracle.pack_sf_ue8m0(m["sfb"], N, 128)
    d = torch.full((G, max_m, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_masked(to_dev(m["a"]), to_dev(msfa), to_dev(m["b"]), to_dev(msfb), d,
                                      to_dev(m["masked_m"]))
    dg.dg_check_device_error()
    got = bits(d)
    prior = np.full((G, max_m, N), SENT, np.uint16)
    want = oracle.m_grouped_fp8_gemm_nt_masked(m["a"], msfa, m["b"], msfb, m["masked_m"], prior)
    rows = np.arange(max_m)[None, :] < m["masked_m"][:, None]
    assert np.array_equal(got[~rows], want[~rows]), "rows past masked_m must stay untouched"
    assert_within_tolerance(got[rows], want[rows], "4096 masked groups")


def test_many_contiguous_experts():
    G, N, K = 256, 256, 256
    counts = synth.rng(84, "counts").integers(0, 300, size=G)
    counts[synth.rng(84, "counts", sub=1).random(G) < 0.4] = 0   # many experts receive no token
    w = synth.make_contiguous(G, N, K, tokens=0, seed=84, counts=counts)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], w["M_sum"], 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
    d = torch.full((w["M_sum"], N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_contiguous(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d,
                                          to_dev(w["m_indices"]))
    dg.dg_check_device_error()
    got = bits(d)
    valid = w["m_indices"] >= 0
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(w["a"], sfa, w["b"], sfb, w["m_indices"])
    assert np.all(got[~valid] == 0), "padding rows must be +0.0"
    assert_within_tolerance(got[valid], want[valid], "256 experts")


def test_k_grouped_many_groups():
    # 64 expert gradients, their K (token) ranges ragged, a quarter of them empty.
    from tests._parity import assert_close_f32
    G, M, N = 64, 128, 256
    ks = (synth.rng(85, "counts").integers(0, 6, size=G) * 128).astype(np.int64)
    ks[synth.rng(85, "counts", sub=1).random(G) < 0.25] = 0
    w = synth.make_k_grouped(M, N, ks, seed=85)
    sfa = oracle.pack_sf_ue8m0_k_grouped(w["sfa"], M, ks)
    sfb = oracle.pack_sf_ue8m0_k_grouped(w["sfb"], N, ks)
    d = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_k_grouped_fp8_gemm_tn_contiguous(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d,
                                           to_dev(ks.astype(np.int32)))
    dg.dg_check_device_error()
    got = d.cpu().numpy()
    want = oracle.k_grouped_fp8_gemm_tn_contiguous(w["a"], sfa, w["b"], sfb, ks)
    assert_close_f32(got, want, "64 K groups")
    for g in np.nonzero(ks == 0)[0]:
        assert np.all(got[g] == 0) and not np.any(np.signbit(got[g]))


def test_fp8_fp4_long_k():
    # E2M1 weights over 256 K blocks (64 packed scale words per row).
    M, N, K = 64, 512, 32768
    w = synth.with_fp4_b(synth.make_dense(M, N, K, seed=86), seed=86)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)[0]
    d = torch.full((M, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_fp4_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), oracle.fp8_fp4_gemm_nt(w["a"], sfa, w["b_fp4"], sfb), "fp8xfp4 K = 32768")
