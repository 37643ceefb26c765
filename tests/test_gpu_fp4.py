"""GPU parity of the FP8 x FP4 GEMMs (E4M3 activations, E2M1 weights packed two per byte)
against the oracle: dense, contiguous and masked layouts, and the kernel plans."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu

SENT = synth.SENTINEL_BF16


def run_dense(w):
    M, N = w["M"], w["N"]
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)[0]
    d = torch.full((M, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_fp4_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    return bits(d), oracle.fp8_fp4_gemm_nt(w["a"], sfa, w["b_fp4"], sfb)


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 128),      # one tile, one K block
    (128, 512, 1024),
    (64, 2112, 512),      # N tail, half an M tile
    (200, 96, 640),       # ragged M, Kb = 5
    (1, 256, 7168),
])
def test_fp8_fp4_dense_parity(M, N, K):
    w = synth.with_fp4_b(synth.make_dense(M, N, K, seed=M + N + K), seed=M + N + K)
    got, want = run_dense(w)
    assert_within_tolerance(got, want, f"fp8xfp4 {M}x{N}x{K}")


def test_fp8_fp4_contiguous_parity():
    G, N, K, counts = 4, 512, 1024, [130, 0, 5, 256]
    w = synth.with_fp4_b(synth.make_contiguous(G, N, K, tokens=0, seed=9, counts=counts), seed=9)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], w["M_sum"], 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)
    d = torch.full((w["M_sum"], N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d,
                                              to_dev(w["m_indices"]))
    dg.dg_check_device_error()
    got = bits(d)
    want = oracle.m_grouped_fp8_fp4_gemm_nt_contiguous(w["a"], sfa, w["b_fp4"], sfb, w["m_indices"])
    valid = w["m_indices"] >= 0
    assert np.all(got[~valid] == 0)
    assert_within_tolerance(got[valid], want[valid], "fp8xfp4 contiguous")


def test_fp8_fp4_masked_parity():
    G, max_m, N, K, masked_m = 4, 256, 512, 1024, [0, 1, 255, 256]
    w = synth.with_fp4_b(synth.make_masked(G, max_m, N, K, seed=10, masked_m=masked_m), seed=10)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], max_m, 1)
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)
    d = torch.full((G, max_m, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_fp4_gemm_nt_masked(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d,
                                          to_dev(w["masked_m"]))
    dg.dg_check_device_error()
    got = bits(d)
    prior = np.full((G, max_m, N), SENT, np.uint16)
    want = oracle.m_grouped_fp8_fp4_gemm_nt_masked(w["a"], sfa, w["b_fp4"], sfb, w["masked_m"], prior)
    rows = np.arange(max_m)[None, :] < np.asarray(masked_m)[:, None]
    assert np.array_equal(got[~rows], want[~rows])
    assert_within_tolerance(got[rows], want[rows], "fp8xfp4 masked")


def test_fp4_weights_equal_their_e4m3_images():
    # Every E2M1 value is an E4M3 value, so the FP4 GEMM must give the FP8 GEMM's bits on the
    # same weights written as E4M3 codes (same sums, same order).
    M, N, K = 256, 512, 2048
    w = synth.with_fp4_b(synth.make_dense(M, N, K, seed=12), seed=12)
    got, _ = run_dense(w)
    vals = oracle.e2m1_decode_table()[oracle.fp4_unpack(w["b_fp4"])]
    b8 = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)[0]
    d8 = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(b8), to_dev(sfb), d8)
    assert np.array_equal(got, bits(d8))


@pytest.fixture
def forced(monkeypatch):
    def setter(cfg=None, split=None):
        for k in ("DG_FORCE_CONFIG", "DG_FORCE_SPLIT"):
            monkeypatch.delenv(k, raising=False)
        if cfg:
            monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
        if split:
            monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    return setter


@pytest.mark.parametrize("cfg,split", [
    ("config_bn256_s4_a1", None), ("config_bn224_s4_a2", None), ("config_bn192_s5_a2", None),
    ("config_bn128_s4_a2", 4), ("config_bn64_s8_a2", 8), ("config_bn32_s8_a2", 2),
    ("config_bn224_s3_m2", None), ("config_bn192_s3_m2", None), ("config_bn208_s3_m2", None),
    ("config_bn128_s5_k2", 4), ("config_bn192_s5_k2", None),
])
def test_fp8_fp4_forced_plans(forced, cfg, split):
    forced(cfg, split)
    w = synth.with_fp4_b(synth.make_dense(256, 1024, 4096, seed=13), seed=13)
    got, want = run_dense(w)
    assert_within_tolerance(got, want, f"{cfg} split={split}")
