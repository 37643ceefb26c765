"""The compile-time kernel variants for decode-style calls (dense or masked, E4M3 B; K-major, BF16
out, no C) against the general kernel: with the configuration and split forced, the same
problem must give bit-identical accumulators whichever variant runs it.

* dense BF16 (the dense variant) vs the NT layout with FP32 output (the general kernel), the
  FP32 result rounded to BF16 (round to nearest even) on the host;
* dense (dense variant) vs masked with one group holding every row (masked variant).
The oracle checks of either path are elsewhere; this pins the variants to each other."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import bits, to_dev

pytestmark = pytest.mark.gpu

PLANS = [("config_bn128_s5_k2", 4), ("config_bn192_s5_k2", 1), ("config_bn128_s4_a2", 2),
         ("config_bn192_s5_a2", 1), ("config_bn64_s8_a2", 2)]
# 64-row A stages take calls of at most 64 rows: the dense comparison (M = 64) only
DENSE_PLANS = PLANS + [("config_bn128_s8_k2_r64", 1), ("config_bn128_s8_k2_r64", 4), ("config_bn128_s8_k2_r64", 8)]


def _bf16_rne_bits(x):
    """FP32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@pytest.fixture
def forced(monkeypatch):
    def setter(cfg, split):
        monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
        monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    return setter


@pytest.mark.parametrize("cfg,split", DENSE_PLANS)
def test_dense_variant_matches_general_kernel(forced, cfg, split):
    forced(cfg, split)
    M, N, K = 64, 704, 2048
    w = synth.make_dense(M, N, K, seed=91, a_outliers=True, b_std=0.02)
    sfa = to_dev(oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0])
    sfb = to_dev(oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0])
    a, b = to_dev(w["a"]), to_dev(w["b"])
    d16 = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    d32 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    dg.dg_fp8_gemm_nt(a, sfa, b, sfb, d16)                       # dense variant
    dg.dg_fp8_gemm(a, sfa, b, sfb, d32, layout="nt")             # FP32 out: general kernel
    dg.dg_check_device_error()
    assert np.array_equal(bits(d16), _bf16_rne_bits(d32.cpu().numpy())), f"{cfg} split {split}"


@pytest.mark.parametrize("cfg,split", [(c, 1) for c, _ in PLANS])
def test_masked_variant_matches_dense_variant(forced, cfg, split):
    forced(cfg, split)
    M, N, K = 200, 704, 2048
    w = synth.make_dense(M, N, K, seed=92, a_outliers=True, b_std=0.02)
    sfa_p = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb_p = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    a, b, sfa, sfb = to_dev(w["a"]), to_dev(w["b"]), to_dev(sfa_p), to_dev(sfb_p)
    dd = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dm = torch.full((1, M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(a, sfa, b, sfb, dd)
    dg.dg_m_grouped_fp8_gemm_nt_masked(a.unsqueeze(0).contiguous(), sfa.unsqueeze(0).contiguous(),
                                       b.unsqueeze(0).contiguous(), sfb.unsqueeze(0).contiguous(), dm,
                                       torch.tensor([M], dtype=torch.int32, device="cuda"))
    dg.dg_check_device_error()
    assert np.array_equal(bits(dd), bits(dm)[0]), f"{cfg} split {split}"
