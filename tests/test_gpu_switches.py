"""Performance switches and schedules leave every result bit-identical.

The L2 weight prefetch before the dependency wait, the evict-first hint on outputs larger than
L2, the SM cap (which changes how many tiles each persistent CTA walks, and so which tiles
leave through the whole-tile ring stores and which through the row stores) and programmatic
dependent launch change only timing: the accumulators see the same MMAs in the same order, so
D must not change by a single bit.  One oracle check per case anchors the common result.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu


def _dense_case(M, N, K, seed):
    w = synth.make_dense(M, N, K, seed=seed, a_outliers=True, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    return w, sfa, sfb


def _run_dense(w, sfa, sfb):
    M, N = w["M"], w["N"]
    d = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    return bits(d)


@pytest.mark.parametrize("shape", [(64, 2112, 7168), (128, 24576, 1536), (100, 704, 2048)])
def test_weight_prefetch_is_bit_neutral(shape, monkeypatch):
    w, sfa, sfb = _dense_case(*shape, seed=41)
    outs = []
    for pf in ("0", "1"):
        monkeypatch.setenv("DG_PREFETCH_B", pf)
        outs.append(_run_dense(w, sfa, sfb))
    assert np.array_equal(outs[0], outs[1])
    assert_within_tolerance(outs[0], oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb), f"prefetch {shape}")


@pytest.mark.parametrize("sms", [8, 37])
@pytest.mark.parametrize("shape,cfg,split", [((128, 24576, 1536), "config_bn192_s5_k2", 1),
                                             ((200, 1408, 1024), "config_bn128_s5_k2", 1),
                                             ((64, 2112, 7168), "config_bn128_s8_k2_r64", 4)])
def test_schedule_and_store_path_are_bit_neutral(shape, cfg, split, sms, monkeypatch):
    # The plan is pinned (the planner's choice depends on the SM count).  With every SM each
    # CTA of the no-split plans computes one tile, its last, which leaves through the operand
    # ring; with a few SMs each CTA walks many tiles and all but its last go out through the
    # row stores.  The split-K plan reduces the same partials in the same order whichever
    # cluster runs them.
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    w, sfa, sfb = _dense_case(*shape, seed=43)
    full = _run_dense(w, sfa, sfb)
    dg.dg_set_num_sms(sms)
    try:
        capped = _run_dense(w, sfa, sfb)
    finally:
        dg.dg_set_num_sms(0)
    assert np.array_equal(full, capped)


def test_masked_schedule_is_bit_neutral(monkeypatch):
    monkeypatch.setenv("DG_FORCE_CONFIG", "config_bn192_s5_k2")
    monkeypatch.setenv("DG_FORCE_SPLIT", "1")
    m = synth.make_masked(4, 256, 7168, 2048, seed=44, masked_m=[72, 235, 70, 29])
    msfa = oracle.pack_sf_ue8m0(m["sfa"], 256, 1)
    msfb = oracle.pack_sf_ue8m0(m["sfb"], 7168, 128)
    args = (to_dev(m["a"]), to_dev(msfa), to_dev(m["b"]), to_dev(msfb))
    outs = []
    for sms in (0, 19):
        dg.dg_set_num_sms(sms)
        try:
            d = torch.full((4, 256, 7168), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
            dg.dg_m_grouped_fp8_gemm_nt_masked(*args, d, to_dev(m["masked_m"]))
            dg.dg_check_device_error()
            outs.append(bits(d))
        finally:
            dg.dg_set_num_sms(0)
    assert np.array_equal(outs[0], outs[1])
    prior = np.full((4, 256, 7168), synth.SENTINEL_BF16, np.uint16)
    want = oracle.m_grouped_fp8_gemm_nt_masked(m["a"], msfa, m["b"], msfb, m["masked_m"], prior)
    rows = np.arange(256)[None, :] < m["masked_m"][:, None]
    assert np.array_equal(outs[0][~rows], want[~rows])
    assert_within_tolerance(outs[0][rows], want[rows], "masked schedule")


def test_evict_first_hint_is_bit_neutral(monkeypatch):
    # An output above 128 MB takes the evict-first stores: 8448 rows x 8192 columns of BF16
    # (138 MB) through the 256-row tiles' TMA boxes; compared with the hint switched off and
    # with the oracle on sampled rows.
    M, N, K = 8448, 8192, 512
    w, sfa, sfb = _dense_case(M, N, K, seed=45)
    outs = []
    for ef in ("1", "0"):
        monkeypatch.setenv("DG_D_EVICT_FIRST", ef)
        outs.append(_run_dense(w, sfa, sfb))
    assert np.array_equal(outs[0], outs[1])
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))
    want = oracle.fp8_gemm_nt(w["a"][rows], oracle.pack_sf_ue8m0(w["sfa"][rows], rows.size, 1)[0], w["b"], sfb)
    assert_within_tolerance(outs[0][rows], want, "evict-first sample")
