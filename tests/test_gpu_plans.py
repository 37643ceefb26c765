"""Every kernel configuration and split-K factor, forced one at a time, against the oracle.

The SM count is capped so that each persistent CTA (or cluster) walks many tiles: the
pipeline, scale-ring and accumulator barriers then go through many phases, across tile
boundaries, which is where ordering mistakes show.  Split-K runs the CTAs of a thread-block
cluster over disjoint K ranges of one tile and reduces through distributed shared memory.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu

CONFIGS = ["config_bn256_s4_a1", "config_bn224_s4_a2", "config_bn192_s5_a2", "config_bn128_s6_a2",
           "config_bn128_s4_a2", "config_bn64_s8_a2", "config_bn32_s8_a2", "config_bn224_s3_m2",
           "config_bn192_s3_m2", "config_bn208_s3_m2", "config_bn128_s5_k2", "config_bn192_s5_k2",
           "config_bn128_s8_k2_r64"]


def _call_or_skip(fn, *args):
    """A forced (configuration, split) pair that does not fit in shared memory is refused
    with DG_ERR_SHAPE before launch; such pairs are never chosen by the planner."""
    try:
        fn(*args)
    except dg.DGError as e:
        if e.status == 2:
            pytest.skip("forced plan does not fit in shared memory")
        raise


@pytest.fixture
def few_sms():
    dg.dg_set_num_sms(8)
    yield
    dg.dg_set_num_sms(0)


def _dense(M, N, K, seed):
    w = synth.make_dense(M, N, K, seed=seed, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    return w, sfa, sfb, oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb)


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("split", [1, 2, 4])
def test_dense_every_plan(cfg, split, few_sms, monkeypatch):
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    M, N, K = 320, 704, 2560          # ragged M and N tails, 20 K blocks (5 groups of 4)
    w, sfa, sfb, want = _dense(M, N, K, seed=len(cfg) + split)
    d = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_fp8_gemm_nt, to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), want, f"{cfg} split {split}")


@pytest.mark.parametrize("split", [2, 3, 4, 5, 6, 8])
def test_split_k_decode_shape(split, monkeypatch):
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    M, N, K = 64, 2112, 7168
    w = synth.make_dense(M, N, K, seed=7, a_outliers=True, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    d = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb), f"decode split {split}")


@pytest.mark.parametrize("cfg", ["config_bn128_s8_k2_r64"])
@pytest.mark.parametrize("M", [1, 37, 64])
@pytest.mark.parametrize("split", [1, 2, 3, 4, 6, 8])
def test_64_row_a_stages(cfg, M, split, few_sms, monkeypatch):
    # The configurations that load only 64 rows of A per stage (their MMAs still read 128 rows,
    # the upper 64 from the next buffer): dense calls of at most 64 rows, on a few SMs so that
    # each CTA (or cluster) walks many tiles, D pre-filled with a sentinel.
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    N, K = 704, 4608
    w, sfa, sfb, want = _dense(M, N, K, seed=M + split)
    d = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_fp8_gemm_nt, to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), want, f"64-row A {cfg}, M {M} split {split}")
    # masked layout, groups of at most 64 rows
    m = synth.make_masked(3, 64, 320, K, seed=M + 5 * split, masked_m=[64, 0, 17])
    msfa = oracle.pack_sf_ue8m0(m["sfa"], 64, 1)
    msfb = oracle.pack_sf_ue8m0(m["sfb"], 320, 128)
    md = torch.full((3, 64, 320), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_m_grouped_fp8_gemm_nt_masked, to_dev(m["a"]), to_dev(msfa), to_dev(m["b"]), to_dev(msfb),
                  md, to_dev(m["masked_m"]))
    dg.dg_check_device_error()
    prior = np.full((3, 64, 320), synth.SENTINEL_BF16, np.uint16)
    wantm = oracle.m_grouped_fp8_gemm_nt_masked(m["a"], msfa, m["b"], msfb, m["masked_m"], prior)
    got = bits(md)
    rows = np.arange(64)[None, :] < m["masked_m"][:, None]
    assert np.array_equal(got[~rows], wantm[~rows])
    assert_within_tolerance(got[rows], wantm[rows], f"64-row A {cfg} masked split {split}")


def test_64_row_a_stages_refuse_taller_calls(monkeypatch):
    # 65 rows of A do not fit 64-row stages: the forced plan is refused before any launch.
    monkeypatch.setenv("DG_FORCE_CONFIG", "config_bn128_s8_k2_r64")
    w, sfa, sfb, _ = _dense(65, 256, 512, seed=1)
    d = torch.empty((65, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    assert e.value.status == 2


@pytest.mark.parametrize("cfg", ["config_bn128_s6_a2", "config_bn128_s4_a2", "config_bn64_s8_a2",
                                 "config_bn224_s3_m2", "config_bn128_s5_k2", "config_bn192_s5_k2"])
@pytest.mark.parametrize("split", [1, 2, 4])
def test_grouped_every_plan(cfg, split, few_sms, monkeypatch):
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    c = synth.make_contiguous(3, 256, 2048, tokens=0, seed=3, counts=[130, 0, 300])
    csfa = oracle.pack_sf_ue8m0(c["sfa"], c["M_sum"], 1)[0]
    csfb = oracle.pack_sf_ue8m0(c["sfb"], 256, 128)
    d = torch.full((c["M_sum"], 256), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_m_grouped_fp8_gemm_nt_contiguous, to_dev(c["a"]), to_dev(csfa), to_dev(c["b"]),
                  to_dev(csfb), d, to_dev(c["m_indices"]))
    dg.dg_check_device_error()
    got = bits(d)
    valid = c["m_indices"] >= 0
    assert np.all(got[~valid] == 0)
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(c["a"], csfa, c["b"], csfb, c["m_indices"])
    assert_within_tolerance(got[valid], want[valid], f"contiguous {cfg} split {split}")

    m = synth.make_masked(3, 200, 320, 2048, seed=4, masked_m=[199, 0, 129])
    msfa = oracle.pack_sf_ue8m0(m["sfa"], 200, 1)
    msfb = oracle.pack_sf_ue8m0(m["sfb"], 320, 128)
    md = torch.full((3, 200, 320), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_masked(to_dev(m["a"]), to_dev(msfa), to_dev(m["b"]), to_dev(msfb), md,
                                      to_dev(m["masked_m"]))
    dg.dg_check_device_error()
    prior = np.full((3, 200, 320), synth.SENTINEL_BF16, np.uint16)
    want = oracle.m_grouped_fp8_gemm_nt_masked(m["a"], msfa, m["b"], msfb, m["masked_m"], prior)
    got = bits(md)
    rows = np.arange(200)[None, :] < m["masked_m"][:, None]
    assert np.array_equal(got[~rows], want[~rows])
    assert_within_tolerance(got[rows], want[rows], f"masked {cfg} split {split}")


@pytest.mark.parametrize("cfg", ["config_bn224_s3_m2", "config_bn192_s3_m2", "config_bn208_s3_m2"])
def test_contiguous_256_row_tiles_straddling_experts(cfg, few_sms, monkeypatch):
    # 256-row tiles (two 128-row halves): expert 0 has one block and expert 1 two, so the first
    # tile holds two experts and runs as two passes; then a trailing all-padding tile.
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    c = synth.make_contiguous(4, 448, 1536, tokens=0, seed=12, counts=[100, 200, 0, 129])
    extra = 256
    c["m_indices"] = np.concatenate([c["m_indices"], np.full(extra, -1, np.int32)])
    c["a"] = np.concatenate([c["a"], np.full((extra, c["K"]), 0x7F, np.uint8)])
    c["sfa"] = np.concatenate([c["sfa"], np.ones((extra, c["K"] // 128), np.float32)])
    c["M_sum"] += extra
    csfa = oracle.pack_sf_ue8m0(c["sfa"], c["M_sum"], 1)[0]
    csfb = oracle.pack_sf_ue8m0(c["sfb"], 448, 128)
    d = torch.full((c["M_sum"], 448), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_contiguous(to_dev(c["a"]), to_dev(csfa), to_dev(c["b"]), to_dev(csfb), d,
                                          to_dev(c["m_indices"]))
    dg.dg_check_device_error()
    got = bits(d)
    valid = c["m_indices"] >= 0
    assert np.all(got[~valid] == 0)
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(c["a"], csfa, c["b"], csfb, c["m_indices"])
    assert_within_tolerance(got[valid], want[valid], f"contiguous 256-row tiles {cfg}")


@pytest.mark.parametrize("cfg", ["config_bn128_s4_a2", "config_bn64_s8_a2", "config_bn32_s8_a2"])
@pytest.mark.parametrize("split", [2, 3, 4, 5, 6, 7, 8])
def test_split_k_rows_per_owner(cfg, split, few_sms, monkeypatch):
    # ceil(V / split) rows of each tile's V valid rows per owning CTA (64, 43, 32, 26, 22, 19 and
    # 16 of a full 128-row tile; the last owner takes fewer); 36 K blocks = 9 groups, so most
    # splits have uneven K ranges; ragged M and N.
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    M, N, K = 200, 448, 4608
    w, sfa, sfb, want = _dense(M, N, K, seed=split * 10 + len(cfg))
    d = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_fp8_gemm_nt, to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), want, f"{cfg} split {split}")
    # masked layout with the same split
    m = synth.make_masked(2, 160, 192, K, seed=split, masked_m=[160, 17])
    msfa = oracle.pack_sf_ue8m0(m["sfa"], 160, 1)
    msfb = oracle.pack_sf_ue8m0(m["sfb"], 192, 128)
    md = torch.full((2, 160, 192), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_masked(to_dev(m["a"]), to_dev(msfa), to_dev(m["b"]), to_dev(msfb), md,
                                      to_dev(m["masked_m"]))
    dg.dg_check_device_error()
    prior = np.full((2, 160, 192), synth.SENTINEL_BF16, np.uint16)
    wantm = oracle.m_grouped_fp8_gemm_nt_masked(m["a"], msfa, m["b"], msfb, m["masked_m"], prior)
    got = bits(md)
    rows = np.arange(160)[None, :] < m["masked_m"][:, None]
    assert np.array_equal(got[~rows], wantm[~rows])
    assert_within_tolerance(got[rows], wantm[rows], f"masked {cfg} split {split}")


@pytest.mark.parametrize("cfg,split", [("config_bn128_s5_k2", 4), ("config_bn128_s4_a2", 2),
                                       ("config_bn128_s5_k2", 2), ("config_bn64_s8_a2", 8)])
def test_split_k_contiguous_trailing_padding(cfg, split, few_sms, monkeypatch):
    # Whole 128-row blocks of padding after the last expert are zero units; on a few SMs each
    # cluster walks several units and its last ones are such zero units, so the units before
    # them take the unit-to-unit handshake path rather than the last-unit one.
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    c = synth.make_contiguous(2, 256, 2048, tokens=0, seed=9, counts=[200, 130])
    K, pad = 2048, 3 * 128
    a = np.concatenate([c["a"], np.full((pad, K), synth.NAN_CODE, np.uint8)])
    sfa_f = np.concatenate([c["sfa"], np.ones((pad, c["sfa"].shape[1]), np.float32)])
    m_idx = np.concatenate([c["m_indices"], np.full(pad, -1, np.int32)])
    M_sum = a.shape[0]
    csfa = oracle.pack_sf_ue8m0(sfa_f, M_sum, 1)[0]
    csfb = oracle.pack_sf_ue8m0(c["sfb"], 256, 128)
    d = torch.full((M_sum, 256), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    _call_or_skip(dg.dg_m_grouped_fp8_gemm_nt_contiguous, to_dev(a), to_dev(csfa), to_dev(c["b"]),
                  to_dev(csfb), d, to_dev(m_idx))
    dg.dg_check_device_error()
    got = bits(d)
    valid = m_idx >= 0
    assert np.all(got[~valid] == 0)
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(a, csfa, c["b"], csfb, m_idx)
    assert_within_tolerance(got[valid], want[valid], f"contiguous + trailing padding {cfg} split {split}")
