"""The benchmark's workloads at full size, through the same calls (and so the same kernel
configurations) the benchmark times, checked against the oracle.

The decode shapes and the masked MoE workload are compared in full.  For the prefill GEMM
(4096 x 7168 x 16384) and the contiguous MoE GEMM (33k rows x 4096 x 7168) the oracle computes
a sample of at least 512 full rows (covering every 128-row block, its first and last row, with
all columns); every element of the GPU result is additionally checked to be finite, and every
padding row to be bit-exact +0.0.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu


def _gpu_packed(sf, mn, gran, groups=None):
    K = sf.shape[-1] * 128
    out = torch.empty(dg.packed_sf_shape(groups, mn, K), dtype=torch.int32, device="cuda")
    dg.dg_pack_sf_ue8m0(to_dev(sf), out, mn, gran)
    return out


MIN_SAMPLED_ROWS = 512


def _sample_rows(nrows, per_block, seed):
    """The first and last row of every 128-row block plus `per_block` distinct random rows of it."""
    rs = np.random.default_rng(seed)
    rows = []
    for b0 in range(0, nrows, 128):
        blk = np.arange(b0, min(nrows, b0 + 128))
        rows += [blk[0], blk[-1]] + list(rs.choice(blk, size=min(per_block, blk.size), replace=False))
    return np.unique(np.array(rows))


@pytest.mark.parametrize("shape_idx", range(len(synth.DECODE_SHAPES)))
def test_decode_shapes_full(shape_idx):
    M, N, K = synth.DECODE_SHAPES[shape_idx]
    w = synth.make_dense(M, N, K, seed=shape_idx, a_outliers=True, b_std=0.02)
    sfa, sfb = _gpu_packed(w["sfa"], M, 1), _gpu_packed(w["sfb"], N, 128)
    d = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), sfa, to_dev(w["b"]), sfb, d)
    dg.dg_check_device_error()
    sfa_ref = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb_ref = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    assert np.array_equal(sfa.cpu().numpy(), sfa_ref) and np.array_equal(sfb.cpu().numpy(), sfb_ref)
    want = oracle.fp8_gemm_nt(w["a"], sfa_ref, w["b"], sfb_ref)
    assert_within_tolerance(bits(d), want, f"decode {M}x{N}x{K}")


def test_prefill_sampled_rows():
    M, N, K = synth.PREFILL_SHAPE
    w = synth.make_dense(M, N, K, seed=10, b_std=0.02)
    sfa, sfb = _gpu_packed(w["sfa"], M, 1), _gpu_packed(w["sfb"], N, 128)
    d = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), sfa, to_dev(w["b"]), sfb, d)
    dg.dg_check_device_error()
    got = bits(d)
    assert np.all(np.isfinite(oracle.bf16_bits_to_float(got)))
    rows = _sample_rows(M, 16, seed=1)
    assert rows.size >= MIN_SAMPLED_ROWS
    sfa_ref = oracle.pack_sf_ue8m0(w["sfa"][rows], rows.size, 1)[0]
    sfb_ref = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    want = oracle.fp8_gemm_nt(w["a"][rows], sfa_ref, w["b"], sfb_ref)
    assert_within_tolerance(got[rows], want, "prefill sample")


def test_contiguous_moe_sampled_rows():
    c = synth.CONTIGUOUS
    w = synth.make_contiguous(c["G"], c["N"], c["K"], c["tokens"], seed=20)
    M_sum, N = w["M_sum"], w["N"]
    sfa = _gpu_packed(w["sfa"], M_sum, 1)
    sfb = _gpu_packed(w["sfb"], N, 128, groups=c["G"])
    d = torch.full((M_sum, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_contiguous(to_dev(w["a"]), sfa, to_dev(w["b"]), sfb, d, to_dev(w["m_indices"]))
    dg.dg_check_device_error()
    got = bits(d)
    m_idx = w["m_indices"]
    assert np.all(got[m_idx < 0] == 0), "padding rows must be +0.0"
    assert np.all(np.isfinite(oracle.bf16_bits_to_float(got[m_idx >= 0])))
    rows = _sample_rows(M_sum, 2, seed=2)
    rows = rows[m_idx[rows] >= 0]
    assert rows.size >= MIN_SAMPLED_ROWS
    sfa_ref = oracle.pack_sf_ue8m0(w["sfa"], M_sum, 1)[0]
    sfb_ref = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
    want = oracle.m_grouped_fp8_gemm_nt_contiguous(w["a"], sfa_ref, w["b"], sfb_ref, m_idx, rows=rows)
    assert_within_tolerance(got[rows], want, "contiguous sample")


def test_masked_moe_full():
    m = synth.MASKED
    w = synth.make_masked(m["G"], m["max_m"], m["N"], m["K"], seed=30)
    G, max_m, N = w["G"], w["max_m"], w["N"]
    sfa = _gpu_packed(w["sfa"], max_m, 1, groups=G)
    sfb = _gpu_packed(w["sfb"], N, 128, groups=G)
    d = torch.full((G, max_m, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_gemm_nt_masked(to_dev(w["a"]), sfa, to_dev(w["b"]), sfb, d, to_dev(w["masked_m"]))
    dg.dg_check_device_error()
    got = bits(d)
    sfa_ref = oracle.pack_sf_ue8m0(w["sfa"], max_m, 1)
    sfb_ref = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
    prior = np.full((G, max_m, N), synth.SENTINEL_BF16, np.uint16)
    want = oracle.m_grouped_fp8_gemm_nt_masked(w["a"], sfa_ref, w["b"], sfb_ref, w["masked_m"], prior)
    rows = np.arange(max_m)[None, :] < w["masked_m"][:, None]
    assert np.array_equal(got[~rows], want[~rows])
    assert_within_tolerance(got[rows], want[rows], "masked full")


# ---------------------------------------------------------------------------
# The shapes the benchmark times beside the step, at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape_idx", range(len(synth.DECODE_SHAPES)))
def test_fp8_fp4_decode_shapes_full(shape_idx):
    M, N, K = synth.DECODE_SHAPES[shape_idx]
    w = synth.with_fp4_b(synth.make_dense(M, N, K, seed=20 + shape_idx, a_outliers=True), seed=20 + shape_idx)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)[0]
    d = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_fp4_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), oracle.fp8_fp4_gemm_nt(w["a"], sfa, w["b_fp4"], sfb), f"fp8xfp4 {M}x{N}x{K}")


def test_fp8_fp4_masked_full():
    m = synth.MASKED
    w = synth.with_fp4_b(synth.make_masked(m["G"], m["max_m"], m["N"], m["K"], seed=0), seed=0)
    G, max_m, N = m["G"], m["max_m"], m["N"]
    sfa = oracle.pack_sf_ue8m0(w["sfa"], max_m, 1)
    sfb = oracle.pack_sf_ue8m0(w["sfb_fp4"], N, 1)
    d = torch.full((G, max_m, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    dg.dg_m_grouped_fp8_fp4_gemm_nt_masked(to_dev(w["a"]), to_dev(sfa), to_dev(w["b_fp4"]), to_dev(sfb), d,
                                          to_dev(w["masked_m"]))
    dg.dg_check_device_error()
    prior = np.full((G, max_m, N), synth.SENTINEL_BF16, np.uint16)
    want = oracle.m_grouped_fp8_fp4_gemm_nt_masked(w["a"], sfa, w["b_fp4"], sfb, w["masked_m"], prior)
    got = bits(d)
    rows = np.arange(max_m)[None, :] < w["masked_m"][:, None]
    assert np.array_equal(got[~rows], want[~rows])
    assert_within_tolerance(got[rows], want[rows], "fp8xfp4 masked full")


def test_nn_layout_fp32_accumulate_prefill_sampled_rows():
    # The prefill shape in the NN layout, D += A B^T in FP32 in place: sampled rows of every
    # 128-row block against the oracle (which adds C exactly).
    M, N, K = synth.PREFILL_SHAPE
    w = synth.make_dense(M, N, K, seed=11, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    b_nn = np.ascontiguousarray(w["b"].T)                          # [K, N]
    c = synth.normal((M, N), 11, "d_fill", std=0.5)
    d = to_dev(c)
    dg.dg_fp8_gemm(to_dev(w["a"]), to_dev(sfa), to_dev(b_nn), to_dev(sfb), d, layout="nn", c=d)
    dg.dg_check_device_error()
    got = d.cpu().numpy()
    assert np.all(np.isfinite(got))
    rows = _sample_rows(M, 16, seed=11)
    assert rows.size >= MIN_SAMPLED_ROWS
    want = oracle.fp8_gemm(w["a"][rows], oracle.pack_sf_ue8m0(w["sfa"][rows], len(rows), 1)[0], b_nn, sfb,
                           layout="nn", c=c[rows], out="f32")
    from tests._parity import assert_close_f32
    assert_close_f32(got[rows], want, "nn f32 accumulate prefill")
