"""GPU parity of the K-grouped weight-gradient GEMM and its per-group scale pack."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_close_f32, to_dev

pytestmark = pytest.mark.gpu


def run(w, c=None, in_place=False, pack_on_gpu=False):
    G, M, N, ks = w["G"], w["M"], w["N"], w["ks"]
    if pack_on_gpu:
        ks_d = to_dev(ks)
        rows = dg.k_grouped_packed_sf_rows(ks)
        sfa = torch.empty((rows, dg.dg_get_tma_aligned_size(M)), dtype=torch.int32, device="cuda")
        sfb = torch.empty((rows, dg.dg_get_tma_aligned_size(N)), dtype=torch.int32, device="cuda")
        dg.dg_pack_sf_ue8m0_k_grouped(to_dev(w["sfa"]), sfa, ks_d, M)
        dg.dg_pack_sf_ue8m0_k_grouped(to_dev(w["sfb"]), sfb, ks_d, N)
        sfa_h, sfb_h = sfa.cpu().numpy(), sfb.cpu().numpy()
    else:
        sfa_h = oracle.pack_sf_ue8m0_k_grouped(w["sfa"], M, ks)
        sfb_h = oracle.pack_sf_ue8m0_k_grouped(w["sfb"], N, ks)
        sfa, sfb = to_dev(sfa_h), to_dev(sfb_h)
    d = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    cd = None
    if c is not None:
        cd = to_dev(c)
        if in_place:
            d.copy_(cd)
            cd = d
    dg.dg_k_grouped_fp8_gemm_tn_contiguous(to_dev(w["a"]), sfa, to_dev(w["b"]), sfb, d, to_dev(ks), c=cd)
    dg.dg_check_device_error()
    want = oracle.k_grouped_fp8_gemm_tn_contiguous(w["a"], sfa_h, w["b"], sfb_h, ks, c=c)
    return d.cpu().numpy(), want, (sfa_h, sfb_h)


@pytest.mark.parametrize("M,N,ks", [
    (256, 384, [256, 0, 384, 128]),          # an empty group, ragged group sizes
    (128, 256, [128]),                       # one group, one K block
    (384, 512, [640, 1152]),                 # Kb = 5 and 9: partly filled packed words
    (64, 1040, [512, 256, 0, 0, 128]),       # M below a tile, N tail, trailing empty groups
])
def test_k_grouped_parity(M, N, ks):
    w = synth.make_k_grouped(M, N, ks, seed=M + N + len(ks))
    got, want, _ = run(w)
    assert_close_f32(got, want, f"k-grouped {M}x{N} ks={ks}")
    for g, k in enumerate(ks):
        if k == 0:
            assert np.all(got[g] == 0) and not np.any(np.signbit(got[g]))


def test_k_grouped_accumulate_and_in_place():
    M, N, ks = 256, 512, [384, 0, 256]
    w = synth.make_k_grouped(M, N, ks, seed=81)
    c = synth.normal((len(ks), M, N), 81, "d_fill", std=2.0)
    got, want, _ = run(w, c=c)
    assert_close_f32(got, want, "with C")
    assert np.array_equal(got[1], c[1])                     # empty group: D = C exactly
    got, want, _ = run(w, c=c, in_place=True)
    assert_close_f32(got, want, "in place")


def test_k_grouped_pack_bit_exact_and_pipeline():
    M, N, ks = 256, 384, [640, 0, 128, 1024, 384]
    w = synth.make_k_grouped(M, N, ks, seed=82)
    got, want, (sfa_g, sfb_g) = run(w, pack_on_gpu=True)
    assert np.array_equal(sfa_g.view(np.uint32), oracle.pack_sf_ue8m0_k_grouped(w["sfa"], M, ks).view(np.uint32))
    assert np.array_equal(sfb_g.view(np.uint32), oracle.pack_sf_ue8m0_k_grouped(w["sfb"], N, ks).view(np.uint32))
    assert_close_f32(got, want, "GPU-packed scales")


def test_k_grouped_all_groups_empty():
    M, N, G = 128, 256, 3
    ks = np.zeros(G, np.int32)
    c = synth.normal((G, M, N), 83, "d_fill")
    d = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    # sum_K = 0: the operands are never read; small valid buffers stand in for them
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    cd = to_dev(c)
    ks_d = to_dev(ks)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = dg.load_library().dg_k_grouped_fp8_gemm_tn_contiguous(
        p(buf), p(buf), p(buf), p(buf), p(cd), p(d), p(ks_d), G, M, N, 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    dg.dg_check_device_error()
    assert np.array_equal(d.cpu().numpy(), c)


def test_k_grouped_weight_gradient_shape_sampled():
    # The MoE weight-gradient shape: 4 experts, M = 4096 (N of the forward GEMM), N = 7168 (its
    # K), 32768 tokens split unevenly; sampled (m, n) blocks checked against the oracle.
    M, N = 4096, 7168
    ks = [9216, 7168, 8448, 7936]
    w = synth.make_k_grouped(M, N, ks, seed=0)
    ks_a = np.asarray(ks, np.int32)
    sfa_h = oracle.pack_sf_ue8m0_k_grouped(w["sfa"], M, ks)
    sfb_h = oracle.pack_sf_ue8m0_k_grouped(w["sfb"], N, ks)
    d = torch.empty((4, M, N), dtype=torch.float32, device="cuda")
    dg.dg_k_grouped_fp8_gemm_tn_contiguous(to_dev(w["a"]), to_dev(sfa_h), to_dev(w["b"]), to_dev(sfb_h), d,
                                           to_dev(ks_a))
    dg.dg_check_device_error()
    rs = synth.rng(0, "perm", 11)
    koff = np.concatenate([[0], np.cumsum(ks)[:-1]])
    for g in range(4):
        ms = np.sort(rs.choice(M, 24, replace=False))
        ns = np.sort(rs.choice(N, 24, replace=False))
        rows = slice(koff[g], koff[g] + ks[g])
        a_g = np.ascontiguousarray(w["a"][rows][:, ms])
        b_g = np.ascontiguousarray(w["b"][rows][:, ns])
        sa = oracle.pack_sf_ue8m0_k_grouped(w["sfa"][koff[g] // 128:(koff[g] + ks[g]) // 128][:, ms], 24, [ks[g]])
        sb = oracle.pack_sf_ue8m0_k_grouped(w["sfb"][koff[g] // 128:(koff[g] + ks[g]) // 128][:, ns], 24, [ks[g]])
        want = oracle.k_grouped_fp8_gemm_tn_contiguous(a_g, sa, b_g, sb, [ks[g]])[0]
        got = d[g].cpu().numpy()[np.ix_(ms, ns)]
        assert_close_f32(got, want, f"group {g}")
