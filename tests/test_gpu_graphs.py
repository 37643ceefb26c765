"""The grouped GEMMs read their group sizes on the device, so one CUDA-graph capture serves every
routing: capture once, change masked_m / ks / m_indices in place, replay, compare with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_close_f32, assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu


def test_masked_gemm_graph_replay_with_new_masks():
    G, max_m, N, K = 4, 256, 512, 1024
    w = synth.make_masked(G, max_m, N, K, seed=61, masked_m=[256, 1, 0, 129])
    sfa = oracle.pack_sf_ue8m0(w["sfa"], max_m, 1)
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)
    a, sa, b, sb = to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb)
    mm = to_dev(w["masked_m"])
    d = torch.full((G, max_m, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dg.dg_m_grouped_fp8_gemm_nt_masked(a, sa, b, sb, d, mm, stream=s)    # warm-up (plans, attributes)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dg.dg_m_grouped_fp8_gemm_nt_masked(a, sa, b, sb, d, mm, stream=s)
    for masks in ([256, 1, 0, 129], [0, 0, 255, 3], [17, 256, 256, 0]):
        d.fill_(synth.SENTINEL_BF16)
        mm.copy_(torch.tensor(masks, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        dg.dg_check_device_error()
        prior = np.full((G, max_m, N), synth.SENTINEL_BF16, np.uint16)
        want = oracle.m_grouped_fp8_gemm_nt_masked(w["a"], sfa, w["b"], sfb, np.array(masks), prior)
        got = bits(d)
        rows = np.arange(max_m)[None, :] < np.asarray(masks)[:, None]
        assert np.array_equal(got[~rows], want[~rows]), f"untouched rows, masks {masks}"
        assert_within_tolerance(got[rows], want[rows], f"graph replay masks {masks}")


def test_k_grouped_gemm_graph_replay_with_new_group_sizes():
    M, N = 256, 384
    ks0 = [256, 128, 384]
    w = synth.make_k_grouped(M, N, ks0, seed=62)
    sum_k = sum(ks0)
    a, b = to_dev(w["a"]), to_dev(w["b"])
    rows = dg.k_grouped_packed_sf_rows([sum_k, 0, 0]) + 3          # room for any split of sum_k
    sfa = torch.zeros((rows, M), dtype=torch.int32, device="cuda")
    sfb = torch.zeros((rows, N), dtype=torch.int32, device="cuda")
    ks = to_dev(np.asarray(ks0, np.int32))
    sfa_f, sfb_f = to_dev(w["sfa"]), to_dev(w["sfb"])
    d = torch.zeros((3, M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        dg.dg_pack_sf_ue8m0_k_grouped(sfa_f, sfa, ks, M, stream=s)
        dg.dg_pack_sf_ue8m0_k_grouped(sfb_f, sfb, ks, N, stream=s)
        dg.dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, ks, stream=s)

    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for split in ([256, 128, 384], [768, 0, 0], [128, 512, 128]):
        ks.copy_(torch.tensor(split, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        dg.dg_check_device_error()
        # the same tokens, regrouped: the oracle quantises per 128 rows, which the regrouping keeps
        sa = oracle.pack_sf_ue8m0_k_grouped(w["sfa"], M, split)
        sb = oracle.pack_sf_ue8m0_k_grouped(w["sfb"], N, split)
        want = oracle.k_grouped_fp8_gemm_tn_contiguous(w["a"], sa, w["b"], sb, split)
        assert_close_f32(d.cpu().numpy(), want, f"graph replay ks {split}")
