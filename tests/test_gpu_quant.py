"""GPU per-token 1x128 quantisation against the oracle, through the C ABI.

Codes and packed scales are integers decided by floating point: both sides take the same
decision (an exact power-of-two scaling, then one round-to-nearest-even), so they are
compared bit for bit, padding words included.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu


def _bf16_values(x_bits):
    return oracle.bf16_bits_to_float(x_bits)


def run_quant(x_bits):
    G, M, K = x_bits.shape
    x = to_dev(x_bits.view(np.int16))
    q = torch.full((G, M, K), 0x5A, dtype=torch.uint8, device="cuda")            # junk: fully overwritten
    sf = torch.full((G,) + dg.packed_sf_shape(None, M, K), 0x13579BDF, dtype=torch.int32, device="cuda")
    dg.dg_quantize_fp8_1x128(x, q, sf)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy()


def check(x_bits, rows=None):
    q, sf = run_quant(x_bits)
    G, M, K = x_bits.shape
    for g in range(G):
        if rows is None:
            want_q, want_sf = oracle.quantize_fp8_1x128(_bf16_values(x_bits[g]))
            assert np.array_equal(q[g], want_q), f"codes of group {g}"
            assert np.array_equal(sf[g].view(np.uint32), want_sf.view(np.uint32)), f"scales of group {g}"
        else:
            # row-local operation: sampled rows, plus the padding words of the scale tensor
            want_q, want_sf = oracle.quantize_fp8_1x128(_bf16_values(x_bits[g, rows]))
            assert np.array_equal(q[g, rows], want_q)
            assert np.array_equal(sf[g][:, rows].view(np.uint32), want_sf[:, :len(rows)].view(np.uint32))
            assert np.all(sf[g][:, M:] == 0)


@pytest.mark.parametrize("G,M,K,wide", [
    (1, 1, 128, False),       # one row, one block: padding words for rows 1..3
    (1, 5, 384, True),        # Kb = 3: a partly filled packed word
    (1, 130, 1152, True),     # Kb = 9, ragged rows
    (3, 64, 2048, True),      # grouped (masked-layout A)
    (2, 257, 7168, False),    # Kb = 56
    (1, 8, 640, True),
])
def test_quantize_parity(G, M, K, wide):
    check(synth.make_activations(G, M, K, seed=M + K, wide=wide))


def test_quantize_ties_and_extremes():
    # Every BF16 magnitude pattern in one row set: all 2**15 positive encodings and their
    # negatives, in 1x128 blocks, so every rounding case (ties included) of every binade appears.
    allbits = np.arange(0x7F80, dtype=np.uint16)             # +0 .. largest finite
    x = np.concatenate([allbits, allbits | 0x8000])
    x = x[: x.size // 1024 * 1024]
    check(x.reshape(1, -1, 1024))                            # blocks of one binade each
    perm = synth.rng(1, "perm", 8).permutation(x.size)
    check(x[perm].reshape(1, -1, 1024))                      # blocks mixing all binades


def test_quantize_full_size_contiguous_activations():
    # The contiguous MoE workload's A before quantisation: 33152 x 7168 BF16, sampled rows.
    M, K = 33152, 7168
    x = synth.make_activations(1, M, K, seed=0)
    rows = np.sort(synth.rng(0, "perm", 7).choice(M, size=96, replace=False))
    check(x, rows=list(rows) + [M - 1])


def test_quantize_then_gemm_matches_oracle():
    # GPU quantisation feeding the GPU GEMM: compare with the oracle GEMM on the oracle's codes.
    M, N, K = 192, 512, 1536
    xa = synth.make_activations(1, M, K, seed=5)
    w = synth.make_dense(M, N, K, seed=6)
    q, sf = run_quant(xa)
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    d = torch.empty((M, N), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(q[0]), to_dev(sf[0]), to_dev(w["b"]), to_dev(sfb), d)
    dg.dg_check_device_error()
    want_q, want_sf = oracle.quantize_fp8_1x128(_bf16_values(xa[0]))
    assert_within_tolerance(bits(d), oracle.fp8_gemm_nt(want_q, want_sf, w["b"], sfb), "quantize -> gemm")
