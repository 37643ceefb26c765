"""Back-to-back launches with programmatic dependent launch, as a decode step runs them.

The benchmark's back-to-back figures capture the calls in one CUDA graph, where each kernel may
start while the one before it finishes (it prefetches and sets up, then waits for that kernel
before touching global memory).  Two checks of that launch configuration:

* a dependent chain quantise -> GEMM -> quantise -> GEMM -> quantise -> GEMM over the decode
  shapes 64x4096x7168, 64x7168x4096 and 64x2112x7168 (split-K clusters and plain grids), each
  kernel reading what the one before it wrote.  Every intermediate buffer holds junk when the
  graph is replayed (once), so a read that ran ahead of its producer would see junk.  Each
  stage is checked against the oracle on the GPU's own input to that stage: codes and packed
  scales bit for bit, GEMM outputs within the tolerance;
* the decode stream: one GEMM shape over distinct weights back to back, each launch writing
  its own output, every output against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu

JUNK_BF16 = 0x7FC1   # a NaN pattern: any read of it would poison the sums


def _weights(M, N, K, seed):
    w = synth.make_dense(M, N, K, seed=seed, b_std=0.02)
    return w["b"], oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]


def _capture(fn, s):
    with torch.cuda.stream(s):
        fn()                                   # eager warm-up: plans, kernel attributes
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


def test_dependent_chain_in_one_graph():
    assert dg.dg_get_pdl(), "the library launches with programmatic dependent launch by default"
    M = 64
    stages = [(4096, 7168, 101), (7168, 4096, 102), (2112, 7168, 103)]   # (N, K, seed)
    x0 = synth.make_activations(1, M, 7168, seed=100)[0]
    x0_d = to_dev(x0.view(np.int16))
    bufs = []
    for N, K, seed in stages:
        b, sfb = _weights(M, N, K, seed)
        bufs.append(dict(N=N, K=K, b=b, sfb=sfb, b_d=to_dev(b), sfb_d=to_dev(sfb),
                         q=torch.empty((M, K), dtype=torch.uint8, device="cuda"),
                         sf=torch.empty(dg.packed_sf_shape(None, M, K), dtype=torch.int32, device="cuda"),
                         d=torch.empty((M, N), dtype=torch.int16, device="cuda")))
    s = torch.cuda.Stream()

    def chain():
        x = x0_d
        for st in bufs:
            dg.dg_quantize_fp8_1x128(x, st["q"], st["sf"], stream=s)
            dg.dg_fp8_gemm_nt(st["q"], st["sf"], st["b_d"], st["sfb_d"], st["d"], stream=s)
            x = st["d"]

    g = _capture(chain, s)
    for st in bufs:
        st["q"].fill_(0x5A)
        st["sf"].fill_(0x13579BDF)
        st["d"].fill_(JUNK_BF16)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    dg.dg_check_device_error()

    x_bits = x0
    for i, st in enumerate(bufs):
        want_q, want_sf = oracle.quantize_fp8_1x128(oracle.bf16_bits_to_float(x_bits))
        q = st["q"].cpu().numpy()
        sf = st["sf"].cpu().numpy()
        assert np.array_equal(q, want_q), f"stage {i}: codes"
        assert np.array_equal(sf.view(np.uint32), want_sf.view(np.uint32)), f"stage {i}: packed scales"
        got = bits(st["d"])
        assert_within_tolerance(got, oracle.fp8_gemm_nt(q, sf, st["b"], st["sfb"]),
                                f"stage {i}: {M}x{st['N']}x{st['K']}")
        x_bits = got


@pytest.mark.parametrize("shape", [(64, 2112, 7168), (128, 7168, 2048)])
def test_decode_stream_in_one_graph(shape):
    M, N, K = shape
    copies = 3
    w = synth.make_dense(M, N, K, seed=110, a_outliers=True, b_std=0.02)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    a_d, sfa_d = to_dev(w["a"]), to_dev(sfa)
    ws = [_weights(M, N, K, 111 + i) for i in range(copies)]
    wd = [(to_dev(b), to_dev(sfb)) for b, sfb in ws]
    ds = [torch.empty((M, N), dtype=torch.int16, device="cuda") for _ in range(copies)]
    s = torch.cuda.Stream()

    def stream():
        for i in range(copies):
            dg.dg_fp8_gemm_nt(a_d, sfa_d, wd[i][0], wd[i][1], ds[i], stream=s)

    g = _capture(stream, s)
    for d in ds:
        d.fill_(JUNK_BF16)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    dg.dg_check_device_error()
    for i, (b, sfb) in enumerate(ws):
        assert_within_tolerance(bits(ds[i]), oracle.fp8_gemm_nt(w["a"], sfa, b, sfb), f"{shape} launch {i}")
