"""GPU parity of dg_fp8_gemm: the NT, NN, TN and TT storage layouts, BF16 or FP32 output, and
FP32 accumulation D = C + A @ B^T (C separate or in place), against the oracle."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_close_f32, assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu

LAYOUTS = ["nt", "nn", "tn", "tt"]


def _stored(w, layout):
    a = w["a"] if layout[0] == "n" else np.ascontiguousarray(w["a"].T)
    b = w["b"] if layout[1] == "t" else np.ascontiguousarray(w["b"].T)
    return a, b


def run(w, layout, out="bf16", c=None, in_place=False):
    M, N = w["M"], w["N"]
    sfa = oracle.pack_sf_ue8m0(w["sfa"], M, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], N, 128)[0]
    a, b = _stored(w, layout)
    if out == "bf16":
        d = torch.full((M, N), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    else:
        d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    cd = None
    if c is not None:
        cd = to_dev(c)
        if in_place:
            d.copy_(cd)
            cd = d
    dg.dg_fp8_gemm(to_dev(a), to_dev(sfa), to_dev(b), to_dev(sfb), d, layout=layout, c=cd)
    dg.dg_check_device_error()
    got = bits(d) if out == "bf16" else d.cpu().numpy()
    want = oracle.fp8_gemm(a, sfa, b, sfb, layout=layout, c=c, out=out)
    return got, want


def check(got, want, out, what):
    if out == "bf16":
        assert_within_tolerance(got, want, what)
    else:
        assert_close_f32(got, want, what)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [
    (128, 512, 1024),
    (256, 2112, 512),     # N tail inside the last 256-column tile
    (64, 256, 384),       # half an M tile
    (384, 96, 640),       # N below one 128-column box, Kb = 5
])
def test_layouts_bf16(layout, M, N, K):
    w = synth.make_dense(M, N, K, seed=M + 3 * N + K)
    got, want = run(w, layout)
    check(got, want, "bf16", f"{layout} {M}x{N}x{K}")


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("with_c", [False, True])
def test_layouts_f32_accumulate(layout, with_c):
    M, N, K = 256, 768, 1536
    w = synth.make_dense(M, N, K, seed=71)
    c = synth.normal((M, N), 71, "d_fill", std=3.0) if with_c else None
    got, want = run(w, layout, out="f32", c=c)
    check(got, want, "f32", f"{layout} C={with_c}")


def test_accumulate_in_place():
    # D = D + A @ B^T with C and D the same buffer (the weight-gradient accumulation pattern)
    M, N, K = 192, 640, 1024
    w = synth.make_dense(M, N, K, seed=72)
    c = synth.normal((M, N), 72, "d_fill", std=5.0)
    for layout in ("nt", "tn"):
        got, want = run(w, layout, out="f32", c=c, in_place=True)
        check(got, want, "f32", f"in place {layout}")


def test_nt_bf16_equals_dg_fp8_gemm_nt_bit_exact():
    w = synth.make_dense(256, 1024, 1536, seed=73)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], 256, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], 1024, 128)[0]
    d0 = torch.empty((256, 1024), dtype=torch.int16, device="cuda")
    d1 = torch.empty_like(d0)
    args = (to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb))
    dg.dg_fp8_gemm_nt(*args, d0)
    dg.dg_fp8_gemm(*args, d1, layout="nt")
    assert torch.equal(d0, d1)


@pytest.mark.parametrize("cfg", ["config_bn128_s6_a2", "config_bn128_s5_k2", "config_bn192_s3_m2"])
def test_layouts_agree_bit_exact(cfg, monkeypatch):
    # Under one plan the four layouts compute the same sums in the same order: identical bits.
    # (The planner may pick different plans for different layouts, and plans differ in the
    # order in which they add the K steps, so the plan is pinned.)
    monkeypatch.setenv("DG_FORCE_CONFIG", cfg)
    monkeypatch.setenv("DG_FORCE_SPLIT", "1")
    w = synth.make_dense(256, 512, 1024, seed=74)
    outs = [run(w, lay, out="f32")[0] for lay in LAYOUTS]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


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


@pytest.mark.parametrize("cfg,split,layout", [
    ("config_bn256_s4_a1", None, "nn"),
    ("config_bn128_s6_a2", None, "tn"),
    ("config_bn128_s4_a2", 2, "nn"),
    ("config_bn128_s4_a2", 4, "tn"),
    ("config_bn64_s8_a2", 2, "tt"),
    ("config_bn224_s3_m2", None, "tt"),     # 256-row tiles with an MN-major A
    ("config_bn192_s3_m2", None, "tt"),
    ("config_bn64_s8_a2", 8, "tt"),
    ("config_bn208_s3_m2", None, "tn"),     # 208 columns: a 16-column epilogue tail, 224-column accumulator stride
    ("config_bn128_s5_k2", 4, "nn"),        # two issuers splitting K, two accumulators added
    ("config_bn192_s5_k2", None, "tt"),
])
def test_forced_plans_with_layouts(forced, cfg, split, layout):
    forced(cfg, split)
    M, N, K = 256, 1024, 4096
    w = synth.make_dense(M, N, K, seed=75)
    c = synth.normal((M, N), 75, "d_fill")
    got, want = run(w, layout, out="f32", c=c)
    check(got, want, "f32", f"{cfg} split={split} {layout}")
    got, want = run(w, layout)
    check(got, want, "bf16", f"{cfg} split={split} {layout} bf16")
