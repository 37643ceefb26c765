"""The C-ABI library: it builds, loads, exports every entry point include/dg.h declares,
and its host-side argument checks return the documented codes.  No compute call is made
(the pointers below are never dereferenced: every case fails validation first)."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_02_gb300 as dg
from moe_grouped_gemm_02_gb300 import build as dg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dg_build.build()
    return dg.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "dg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "dg_fp8_gemm_nt" in names and "dg_pack_sf_ue8m0" in names
    for n in names:
        assert hasattr(lib, n), f"{n} is declared in dg.h but not exported"
    assert set(dg.EXPORTS) == set(names)


def test_helpers(lib):
    assert lib.dg_get_mk_alignment_for_contiguous_layout() == 128
    assert [lib.dg_get_tma_aligned_size(n, 4) for n in (1, 4, 5, 2112)] == [4, 4, 8, 2112]
    assert lib.dg_get_tma_aligned_size(3, 1) == 16
    assert lib.dg_get_tma_aligned_size(3, 3) == -1
    assert lib.dg_status_string(0) == b"ok"
    assert b"timed out" in lib.dg_status_string(6)


P = ctypes.c_void_p
GOOD = P(0x10000)        # 16-byte aligned fake addresses, never dereferenced
ODD = P(0x10008)


def test_dense_validation(lib):
    f = lib.dg_fp8_gemm_nt
    assert f(None, GOOD, GOOD, GOOD, GOOD, 128, 512, 1024, None) == 1       # null pointer
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, -1, 512, 1024, None) == 1        # negative M
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 128, 0, 1024, None) == 1         # N == 0
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 128, 512, 1000, None) == 2       # K % 128
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 128, 500, 1024, None) == 2       # N % 8
    assert f(GOOD, GOOD, GOOD, GOOD, ODD, 128, 512, 1024, None) == 3        # misaligned D
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 512, 1024, None) == 0         # empty: no-op


def test_grouped_validation(lib):
    c = lib.dg_m_grouped_fp8_gemm_nt_contiguous
    assert c(GOOD, GOOD, GOOD, GOOD, GOOD, None, 256, 512, 1024, 4, None) == 1    # no m_indices
    assert c(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 200, 512, 1024, 4, None) == 2    # M_sum % 128
    assert c(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 256, 512, 1024, 0, None) == 1    # G == 0
    assert c(GOOD, ODD, GOOD, GOOD, GOOD, GOOD, 256, 512, 1024, 4, None) == 3
    assert c(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 0, 512, 1024, 4, None) == 0      # empty
    m = lib.dg_m_grouped_fp8_gemm_nt_masked
    assert m(GOOD, GOOD, GOOD, GOOD, GOOD, None, 4, 256, 512, 1024, None) == 1
    assert m(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 5000, 256, 512, 1024, None) == 2  # too many groups
    assert m(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 4, 256, 512, 1100, None) == 2
    assert m(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 4, 0, 512, 1024, None) == 0      # empty


def test_pack_validation(lib):
    f = lib.dg_pack_sf_ue8m0
    assert f(GOOD, GOOD, 1, 64, 1024, 2, 128, None) == 1      # gran_mn must be 1 or 128
    assert f(GOOD, GOOD, 1, 64, 1024, 1, 64, None) == 1       # gran_k must be 128
    assert f(GOOD, GOOD, 1, 64, 1000, 1, 128, None) == 2
    assert f(GOOD, ODD, 1, 64, 1024, 1, 128, None) == 3
    assert f(GOOD, GOOD, 1, 0, 1024, 1, 128, None) == 0


def test_quantize_validation(lib):
    f = lib.dg_quantize_fp8_1x128
    assert f(None, GOOD, GOOD, 1, 64, 1024, None) == 1        # null input
    assert f(GOOD, GOOD, GOOD, 0, 64, 1024, None) == 1        # G == 0
    assert f(GOOD, GOOD, GOOD, 1, 64, 1000, None) == 2        # K % 128
    assert f(GOOD, GOOD, ODD, 1, 64, 1024, None) == 3         # misaligned scales
    assert f(GOOD, GOOD, GOOD, 1, 0, 1024, None) == 0         # empty: no-op


def test_fp4_validation(lib):
    f = lib.dg_fp8_fp4_gemm_nt
    ODD16 = P(0x10010)       # 16-byte but not 32-byte aligned
    assert f(GOOD, GOOD, ODD16, GOOD, GOOD, 128, 512, 1024, None) == 3
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 128, 512, 1000, None) == 2
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, 0, 512, 1024, None) == 0
    c = lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous
    assert c(GOOD, GOOD, ODD16, GOOD, GOOD, GOOD, 256, 512, 1024, 4, None) == 3
    m = lib.dg_m_grouped_fp8_fp4_gemm_nt_masked
    assert m(GOOD, GOOD, GOOD, GOOD, GOOD, None, 4, 256, 512, 1024, None) == 1


def test_layout_gemm_validation(lib):
    f = lib.dg_fp8_gemm
    F32, BF16 = 1, 0
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, 128, 512, 1024, 4, BF16, None) == 1     # no such layout
    assert f(GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 128, 512, 1024, 0, BF16, None) == 1     # C needs FP32 D
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, 128, 512, 1024, 0, 2, None) == 1        # out flag 0/1
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, 120, 512, 1024, 2, F32, None) == 2     # TN: M % 16
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, 128, 520, 1024, 1, F32, None) == 2     # NN: N % 16
    assert f(GOOD, GOOD, GOOD, GOOD, ODD, GOOD, 128, 512, 1024, 0, F32, None) == 3      # misaligned C
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, 0, 512, 1024, 3, F32, None) == 0       # empty


def test_k_grouped_validation(lib):
    f = lib.dg_k_grouped_fp8_gemm_tn_contiguous
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, None, 4, 256, 512, 1024, None) == 1   # no ks
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, 0, 256, 512, 1024, None) == 1   # G == 0
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, 4, 250, 512, 1024, None) == 2   # M % 16
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, 4, 256, 512, 1000, None) == 2   # sum_K % 128
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, 5000, 256, 512, 1024, None) == 2  # too many groups
    assert f(GOOD, GOOD, GOOD, GOOD, ODD, GOOD, GOOD, 4, 256, 512, 1024, None) == 3    # misaligned C
    assert f(GOOD, GOOD, GOOD, GOOD, None, GOOD, GOOD, 4, 0, 512, 1024, None) == 0     # empty
    p = lib.dg_pack_sf_ue8m0_k_grouped
    assert p(GOOD, GOOD, None, 4, 256, 1024, None) == 1                                 # no ks
    assert p(GOOD, GOOD, GOOD, 4, 256, 1000, None) == 2                                 # sum_K % 128
    assert p(GOOD, ODD, GOOD, 4, 256, 1024, None) == 3                                  # misaligned out
    assert p(GOOD, GOOD, GOOD, 4, 0, 1024, None) == 0                                   # empty
