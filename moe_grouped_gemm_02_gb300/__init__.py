"""GB300-native FP8 block-scaled GEMM (dense and M-grouped MoE): the Python binding.

A thin ctypes layer over libdg.so, whose C ABI is declared in include/dg.h.  The functions
below carry the same names as the C entry points and do argument marshalling only (tensor
shapes -> sizes, tensors -> device pointers, the current torch stream -> cudaStream_t);
every step of the computation runs in the library's CUDA kernels.  There is no fallback:
if libdg.so is missing or the device is unsupported, the calls raise.

Tensor conventions (all CUDA, contiguous):
  FP8 operands     torch.uint8 or torch.float8_e4m3fn
  packed scales    torch.int32, [G?][Kp][tma_aligned_size(rows)]
  outputs          torch.bfloat16 (or int16/uint16 views of the same bytes)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdg.so")

_STATUS = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_SHAPE", 3: "DG_ERR_ALIGNMENT",
           4: "DG_ERR_UNSUPPORTED_DEVICE", 5: "DG_ERR_CUDA", 6: "DG_ERR_TIMEOUT", 7: "DG_ERR_CONTRACT"}

EXPORTS = ("dg_fp8_gemm_nt", "dg_m_grouped_fp8_gemm_nt_contiguous", "dg_m_grouped_fp8_gemm_nt_masked",
           "dg_pack_sf_ue8m0", "dg_get_mk_alignment_for_contiguous_layout", "dg_get_tma_aligned_size",
           "dg_set_num_sms", "dg_get_num_sms", "dg_set_pdl", "dg_get_pdl", "dg_status_string",
           "dg_check_device_error", "dg_quantize_fp8_1x128", "dg_fp8_gemm",
           "dg_k_grouped_fp8_gemm_tn_contiguous", "dg_pack_sf_ue8m0_k_grouped", "dg_fp8_fp4_gemm_nt",
           "dg_m_grouped_fp8_fp4_gemm_nt_contiguous", "dg_m_grouped_fp8_fp4_gemm_nt_masked")

LAYOUTS = {"nt": 0, "nn": 1, "tn": 2, "tt": 3}


class DGError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {_STATUS.get(status, status)} ({status_string(status)})")


_lib = None


def load_library() -> ctypes.CDLL:
    """Loads libdg.so (built in-tree by moe_grouped_gemm_02_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m moe_grouped_gemm_02_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.dg_fp8_gemm_nt.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
    lib.dg_m_grouped_fp8_gemm_nt_contiguous.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.dg_m_grouped_fp8_gemm_nt_masked.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.dg_pack_sf_ue8m0.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp]
    lib.dg_quantize_fp8_1x128.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    lib.dg_fp8_gemm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.dg_k_grouped_fp8_gemm_tn_contiguous.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.dg_pack_sf_ue8m0_k_grouped.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    lib.dg_fp8_fp4_gemm_nt.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
    lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.dg_m_grouped_fp8_fp4_gemm_nt_masked.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    for name in ("dg_fp8_gemm_nt", "dg_m_grouped_fp8_gemm_nt_contiguous", "dg_m_grouped_fp8_gemm_nt_masked",
                 "dg_pack_sf_ue8m0", "dg_check_device_error", "dg_quantize_fp8_1x128", "dg_fp8_gemm",
                 "dg_k_grouped_fp8_gemm_tn_contiguous", "dg_pack_sf_ue8m0_k_grouped", "dg_fp8_fp4_gemm_nt",
                 "dg_m_grouped_fp8_fp4_gemm_nt_contiguous", "dg_m_grouped_fp8_fp4_gemm_nt_masked"):
        getattr(lib, name).restype = i32
    lib.dg_check_device_error.argtypes = [vp]
    lib.dg_get_mk_alignment_for_contiguous_layout.argtypes = []
    lib.dg_get_mk_alignment_for_contiguous_layout.restype = i32
    lib.dg_get_tma_aligned_size.argtypes = [i32, i32]
    lib.dg_get_tma_aligned_size.restype = i32
    lib.dg_set_num_sms.argtypes = [i32]
    lib.dg_set_num_sms.restype = None
    lib.dg_get_num_sms.argtypes = []
    lib.dg_get_num_sms.restype = i32
    lib.dg_set_pdl.argtypes = [i32]
    lib.dg_set_pdl.restype = None
    lib.dg_get_pdl.argtypes = []
    lib.dg_get_pdl.restype = i32
    lib.dg_status_string.argtypes = [i32]
    lib.dg_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().dg_status_string(int(status)).decode()


def _check(call: str, status: int) -> None:
    if status != 0:
        raise DGError(call, status)


# The pointer and stream arguments go to ctypes as plain integers (the argument types above
# convert them): a call's marshalling then costs a few microseconds, less than the decode-size
# GEMMs it launches.  The current stream comes from torch's raw accessor where it has one
# (torch.cuda.current_stream() builds a Stream object, ~3 us per call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _ptr(t: torch.Tensor, what: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream


def dg_get_mk_alignment_for_contiguous_layout() -> int:
    return load_library().dg_get_mk_alignment_for_contiguous_layout()


def dg_get_tma_aligned_size(mn: int, elem_bytes: int = 4) -> int:
    return load_library().dg_get_tma_aligned_size(int(mn), int(elem_bytes))


def dg_set_num_sms(n: int) -> None:
    load_library().dg_set_num_sms(int(n))


def dg_get_num_sms() -> int:
    return load_library().dg_get_num_sms()


def dg_set_pdl(enable: bool) -> None:
    load_library().dg_set_pdl(1 if enable else 0)


def dg_get_pdl() -> bool:
    return bool(load_library().dg_get_pdl())


def dg_check_device_error(stream=None) -> None:
    _check("dg_check_device_error", load_library().dg_check_device_error(_stream(stream)))


def dg_fp8_gemm_nt(a, sfa, b, sfb, d, stream=None) -> None:
    """d[M, N] = a[M, K] @ b[N, K]^T with packed UE8M0 scales sfa [Kp][al4(M)], sfb [Kp][al4(N)]."""
    M, K = a.shape
    N = b.shape[0]
    _check("dg_fp8_gemm_nt", load_library().dg_fp8_gemm_nt(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"), M, N, K, _stream(stream)))


def dg_fp8_gemm(a, sfa, b, sfb, d, layout: str = "nt", c=None, stream=None) -> None:
    """d = c + a @ b^T in layout 'nt', 'nn', 'tn' or 'tt' (A 'n': [M, K], 't': [K, M];
    B 't': [N, K], 'n': [K, N]); d BF16 (int16/bfloat16 storage) or float32, c float32 or None."""
    a_t, b_n = layout[0] == "t", layout[1] == "n"
    K, M = a.shape if a_t else a.shape[::-1]
    N = b.shape[1] if b_n else b.shape[0]
    out_f32 = 1 if d.dtype == torch.float32 else 0
    cp = None if c is None else _ptr(c, "c")
    _check("dg_fp8_gemm", load_library().dg_fp8_gemm(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), cp, _ptr(d, "d"), M, N, K,
        LAYOUTS[layout], out_f32, _stream(stream)))


def dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, d, ks, c=None, stream=None) -> None:
    """d[g] = c[g] + a_g^T @ b_g for the K row ranges of ks (device int32 [G]); a [sum_K, M],
    b [sum_K, N], d and c float32 [G, M, N]."""
    sum_K, M = a.shape
    N = b.shape[1]
    G = ks.shape[0]
    cp = None if c is None else _ptr(c, "c")
    _check("dg_k_grouped_fp8_gemm_tn_contiguous", load_library().dg_k_grouped_fp8_gemm_tn_contiguous(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), cp, _ptr(d, "d"), _ptr(ks, "ks"),
        G, M, N, sum_K, _stream(stream)))


def dg_pack_sf_ue8m0_k_grouped(sf, out, ks, mn: int, stream=None) -> None:
    """Packs float32 scales sf [sum_K/128][mn] per group (ks: device int32 [G]) into
    out int32 [sum_g ceil(ks[g]/512)][al4(mn)]."""
    _check("dg_pack_sf_ue8m0_k_grouped", load_library().dg_pack_sf_ue8m0_k_grouped(
        _ptr(sf, "sf"), _ptr(out, "out"), _ptr(ks, "ks"), ks.shape[0], int(mn), sf.shape[0] * 128,
        _stream(stream)))


def k_grouped_packed_sf_rows(ks) -> int:
    """Rows of a K-grouped packed scale tensor: sum over groups of ceil(ks[g] / 512)."""
    return int(sum((int(k) // 128 + 3) // 4 for k in ks))


def dg_fp8_fp4_gemm_nt(a, sfa, b, sfb, d, stream=None) -> None:
    """d[M, N] = a[M, K] (E4M3) @ b^T, b E2M1 packed [N, K/2] (element 2i in the low nibble)."""
    M, K = a.shape
    N = b.shape[0]
    _check("dg_fp8_fp4_gemm_nt", load_library().dg_fp8_fp4_gemm_nt(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"), M, N, K, _stream(stream)))


def dg_m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, d, m_indices, stream=None) -> None:
    """The contiguous-layout grouped GEMM with E2M1 experts b [G, N, K/2]."""
    M_sum, K = a.shape
    G, N, _ = b.shape
    _check("dg_m_grouped_fp8_fp4_gemm_nt_contiguous", load_library().dg_m_grouped_fp8_fp4_gemm_nt_contiguous(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"),
        _ptr(m_indices, "m_indices"), M_sum, N, K, G, _stream(stream)))


def dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, stream=None) -> None:
    """The masked-layout grouped GEMM with E2M1 experts b [G, N, K/2]."""
    G, max_m, K = a.shape
    N = b.shape[1]
    _check("dg_m_grouped_fp8_fp4_gemm_nt_masked", load_library().dg_m_grouped_fp8_fp4_gemm_nt_masked(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"),
        _ptr(masked_m, "masked_m"), G, max_m, N, K, _stream(stream)))


def dg_m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, d, m_indices, stream=None) -> None:
    """d[M_sum, N]: row m = a[m] @ b[m_indices[m]]^T, +0.0 where m_indices[m] == -1."""
    M_sum, K = a.shape
    G, N, _ = b.shape
    _check("dg_m_grouped_fp8_gemm_nt_contiguous", load_library().dg_m_grouped_fp8_gemm_nt_contiguous(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"),
        _ptr(m_indices, "m_indices"), M_sum, N, K, G, _stream(stream)))


def dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, stream=None) -> None:
    """d[g, m] = a[g, m] @ b[g]^T for m < masked_m[g] (device tensor); other rows untouched."""
    G, max_m, K = a.shape
    N = b.shape[1]
    _check("dg_m_grouped_fp8_gemm_nt_masked", load_library().dg_m_grouped_fp8_gemm_nt_masked(
        _ptr(a, "a"), _ptr(sfa, "sfa"), _ptr(b, "b"), _ptr(sfb, "sfb"), _ptr(d, "d"),
        _ptr(masked_m, "masked_m"), G, max_m, N, K, _stream(stream)))


def dg_pack_sf_ue8m0(sf, out, mn: int, gran_mn: int, stream=None) -> None:
    """Packs float32 scales sf [G?][ceil(mn/gran_mn)][Kb] into out int32 [G?][Kp][al4(mn)]."""
    G = sf.shape[0] if sf.dim() == 3 else 1
    Kb = sf.shape[-1]
    _check("dg_pack_sf_ue8m0", load_library().dg_pack_sf_ue8m0(
        _ptr(sf, "sf"), _ptr(out, "out"), G, int(mn), Kb * 128, int(gran_mn), 128, _stream(stream)))


def dg_quantize_fp8_1x128(x, q, sf, stream=None) -> None:
    """Quantises bf16 x [G?][M][K] into e4m3 codes q (same shape, uint8) and packed scales
    sf int32 [G?][Kp][al4(M)]."""
    G = x.shape[0] if x.dim() == 3 else 1
    M, K = x.shape[-2], x.shape[-1]
    _check("dg_quantize_fp8_1x128", load_library().dg_quantize_fp8_1x128(
        _ptr(x, "x"), _ptr(q, "q"), _ptr(sf, "sf"), G, M, K, _stream(stream)))


def packed_sf_shape(groups: int | None, mn: int, K: int) -> tuple:
    """Shape of a packed scale tensor for `mn` rows and K (helper for allocating outputs)."""
    kp = (K // 128 + 3) // 4
    al = (mn + 3) // 4 * 4
    return (kp, al) if groups is None else (groups, kp, al)
