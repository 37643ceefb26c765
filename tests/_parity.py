"""Shared helpers for the GPU parity tests: device upload and the tolerance check.

The tolerance is the one stated for the FP8 GEMM family's results: per element
|D - ref| <= 8e-3 * |ref| + 1e-3 * rms(ref), and globally
1 - 2 * sum(D * ref) / sum(D^2 + ref^2) <= 1e-4, where ref is the oracle's BF16 result and
rms is taken over the valid (computed) elements of the whole call.
"""
import numpy as np
import torch

import oracle

REL_TOL = 8e-3
RMS_TOL = 1e-3
GLOBAL_TOL = 1e-4


def to_dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_within_tolerance(d_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> dict:
    d = oracle.bf16_bits_to_float(d_bits).ravel()
    r = oracle.bf16_bits_to_float(ref_bits).ravel()
    assert np.all(np.isfinite(d)), f"{what}: non-finite values in the GPU result"
    if d.size == 0:
        return {}
    rms = float(np.sqrt(np.mean(r * r)))
    err = np.abs(d - r)
    bound = REL_TOL * np.abs(r) + RMS_TOL * rms
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {d.size} elements out of tolerance; first at flat "
                           f"{bad[:5]}: got {d[bad[:5]]}, want {r[bad[:5]]}, rms {rms}")
    den = float(np.sum(d * d + r * r))
    diff = 1.0 - 2.0 * float(np.sum(d * r)) / den if den > 0 else 0.0
    assert diff <= GLOBAL_TOL, f"{what}: global diff {diff}"
    return dict(max_rel=float(np.max(err / np.maximum(np.abs(r), 1e-30))), diff=diff,
                max_err_over_rms=float(np.max(err)) / max(rms, 1e-30))


def assert_close_f32(got: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    """The same per-element and global bounds, for FP32 results (ref: the oracle's FP32)."""
    d = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    assert np.all(np.isfinite(d)), f"{what}: non-finite values in the GPU result"
    if d.size == 0:
        return {}
    rms = float(np.sqrt(np.mean(r * r)))
    err = np.abs(d - r)
    bad = np.nonzero(err > REL_TOL * np.abs(r) + RMS_TOL * rms)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {d.size} elements out of tolerance; first at flat "
                           f"{bad[:5]}: got {d[bad[:5]]}, want {r[bad[:5]]}, rms {rms}")
    den = float(np.sum(d * d + r * r))
    diff = 1.0 - 2.0 * float(np.sum(d * r)) / den if den > 0 else 0.0
    assert diff <= GLOBAL_TOL, f"{what}: global diff {diff}"
    return dict(max_err_over_rms=float(np.max(err)) / max(rms, 1e-30), diff=diff)
