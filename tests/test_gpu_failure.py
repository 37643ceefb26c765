"""Failure detection on the GPU without a fault: a barrier wait that runs out.

The test hook DG_DEBUG_DROP_LOAD makes the GEMM's producer skip one load stage, so the stage's
barrier is never completed; DG_TIMEOUT_MS bounds the wait.  The kernel must record the timeout
in its device error word, leave every loop, free its tensor memory and return: the host sees
DG_ERR_TIMEOUT from dg_check_device_error, and the next call on the same context is correct.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import assert_within_tolerance, bits, to_dev

pytestmark = pytest.mark.gpu


def _run(w, sfa, sfb):
    d = torch.empty((w["M"], w["N"]), dtype=torch.int16, device="cuda")
    dg.dg_fp8_gemm_nt(to_dev(w["a"]), to_dev(sfa), to_dev(w["b"]), to_dev(sfb), d)
    return d


@pytest.mark.parametrize("split", [1, 2])
def test_timeout_reported_and_context_survives(split, monkeypatch):
    w = synth.make_dense(256, 512, 2048, seed=31)
    sfa = oracle.pack_sf_ue8m0(w["sfa"], 256, 1)[0]
    sfb = oracle.pack_sf_ue8m0(w["sfb"], 512, 128)[0]
    dg.dg_check_device_error()                       # start from a clean error word
    monkeypatch.setenv("DG_FORCE_SPLIT", str(split))
    monkeypatch.setenv("DG_TIMEOUT_MS", "50")
    monkeypatch.setenv("DG_DEBUG_DROP_LOAD", "2")
    _run(w, sfa, sfb)
    with pytest.raises(dg.DGError) as exc:
        dg.dg_check_device_error()
    assert exc.value.status == 6                     # DG_ERR_TIMEOUT
    dg.dg_check_device_error()                       # the word was cleared
    monkeypatch.delenv("DG_DEBUG_DROP_LOAD")
    d = _run(w, sfa, sfb)
    dg.dg_check_device_error()
    assert_within_tolerance(bits(d), oracle.fp8_gemm_nt(w["a"], sfa, w["b"], sfb), "after timeout")
