"""dg_pack_sf_ue8m0 on the GPU against the oracle's pack: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_02_gb300 as dg
from tests._parity import to_dev

pytestmark = pytest.mark.gpu


def _gpu_pack(sf: np.ndarray, mn: int, gran: int) -> np.ndarray:
    G = sf.shape[0]
    Kb = sf.shape[-1]
    out = torch.full(dg.packed_sf_shape(G, mn, Kb * 128), -1, dtype=torch.int32, device="cuda")
    dg.dg_pack_sf_ue8m0(to_dev(sf), out, mn, gran)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("G,MN,gran,Kb", [(1, 128, 1, 8), (1, 5, 1, 5), (2, 4096, 1, 56), (4, 130, 128, 9),
                                          (3, 7168, 128, 16), (1, 1, 1, 1), (2, 2112, 128, 56), (1, 33, 1, 3),
                                          (3, 257, 1, 17),     # partial last tile of 128 rows, odd word count
                                          (1, 70, 1, 400)])    # 100 words per row: 13 word tiles, the last partial
def test_pack_powers_of_two(G, MN, gran, Kb):
    rs = np.random.default_rng(G * 1000 + MN + Kb)
    MNb = -(-MN // gran)
    sf = np.ldexp(1.0, rs.integers(-127, 128, size=(G, MNb, Kb))).astype(np.float32)
    got = _gpu_pack(sf, MN, gran)
    want = oracle.pack_sf_ue8m0(sf, MN, gran)
    assert np.array_equal(got, want)


def test_pack_rounding_and_specials():
    rs = np.random.default_rng(5)
    G, MN, Kb = 2, 300, 12
    vals = (rs.standard_normal((G, MN, Kb)) * 10.0 ** rs.integers(-45, 39, (G, MN, Kb))).astype(np.float32)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, -1.0, 1e-45, 5.877472e-39, 8.8e-39,
                         1.1754944e-38, 1.7014118e38, 2.5e38, 3.4e38, 1.0, 0.75, 3.0], dtype=np.float32)
    flat = vals.reshape(-1)
    flat[:specials.size] = specials
    flat[-specials.size:] = specials
    got = _gpu_pack(vals, MN, 1)
    want = oracle.pack_sf_ue8m0(vals, MN, 1)
    assert np.array_equal(got, want)
