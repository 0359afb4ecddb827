"""GPU rate / SNR calibration against the CPU oracle."""
import numpy as np
import pytest

import oracle as O
import oracle.calibration_oracle as C
from synthetic import gaussian_matrix
from tests.gpu_util import cuda, to_dev

pytestmark = pytest.mark.gpu


def test_error_sums_match_numpy():
    torch, L = cuda()
    rng = np.random.default_rng(5)
    W = rng.standard_normal((37, 384)).astype(np.float32)
    Wh = (W + 0.01 * rng.standard_normal(W.shape)).astype(np.float32)
    sums = torch.empty(2, dtype=torch.float64, device="cuda")
    L.lq_error_sums(to_dev(torch, W), to_dev(torch, Wh), sums)
    torch.cuda.synchronize()
    got = sums.cpu().numpy()
    ref = [float((W.astype(np.float64) ** 2).sum()), float(((W.astype(np.float64) - Wh) ** 2).sum())]
    np.testing.assert_allclose(got, ref, rtol=1e-12)


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_calibrate_matches_oracle(lattice):
    """Same sample, same bisection: the GPU lands on the oracle's scale, rate and SNR."""
    torch, L = cuda()
    W = gaussian_matrix(4, 1024, 1.0, 77)
    d = O.splitmix64_signs(1, 1024)
    beta_o, bps_o, snr_o = C.calibrate_bps(W, lattice, 256, d, 4.0)
    ws = torch.empty(L.lq_calibrate_workspace_size(lattice, 4, 1024, 256), dtype=torch.uint8, device="cuda")
    beta, bps, snr = L.lq_calibrate_bps(lattice, 256, 4.0, to_dev(torch, W), 1, ws)
    assert abs(beta / beta_o - 1) < 1e-3, (beta, beta_o)
    assert abs(bps - bps_o) < 5e-3 and bps <= 4.0
    assert abs(snr - snr_o) < 0.05, (snr, snr_o)


def test_snr_grows_six_db_per_bit():
    """E8 on a 1024 x 4096 Gaussian sample at 3, 4 and 5 bps: each extra bit buys about
    6.02 dB (high-resolution rate-distortion slope)."""
    torch, L = cuda()
    from synthetic import torch_gaussian_matrix
    W = torch_gaussian_matrix(1024, 4096, 1.0, 3000, device="cuda")
    ws = torch.empty(L.lq_calibrate_workspace_size("e8", 1024, 4096, 256), dtype=torch.uint8, device="cuda")
    res = [L.lq_calibrate_bps("e8", 256, b, W, 0, ws) for b in (3.0, 4.0, 5.0)]
    for (beta, bps, snr), target in zip(res, (3.0, 4.0, 5.0)):
        assert target - 0.01 < bps <= target
    d1, d2 = res[1][2] - res[0][2], res[2][2] - res[1][2]
    assert 5.5 < d1 < 6.5 and 5.5 < d2 < 6.5, (d1, d2)
