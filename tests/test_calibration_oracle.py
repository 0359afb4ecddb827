"""Pins of the rate / SNR calibration oracle (CPU only)."""
import math

import numpy as np
import pytest

import oracle as O
import oracle.calibration_oracle as C
from synthetic import gaussian_matrix


@pytest.fixture(scope="module")
def sample():
    return gaussian_matrix(4, 1024, 1.0, 77), O.splitmix64_signs(1, 1024)


def test_snr_definition_on_a_hand_case():
    W = np.array([[3.0, 4.0]])
    assert C.snr_db(W, np.array([[3.0, 3.0]])) == pytest.approx(10 * math.log10(25.0))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_closed_form_beta_reaches_the_target_snr(lattice, sample):
    """High-resolution formula (error per coordinate G V^(2/n) s^2 with the textbook G)
    against the measured SNR of the oracle quantizer at 20 and 26 dB."""
    W, d = sample
    for target in (20.0, 26.0):
        _, snr = C.rate_and_snr(W, lattice, 256, d, C.beta_for_snr(lattice, target))
        assert abs(snr - target) < 0.2, (lattice, target, snr)


def test_rate_decreases_with_beta(sample):
    W, d = sample
    rates = [C.rate_bits(W, "e8", 256, d, b) for b in (0.0625, 0.125, 0.25, 0.5, 1.0, 2.0)]
    assert all(a > b for a, b in zip(rates, rates[1:])), rates


def test_calibrated_scale_at_four_bits(sample):
    """E8 at 4.0 bps: the rate lands at (just under) the target and the SNR sits
    between the Gaussian rate-distortion bound 6.02 R dB and that bound minus
    the entropy-coded scalar gap (10 log10(pi e / 6) = 1.53 dB) minus the Rice
    code's overhead; E8 beats the scalar lattice Z at the same rate."""
    W, d = sample
    beta, bps, snr = C.calibrate_bps(W, "e8", 256, d, 4.0)
    assert 3.99 <= bps <= 4.0
    assert 6.02 * 4.0 - 2.5 < snr < 6.02 * 4.0, snr
    _, bps_z, snr_z = C.calibrate_bps(W, "z1", 256, d, 4.0)
    assert snr > snr_z
    # one bisection step further down in beta already exceeds the rate
    above = C.rate_bits(W, "e8", 256, d, float(np.float32(beta * 2 ** -(12 / 2 ** 24))))
    assert above >= bps * W.size
