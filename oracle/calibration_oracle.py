"""Plain CPU oracle of the rate / SNR calibration of the lattice quantizer.

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.

Source: HyperQuant (github release page of moonmath-ai/HyperQuant), usage
section and "bps" table: the quantizer runs on a continuous bits-per-scalar
axis; rates (bps) are related to the SNRs they reach by measurement, and a
lattice scale ("alpha") is set from a target SNR.  The pages give the
calls, not the procedure; the readings taken here (also in the design notes):

* SNR of a quantized matrix: 10 log10(sum w^2 / sum (w - w^)^2), in dB.
* Rate: bits per weight of the bit-stripped Rice stream (``rice_oracle``).
* Scale for a target SNR, closed form in the high-resolution regime: the error
  per coordinate is G V^(2/n) s^2 with s = beta * RMS (G the normalised second
  moment, V the covolume of the lattice at its native scale; Conway & Sloane
  ch. 2 and 21), so beta = sqrt(10^(-SNR/10) / (G V^(2/n))).
* Scale for a target rate: bisection on log2(beta) over [-8, 4], 24 halvings;
  the rate decreases as beta grows; the answer is the upper end of the final
  bracket (rate <= target), reported with its rate and SNR.  A probe whose
  codes leave int8 counts as above the target (the scale is too fine for the
  code range).
"""
from __future__ import annotations

import math

import numpy as np

from . import lattice_oracle as LO
from . import rice_oracle as R

# Conway & Sloane, table 2.3 (normalised second moments) and the native scales
# used by the quantizer (E8 and D4 with minimal norm^2 2, A2 with minimal
# distance 1, Z with spacing 1).
G_TEXTBOOK = {"e8": 929.0 / 12960.0, "d4": 0.0766032, "a2": 5.0 / (36.0 * math.sqrt(3.0)), "z1": 1.0 / 12.0}

LOG2_BETA_LO, LOG2_BETA_HI, BISECT_STEPS = -8.0, 4.0, 24


def snr_db(W: np.ndarray, W_hat: np.ndarray) -> float:
    W = np.asarray(W, dtype=np.float64)
    err = W - np.asarray(W_hat, dtype=np.float64)
    return 10.0 * math.log10(float((W * W).sum()) / float((err * err).sum()))


def beta_for_snr(lattice: str, snr: float) -> float:
    n = LO.LATTICE_DIM[lattice]
    return math.sqrt(10.0 ** (-snr / 10.0) / (G_TEXTBOOK[lattice] * LO.covolume(lattice) ** (2.0 / n)))


def rate_and_snr(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, beta: float):
    """(bits per weight of the Rice stream, SNR in dB) of W quantized at beta."""
    q = LO.quantize(W, lattice, T, signs, beta)
    _, _, total = R.encode(q.codes, lattice, T)
    W_hat = LO.dequantize(q.codes, q.scales, signs, T, lattice)
    return total / float(W.size), snr_db(W, W_hat)


def rate_bits(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, beta: float):
    """Bits of the Rice stream at beta, or None when a code leaves int8."""
    q = LO.quantize(W, lattice, T, signs, beta)
    if q.range_error:
        return None
    return R.encode(q.codes, lattice, T)[2]


def calibrate_bps(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, target_bps: float):
    """beta whose Rice rate on W is at most target_bps, by bisection on log2(beta).

    Returns (beta, bps, snr_db)."""
    lo, hi = LOG2_BETA_LO, LOG2_BETA_HI
    target_bits = target_bps * W.size
    for _ in range(BISECT_STEPS):
        mid = 0.5 * (lo + hi)
        bits = rate_bits(W, lattice, T, signs, float(np.float32(2.0 ** mid)))
        if bits is None or bits > target_bits:
            lo = mid
        else:
            hi = mid
    beta = float(np.float32(2.0 ** hi))
    bps, snr = rate_and_snr(W, lattice, T, signs, beta)
    return beta, bps, snr
