"""Pins of the scale-format oracle (oracle/scale_formats.py) to facts outside it:
library float conversions, exact reconstructions of lattice points, powers of two."""
import numpy as np
import pytest

import oracle as O
from oracle import scale_formats as F


def test_bf16_rounding_matches_torch_and_hand_cases():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    # float32 inputs (no double rounding on the torch side): normal, tiny and exact ties
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),          # bf16 subnormals
        np.float32(1.0) + np.arange(-64, 64, dtype=np.float32) * np.float32(2.0 ** -9),  # every other a tie
        np.array([3.3895e38, 3.39e38, -0.0, 0.0], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = F.round_to_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    # hand cases: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3 2^-8 -> 1 + 2^-6
    np.testing.assert_array_equal(F.round_to_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)])),
                                  [1.0, 1 + 2 ** -6, -1.0])


def test_f16_rounding_matches_numpy_and_hand_cases():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 100.0,
        rng.standard_normal(2000) * 1e-6,                                 # fp16 subnormals
        1.0 + np.arange(-64, 64) * 2.0 ** -12,                            # every other a tie
        np.array([65504.0, 65519.0, 65520.0, 7e4, 2.0 ** -25, 3 * 2.0 ** -26])])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(F.round_to_f16(x), ref)
    np.testing.assert_array_equal(F.round_to_f16(np.array([65520.0, 2.0 ** -25])), [np.inf, 0.0])


def _lattice_rows(lattice, rows, cols, T, rng):
    """Rows that are permutations (of whole lattice blocks) of one base row of
    lattice points: every row has the same RMS, tiles inside a row differ."""
    n = O.LATTICE_DIM[lattice]
    mags = np.repeat(rng.uniform(0.5, 6.0, cols // T), T)             # tile-dependent magnitudes
    y = rng.standard_normal(cols) * mags
    base = O.nearest_point(lattice, y.reshape(-1, n)).reshape(-1, n)
    P = np.stack([base[rng.permutation(base.shape[0])].reshape(-1) for _ in range(rows)])
    return P


@pytest.mark.parametrize("lattice", O.LATTICES)
def test_row_bf16_recovers_lattice_points_exactly(lattice):
    """W = D H (s_r p) / sqrt(T) with lattice points p and bf16 scales s_r, beta =
    1 / RMS(p): the row format returns the codes 2p (A2: (2x, 2y/sqrt3)) and the
    scales s_r exactly; dequantize gives W back and the GEMV equals W x."""
    rng = np.random.default_rng(2)
    rows, cols, T = 6, 1024, 256
    P = _lattice_rows(lattice, rows, cols, T, rng)
    rms = np.sqrt(np.mean(P[0] ** 2))
    s = F.round_to_bf16(rng.uniform(0.001, 0.05, rows))
    d = O.splitmix64_signs(5, cols)
    W = O.inverse_rht_tiles(s[:, None] * P, d, T)
    q = F.quantize_formatted(W, lattice, T, d, 1.0 / rms, "row_bf16")
    n = O.LATTICE_DIM[lattice]
    want = O.point_to_codes(lattice, P.reshape(rows, -1, n)).reshape(rows, cols)
    np.testing.assert_array_equal(q.codes_wide, want)
    np.testing.assert_array_equal(q.scales, s)
    np.testing.assert_allclose(F.dequantize_formatted(q.codes, q.scales, "row_bf16", d, T, lattice), W,
                               rtol=0, atol=1e-14)
    x = rng.standard_normal((3, cols))
    np.testing.assert_allclose(F.gemv_formatted(q.codes, q.scales, "row_bf16", d, T, lattice, x), x @ W.T,
                               rtol=1e-12, atol=1e-14)
    assert not q.range_error and not q.nonfinite


@pytest.mark.parametrize("lattice", O.LATTICES)
def test_tile_f16_recovers_lattice_points_exactly(lattice):
    """Same construction with one fp16 scale per tile; every tile is a block
    permutation of one base tile, so one beta fits all tiles."""
    rng = np.random.default_rng(3)
    rows, cols, T = 5, 768, 128
    n = O.LATTICE_DIM[lattice]
    base = O.nearest_point(lattice, (rng.standard_normal(T) * 3.0).reshape(-1, n)).reshape(-1, n)
    P = np.stack([np.concatenate([base[rng.permutation(T // n)].reshape(-1) for _ in range(cols // T)])
                  for _ in range(rows)])
    rms = np.sqrt(np.mean(base.reshape(-1) ** 2))
    s = F.round_to_f16(rng.uniform(0.01, 20.0, (rows, cols // T)))
    d = O.splitmix64_signs(6, cols)
    W = O.inverse_rht_tiles(np.repeat(s, T, axis=1) * P, d, T)
    q = F.quantize_formatted(W, lattice, T, d, 1.0 / rms, "tile_f16")
    want = O.point_to_codes(lattice, P.reshape(rows, -1, n)).reshape(rows, cols)
    np.testing.assert_array_equal(q.codes_wide, want)
    np.testing.assert_array_equal(q.scales, s)
    np.testing.assert_allclose(F.dequantize_formatted(q.codes, q.scales, "tile_f16", d, T, lattice), W,
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("fmt", F.SCALE_FORMATS)
def test_power_of_two_scaling(fmt):
    """Multiplying W by 2^k multiplies every stored scale by 2^k and keeps the codes."""
    rng = np.random.default_rng(4)
    W = rng.standard_normal((9, 512)) * 0.02
    d = O.splitmix64_signs(7, 512)
    a = F.quantize_formatted(W, "e8", 256, d, 0.25, fmt)
    b = F.quantize_formatted(W * 8.0, "e8", 256, d, 0.25, fmt)
    np.testing.assert_array_equal(a.codes, b.codes)
    np.testing.assert_array_equal(a.scales * 8.0, b.scales)


def test_row_scale_is_beta_times_row_rms():
    """The row scale is beta times the RMS of the raw row (the tile Hadamards are
    orthonormal), rounded to bf16; a constant row c gives exactly bf16(beta |c|)."""
    rng = np.random.default_rng(5)
    W = rng.standard_normal((4, 2048)) * rng.uniform(0.01, 1.0, (4, 1))
    W[3] = -0.375
    d = O.splitmix64_signs(8, 2048)
    q = F.quantize_formatted(W, "d4", 512, d, 0.3, "row_bf16")
    np.testing.assert_allclose(q.scales_exact, 0.3 * np.sqrt(np.mean(W * W, axis=1)), rtol=1e-13)
    np.testing.assert_array_equal(q.scales, F.round_to_bf16(q.scales_exact))
    assert q.scales[3] == F.round_to_bf16(np.array([0.3 * 0.375]))[0]


def test_tile_f32_format_is_the_default_quantizer():
    rng = np.random.default_rng(6)
    W = rng.standard_normal((7, 1024)) * 0.02
    d = O.splitmix64_signs(9, 1024)
    a = F.quantize_formatted(W, "e8", 256, d, 0.25, "tile_f32")
    b = O.quantize(W, "e8", 256, d, 0.25)
    np.testing.assert_array_equal(a.codes, b.codes)
    np.testing.assert_array_equal(a.scales.astype(np.float32), b.scales)


def test_f16_overflow_is_a_range_error_and_nonfinite_rows_flag():
    rng = np.random.default_rng(7)
    W = rng.standard_normal((3, 256))
    W[1] *= 1e6                          # beta * RMS above the fp16 range
    d = O.splitmix64_signs(10, 256)
    q = F.quantize_formatted(W, "z1", 256, d, 0.25, "tile_f16")
    assert q.range_error and np.isinf(q.scales[1, 0])
    W2 = W.copy()
    W2[2, 5] = np.nan
    q2 = F.quantize_formatted(W2, "z1", 128, d, 0.25, "row_bf16")
    assert q2.nonfinite and np.all(q2.codes[2] == 0)
