"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, textbook lattice constants, library routines, brute force, figures
printed on the HyperQuant page, and cases worked by hand (tests/golden/)."""
import json
import os

import numpy as np
import pytest
import scipy.linalg

import oracle as O
from synthetic import gaussian_matrix, gaussian_vectors, small_fp32_case


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- a1 signs
def test_signs_balanced_and_deterministic():
    C = 14336
    d = O.splitmix64_signs(7, C)
    assert d.dtype == np.int8 and set(np.unique(d)) == {-1, 1}
    assert abs(d.astype(np.float64).mean()) < 4.0 / np.sqrt(C)
    assert np.array_equal(d, O.splitmix64_signs(7, C))
    assert not np.array_equal(d, O.splitmix64_signs(8, C))
    # a prefix does not depend on the requested length
    assert np.array_equal(O.splitmix64_signs(7, 100), d[:100])


def test_splitmix_output_bits_balanced():
    outs = np.array(O.splitmix64(123, 4096), dtype=np.uint64)
    assert len(set(outs.tolist())) == 4096
    for bit in (0, 17, 31, 32, 63):
        frac = float(((outs >> np.uint64(bit)) & np.uint64(1)).mean())
        assert abs(frac - 0.5) < 4.0 / np.sqrt(4096)


# ---------------------------------------------------------------- a3 RHT
@pytest.mark.parametrize("T", [2, 8, 128, 256, 512])
def test_hadamard_matches_library_and_is_orthogonal(T):
    H = O.hadamard_matrix(T)
    assert np.array_equal(H, scipy.linalg.hadamard(T).astype(np.float64))
    assert np.array_equal(H @ H.T, T * np.eye(T))


def test_rht_orthonormal_and_identity():
    rng = np.random.default_rng(1)
    T, C = 256, 1024
    W = rng.standard_normal((5, C))
    x = rng.standard_normal((3, C))
    d = O.splitmix64_signs(3, C)
    Wt = O.rht_tiles(W, d, T)
    xt = O.rht_activations(x, d, T)
    # per-tile norms preserved
    for t in range(C // T):
        sl = slice(t * T, (t + 1) * T)
        np.testing.assert_allclose(np.linalg.norm(Wt[:, sl], axis=1),
                                   np.linalg.norm(W[:, sl], axis=1), rtol=1e-12)
    # rotated inner products equal the plain product: sum_t (H D w_t).(H D x_t)/T = w.x
    np.testing.assert_allclose(Wt @ xt.T, W @ x.T, rtol=1e-11, atol=1e-11)
    # the inverse undoes the forward transform
    np.testing.assert_allclose(O.inverse_rht_tiles(Wt, d, T), W, rtol=1e-12, atol=1e-12)


def test_identity_in_matrix_form():
    """(W H D)(D H^T x)/n = W x on one tile, with H the library Hadamard matrix."""
    rng = np.random.default_rng(2)
    n = 512
    W = rng.standard_normal((7, n))
    x = rng.standard_normal(n)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    D = np.diag(O.splitmix64_signs(11, n).astype(np.float64))
    np.testing.assert_allclose((W @ H @ D) @ (D @ H.T @ x) / n, W @ x, rtol=1e-11, atol=1e-11)
    # the oracle's transform of one row is H D w / sqrt(n)
    np.testing.assert_allclose(O.rht_tiles(W, np.diag(D).astype(np.int8), n),
                               (W @ D @ H.T) / np.sqrt(n), rtol=1e-12, atol=1e-13)


def test_spike_maps_to_flat():
    T = 256
    d = O.splitmix64_signs(5, T)
    for j in (0, 1, 77, 255):
        w = np.zeros((1, T))
        w[0, j] = 1.0
        wt = O.rht_tiles(w, d, T)[0]
        assert np.allclose(np.abs(wt), 1.0 / np.sqrt(T), atol=1e-15)
        # entry i has the sign (-1)^popcount(i & j) * d_j
        expect = d[j] * np.array([(-1) ** bin(i & j).count("1") for i in range(T)]) / np.sqrt(T)
        np.testing.assert_allclose(wt, expect, atol=1e-15)


def test_rht_spreads_outliers_on_small_case():
    """RHT removes outlier coordinates (HyperQuant page, 'Key algorithmic ingredients')."""
    W, _ = small_fp32_case(0)
    d = O.splitmix64_signs(0, W.shape[1])
    Wt = O.rht_tiles(W, d, 256)
    rms = np.sqrt(np.mean(W.astype(np.float64) ** 2))
    assert np.max(np.abs(W)) / rms > 15.0
    assert np.max(np.abs(Wt)) / rms < 7.0


# ---------------------------------------------------------------- a5 lattices
def _enumerate_min_vectors(lattice, radius_codes):
    n = O.LATTICE_DIM[lattice]
    rng = np.arange(-radius_codes, radius_codes + 1)
    grid = np.array(np.meshgrid(*([rng] * n), indexing="ij")).reshape(n, -1).T
    grid = grid[O.code_membership_ok(lattice, grid)]
    nz = grid[np.any(grid != 0, axis=1)]
    p = O.codes_to_point(lattice, nz)
    norms = np.sum(p * p, axis=1)
    m = norms.min()
    return m, int(np.sum(np.isclose(norms, m, rtol=0, atol=1e-12)))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_kissing_numbers(lattice, golden_dir):
    tb = _load(golden_dir, "textbook_lattices.json")
    m, count = _enumerate_min_vectors(lattice, 2)
    assert count == tb["kissing_number"][lattice]
    assert np.isclose(m, tb["minimal_norm2"][lattice], atol=1e-12)


def test_hand_cases(golden_dir):
    cases = _load(golden_dir, "decode_hand_cases.json")["cases"]
    for c in cases:
        y = np.array(c["y"], dtype=np.float64)[None, :]
        p = O.nearest_point(c["lattice"], y)
        codes = O.point_to_codes(c["lattice"], p)[0]
        assert codes.tolist() == c["codes"], c
        assert np.isclose(O.block_sqdist(c["lattice"], y, codes[None, :])[0], c["dist2"], atol=1e-12)


@pytest.mark.parametrize("lattice,n_blocks", [("e8", 3000), ("d4", 3000), ("a2", 3000), ("z1", 2000)])
def test_decoder_equals_brute_force(lattice, n_blocks):
    """Conway-Sloane decoders against exhaustive search, on random and near-tie blocks."""
    n = O.LATTICE_DIM[lattice]
    rng = np.random.default_rng(100 + n)
    y = rng.standard_normal((n_blocks, n)) * 2.0
    # near-tie blocks: half-integers and integers with tiny perturbations
    y[: n_blocks // 4] = (np.round(y[: n_blocks // 4] * 2) / 2
                          + rng.standard_normal((n_blocks // 4, n)) * 1e-3)
    p = O.nearest_point(lattice, y)
    c = O.point_to_codes(lattice, p)
    assert np.all(O.code_membership_ok(lattice, c))
    d = O.block_sqdist(lattice, y, c)
    for i in range(n_blocks):
        best, tied = O.brute_nearest(lattice, y[i])
        assert d[i] <= best + 1e-12, (i, y[i], c[i], tied)
        assert any(np.array_equal(c[i], t) for t in tied)


def test_z1_is_numpy_rint():
    y = np.random.default_rng(3).standard_normal(10000) * 5
    y[:4] = [0.5, 1.5, -2.5, -0.5]
    np.testing.assert_array_equal(O.nearest_z1(y), np.rint(y))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_lattice_points_decode_to_themselves(lattice):
    n = O.LATTICE_DIM[lattice]
    rng = np.random.default_rng(4)
    raw = rng.integers(-9, 10, size=(5000, n))
    # make valid codes: take decoded points of random y, then perturb slightly
    p0 = O.nearest_point(lattice, raw * 0.37)
    p1 = O.nearest_point(lattice, p0 + rng.standard_normal(p0.shape) * 1e-9)
    np.testing.assert_allclose(p1, p0, atol=1e-12)


def test_e8_symmetries():
    rng = np.random.default_rng(5)
    y = rng.standard_normal((4000, 8)) * 1.5
    p = O.nearest_e8(y)
    d = np.sum((y - p) ** 2, axis=1)
    # sign flip: -decode(-y) is at the same distance (equal away from ties)
    pn = -O.nearest_e8(-y)
    np.testing.assert_allclose(np.sum((y - pn) ** 2, axis=1), d, atol=1e-12)
    # coordinate permutation commutes with decoding (distances equal)
    perm = rng.permutation(8)
    pp = O.nearest_e8(y[:, perm])
    np.testing.assert_allclose(np.sum((y[:, perm] - pp) ** 2, axis=1), d, atol=1e-12)


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_normalized_second_moment_matches_textbook(lattice, golden_dir):
    """Uniform points modulo a sublattice of periods give errors uniform on the Voronoi cell."""
    tb = _load(golden_dir, "textbook_lattices.json")
    n = O.LATTICE_DIM[lattice]
    rng = np.random.default_rng(6)
    N = 400000 if n > 1 else 200000
    if lattice == "a2":
        y = rng.random((N, 2)) * np.array([1.0, np.sqrt(3.0)])
    else:
        y = rng.random((N, n)) * 2.0
    p = O.nearest_point(lattice, y)
    mse = float(np.mean(np.sum((y - p) ** 2, axis=1)))
    G = O.normalized_second_moment(lattice, mse)
    assert abs(G / tb["normalized_second_moment"][lattice]["value"] - 1.0) < 0.01
    assert np.isclose(O.covolume(lattice), tb["covolume"][lattice])


def test_e8_granular_gain_matches_page(golden_dir):
    figs = _load(golden_dir, "pages_figures.json")["e8_granular_gain_db"]
    rng = np.random.default_rng(7)
    y = rng.random((400000, 8)) * 2.0
    p = O.nearest_e8(y)
    G8 = O.normalized_second_moment("e8", float(np.mean(np.sum((y - p) ** 2, axis=1))))
    gain_db = 10.0 * np.log10((1.0 / 12.0) / G8)
    assert abs(gain_db - figs["value"]) <= figs["printed_precision"]


# ---------------------------------------------------------------- a4-a6 quantize
def test_quantize_spike_closed_form():
    """A unit spike at column j: w~ = H_j d_j / sqrt(T), s = beta/sqrt(T), y = +-1/beta."""
    T, C, beta = 256, 512, 0.25
    d = O.splitmix64_signs(9, C)
    W = np.zeros((3, C))
    W[0, 5] = 1.0
    W[1, 300] = -2.0
    W[2, 0] = 1.0
    W[2, 511] = 1.0
    q = O.quantize(W, "e8", T, d, beta)
    assert q.scales[0, 0] == np.float32(beta / 16.0) and q.scales[0, 1] == 0.0
    assert q.scales[1, 1] == np.float32(2.0 * beta / 16.0)
    i = np.arange(T)
    pat5 = np.array([(-1) ** bin(k & 5).count("1") for k in i])
    np.testing.assert_array_equal(q.codes[0, :T], (8 * d[5] * pat5).astype(np.int8))
    assert np.all(q.codes[0, T:] == 0)
    pat44 = np.array([(-1) ** bin(k & 44).count("1") for k in i])   # 300 = 256 + 44
    np.testing.assert_array_equal(q.codes[1, T:], (-8 * d[300] * pat44).astype(np.int8))
    # reconstruction is exact for lattice-exact tiles
    np.testing.assert_allclose(O.dequantize(q.codes, q.scales, d, T, "e8"), W, atol=1e-15)


def test_quantize_scale_is_beta_rms_of_original_tile():
    W, _ = small_fp32_case(0)
    d = O.splitmix64_signs(0, W.shape[1])
    q = O.quantize(W, "e8", 256, d, 0.25)
    rms = np.sqrt(np.mean(W.astype(np.float64).reshape(256, 4, 256) ** 2, axis=-1))
    np.testing.assert_allclose(q.scales, (0.25 * rms).astype(np.float32), rtol=1e-7)


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_quantize_codes_are_brute_force_nearest(lattice):
    n = O.LATTICE_DIM[lattice]
    W = gaussian_matrix(8, 512, 0.02, 11, outlier_frac=0.01, dtype="fp32")
    d = O.splitmix64_signs(1, 512)
    q = O.quantize(W, lattice, 128, d, 0.5)
    yb = q.y.reshape(-1, n)
    cb = q.codes_wide.reshape(-1, n)
    assert np.all(O.code_membership_ok(lattice, cb))
    dist = O.block_sqdist(lattice, yb, cb)
    for i in range(0, yb.shape[0], 3):
        best, _ = O.brute_nearest(lattice, yb[i])
        assert dist[i] <= best + 1e-12


def test_quantize_relative_mse_matches_high_resolution_formula():
    """Relative MSE ~ beta^2 G_E8 for Gaussian data (error uniform on the cell)."""
    W = gaussian_matrix(64, 4096, 0.02, 12, dtype="fp32")
    d = O.splitmix64_signs(2, 4096)
    for beta in (0.125, 0.25):
        q = O.quantize(W, "e8", 256, d, beta)
        What = O.dequantize(q.codes, q.scales, d, 256, "e8")
        rel = np.sum((What - W) ** 2) / np.sum(W.astype(np.float64) ** 2)
        assert abs(rel / (beta ** 2 * 929.0 / 12960.0) - 1.0) < 0.03


def test_quantize_zero_nonfinite_and_range_flags():
    T = 128
    d = O.splitmix64_signs(0, 256)
    W = np.zeros((2, 256))
    W[0, 0] = np.nan
    W[1, 130] = 1.0
    q = O.quantize(W, "e8", T, d, 0.25)
    assert q.nonfinite and not q.range_error
    assert np.all(q.codes[0] == 0) and q.scales[0, 1] == 0.0
    # a spike gives y = +-1/beta, code 2/beta: beta = 0.01 puts it at 200 > 127
    q2 = O.quantize(W[1:], "e8", T, d, 0.01)
    assert q2.range_error


# ---------------------------------------------------------------- a7-a11 products
@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_tile_sum_product_equals_dense_reconstruction(lattice):
    W = gaussian_matrix(48, 1024, 0.02, 13, dtype="bf16")
    d = O.splitmix64_signs(4, 1024)
    q = O.quantize(W, lattice, 256, d, 0.25)
    x = gaussian_vectors(5, 1024, 14, dtype="bf16")
    y1 = O.gemv(q.codes, q.scales, d, 256, lattice, x)
    y2 = O.dense_reconstruction_matmul(q.codes, q.scales, d, 256, lattice, x)
    np.testing.assert_allclose(y1, y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.gemm(q.codes, q.scales, d, 256, lattice, x), y1, rtol=0, atol=0)


def test_gemv_close_to_unquantized_product():
    """The product from the codes approximates W x with the quantizer's relative error."""
    W = gaussian_matrix(256, 4096, 0.02, 15, dtype="bf16")
    d = O.splitmix64_signs(5, 4096)
    q = O.quantize(W, "e8", 256, d, 0.25)
    x = gaussian_vectors(1, 4096, 16, dtype="bf16")
    y = O.gemv(q.codes, q.scales, d, 256, "e8", x)
    exact = x.astype(np.float64) @ W.astype(np.float64).T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 2.0 * np.sqrt(0.25 ** 2 * 929.0 / 12960.0)


# ---------------------------------------------------------------- layout / rule
def test_compression_matches_page(golden_dir):
    f = _load(golden_dir, "pages_figures.json")["int8_codes_16bit_norm_compression"]
    assert abs(O.compression_ratio(256) - f["value"]) <= f["printed_precision"]
    assert abs(O.compression_ratio(128, scale_bits=16) - f["value"]) <= f["printed_precision"]


def test_tile_rule_matches_page(golden_dir):
    f = _load(golden_dir, "pages_figures.json")["hadamard_tile_sizes"]
    for c in f["cases"]:
        assert O.pick_tile(c["cols"], c["requested"], tuple(f["allowed"])) == c["expect"], c


def test_code_entropy_matches_hand_worked_cases(golden_dir):
    """code_entropy_bits against entropies worked out by hand from the counts
    (tests/golden/entropy_hand_cases.json): a dropped minus sign, a natural log
    in place of log2, or counting distinct values instead of occurrences each
    fail one of them."""
    with open(os.path.join(golden_dir, "entropy_hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        got = O.code_entropy_bits(np.asarray(case["codes"], dtype=np.int8))
        assert abs(got - case["bits"]) < 1e-12, (case, got)


def test_code_entropy_bounds_and_relabelling():
    """0 <= H <= log2(number of distinct values), with equality for equal counts,
    and H does not depend on which int8 values carry the counts."""
    rng = np.random.default_rng(3)
    c = rng.integers(-20, 21, size=5000).astype(np.int8)
    h = O.code_entropy_bits(c)
    assert 0.0 < h <= np.log2(len(np.unique(c))) + 1e-12
    perm = rng.permutation(np.arange(-20, 21))
    relabelled = perm[c.astype(np.int64) + 20].astype(np.int8)
    assert abs(O.code_entropy_bits(relabelled) - h) < 1e-12
    equal = np.repeat(np.arange(-16, 16), 7).astype(np.int8)
    assert abs(O.code_entropy_bits(equal) - 5.0) < 1e-12
