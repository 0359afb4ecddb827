"""Pins of the subtractive-dither oracle (oracle/dither.py): published SplitMix64
outputs, Voronoi-cell membership, the textbook second moments of the cells, and
the Zamir-Feder properties of subtractive dither (zero-mean error of fixed
second moment whatever the input; unbiased reconstruction on average)."""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from oracle import dither as D

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_vectors.json")
# Conway & Sloane table 2.3 (normalised second moments); cell volumes at the quantizer's scales
G = {"e8": 929.0 / 12960.0, "d4": 0.0766032, "a2": 5.0 / (36.0 * math.sqrt(3.0)), "z1": 1.0 / 12.0}
V = {"e8": 1.0, "d4": 2.0, "a2": math.sqrt(3.0) / 2.0, "z1": 1.0}


def second_moment(lat):
    n = O.LATTICE_DIM[lat]
    return G[lat] * V[lat] ** (2.0 / n)


def test_splitmix64_published_outputs():
    g = json.load(open(GOLDEN))
    got0 = D.splitmix64_at(0, np.arange(5))
    assert [int(x) for x in got0] == [int(h, 16) for h in g["seed_0"]]
    got1 = D.splitmix64_at(1234567, np.arange(5))
    assert [int(x) for x in got1] == g["seed_1234567"]
    # the counter form equals the sequential generator anywhere in the stream
    assert [int(x) for x in D.splitmix64_at(99, np.arange(1000, 1010))] == O.splitmix64(99, 1010)[1000:]


def test_uniform_draws_are_top_24_bits():
    w = D.dither_uniform(5, 3, 7)
    outs = O.splitmix64(5, 21)
    np.testing.assert_array_equal(w.reshape(-1), [(z >> 40) / 2.0 ** 24 for z in outs])
    assert w.min() >= 0.0 and w.max() < 1.0


@pytest.mark.parametrize("lat", O.LATTICES)
def test_dither_is_uniform_on_the_voronoi_cell(lat):
    n = O.LATTICE_DIM[lat]
    u = D.dither_vectors(lat, 17, 4000, 64 if n != 2 else 64)
    blocks = u.reshape(-1, n)
    # every sample lies in the cell of the origin
    assert np.all(O.nearest_point(lat, blocks) == 0.0)
    # mean zero and the textbook second moment G V^(2/n) per coordinate
    N = blocks.shape[0]
    sd = math.sqrt(second_moment(lat))
    assert np.all(np.abs(blocks.mean(axis=0)) < 5 * sd / math.sqrt(N))
    m2 = float((blocks ** 2).mean())
    assert abs(m2 / second_moment(lat) - 1.0) < 0.02


@pytest.mark.parametrize("lat", O.LATTICES)
def test_subtractive_error_is_input_independent(lat):
    """For fixed inputs -- a lattice point, a point of large error without
    dither, a random point -- Q(y + u) - u - y has mean zero and second moment
    G V^(2/n) per coordinate over the dither draws."""
    n = O.LATTICE_DIM[lat]
    rng = np.random.default_rng(3)
    ys = [np.zeros(n), np.full(n, 0.5), rng.standard_normal(n) * 3.0]
    for y in ys:
        u = D.dither_vectors(lat, 101, 6000, n).reshape(-1, n)
        e = O.nearest_point(lat, y + u) - u - y
        assert np.all(O.nearest_point(lat, -e) == 0.0)           # the error lies in -V
        sd = math.sqrt(second_moment(lat))
        assert np.all(np.abs(e.mean(axis=0)) < 5 * sd / math.sqrt(e.shape[0]))
        assert abs(float((e ** 2).mean()) / second_moment(lat) - 1.0) < 0.05


@pytest.mark.parametrize("lat", ["e8", "a2"])
@pytest.mark.parametrize("fmt", ["tile_f32", "tile_f16"])
def test_dithered_quantizer_reconstruction(lat, fmt):
    """Through the RHT and the scale: the reconstruction error per weight has
    mean zero and second moment G V^(2/n) s^2 (rotations keep it), and the
    average of the reconstructions over dither seeds converges to W."""
    rng = np.random.default_rng(4)
    rows, cols, T = 16, 512, 128
    W = rng.standard_normal((rows, cols)) * 0.02
    d = O.splitmix64_signs(9, cols)
    errs, mean_rec = [], np.zeros_like(W)
    seeds = range(40)
    for k in seeds:
        q = D.quantize_dithered(W, lat, T, d, 0.5, 1000 + k, fmt)
        R = D.dequantize_dithered(q.codes, q.scales, d, T, lat, 1000 + k)
        errs.append(R - W)
        mean_rec += R / len(seeds)
        assert not q.range_error
    E = np.stack(errs)
    s2 = np.repeat(q.scales, T, axis=1) ** 2
    ratio = float((E ** 2).mean(axis=0).mean() / (second_moment(lat) * s2.mean()))
    assert abs(ratio - 1.0) < 0.05
    # mean error shrinks like 1/sqrt(#seeds): far below a single draw's RMS error
    assert np.sqrt(((mean_rec - W) ** 2).mean()) < 0.25 * np.sqrt((E ** 2).mean())


def test_zero_dither_box_reduces_to_plain_quantizer():
    """With the dither forced to zero the dithered path is the plain quantizer."""
    rng = np.random.default_rng(5)
    W = rng.standard_normal((8, 256)) * 0.02
    d = O.splitmix64_signs(2, 256)
    orig = D.dither_vectors
    try:
        D.dither_vectors = lambda lat, seed, r, c: np.zeros((r, c))
        q = D.quantize_dithered(W, "e8", 256, d, 0.25, 7)
    finally:
        D.dither_vectors = orig
    np.testing.assert_array_equal(q.codes, O.quantize(W, "e8", 256, d, 0.25).codes)
