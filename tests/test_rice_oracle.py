"""Pins of the Rice-format oracle (CPU only): hand-worked segments, codeword
definition, round trips on quantizer output, K optimality, rate sanity."""
import json
import os

import numpy as np
import pytest

import oracle as O
import oracle.rice_oracle as R
from synthetic import gaussian_matrix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rice_hand_cases.json")


@pytest.fixture(scope="module")
def hand():
    return json.load(open(GOLDEN))


def test_rice_codewords_by_hand(hand):
    for c in hand["rice_codewords"]:
        assert R.rice_bits(c["z"], c["K"]) == c["bits"], c
        assert R.rice_length(c["z"], c["K"]) == len(c["bits"])


def test_segments_by_hand(hand):
    for c in hand["segments"]:
        n = R.LATTICE_DIM[c["lattice"]]
        assert len(c["codes"]) == n
        assert R.best_k(c["lattice"], c["codes"]) == c["K"], c
        bits = R.segment_bits(c["lattice"], c["codes"])
        assert len(bits) == c["nbits"], c
        assert R.pack_bits(bits).tolist() == c["words"], c
        words, offs, total = R.encode(np.array([c["codes"]]), c["lattice"], n)
        assert total == c["nbits"] and offs.tolist() == [[0]] and words.tolist() == c["words"]
        assert R.decode(words, offs, c["lattice"], n).tolist() == [c["codes"]]


def test_two_segments_by_hand(hand):
    c = hand["two_segments"]
    words, offs, total = R.encode(np.array(c["codes"]), c["lattice"], c["tile"])
    assert offs.tolist() == c["offsets"] and total == c["nbits"] and words.tolist() == c["words"]


def test_zigzag_is_a_bijection_on_small_integers():
    zs = [R.zigzag(u) for u in range(-64, 64)]
    assert sorted(zs) == list(range(128))
    assert all(R.unzigzag(R.zigzag(u)) == u for u in range(-64, 64))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_round_trip_on_quantizer_codes(lattice):
    """Codes from the oracle quantizer (outliers included) survive encode/decode; the
    stripped bits are exactly the ones the lattice pins (strip_block asserts them)."""
    W = gaussian_matrix(6, 512, 0.02, 41, outlier_frac=0.01, dtype="bf16")
    q = O.quantize(W, lattice, 256, O.splitmix64_signs(5, 512), 0.25)
    words, offs, total = R.encode(q.codes, lattice, 256)
    assert offs[0, 0] == 0 and np.all(np.diff(offs.reshape(-1).astype(np.int64)) > 0)
    assert R.decode(words, offs, lattice, 256).tolist() == q.codes.tolist()
    assert len(words) == (total + 31) // 32


def test_pinned_bits_are_really_pinned():
    """On E8 codes the parity of every coordinate equals the block's first and the
    halved sum is even -- the two facts the stripping relies on (Conway & Sloane:
    E8 = D8 u (D8 + 1/2))."""
    rng = np.random.default_rng(3)
    y = rng.normal(0, 3, size=(2000, 8))
    c = O.point_to_codes("e8", O.nearest_e8(y)).astype(np.int64)
    assert np.all((c & 1) == (c[:, :1] & 1))
    assert np.all(((c >> 1).sum(axis=1) & 1) == 0)
    assert np.all(c.sum(axis=1) % 4 == 0)


def test_chosen_k_is_optimal():
    rng = np.random.default_rng(7)
    for _ in range(20):
        y = rng.normal(0, rng.uniform(0.5, 12), size=(16, 8))
        codes = O.point_to_codes("e8", O.nearest_e8(y)).astype(np.int64).reshape(-1).tolist()
        K = R.best_k("e8", codes)
        lens = [len(R.segment_bits("e8", codes, k)) for k in range(8)]
        assert lens[K] == min(lens) and lens.index(min(lens)) == K


def test_rate_near_four_bits_at_beta_quarter():
    """E8 at beta = 1/4 on Gaussian weights: the stream lands near the pages' ~4 bps
    operating point (the entropy of the codes is about log2(sqrt(2 pi e)/beta) = 4.05
    bits per coordinate; stripping removes about 1 bit per 8 coordinates)."""
    W = gaussian_matrix(4, 2048, 0.02, 43, dtype="bf16")
    q = O.quantize(W, "e8", 256, O.splitmix64_signs(6, 2048), 0.25)
    words, offs, total = R.encode(q.codes, "e8", 256)
    bps = R.bits_per_weight(total, 4, 2048)
    assert 3.6 < bps < 4.6, bps


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_round_trip_on_arbitrary_lattice_codes(lattice):
    """Random valid codes of any size (not only what the quantizer produces at
    beta = 1/4: runs far longer than K, codes near the int8 ends) survive
    encode -> decode, and every segment decodes from its own offset alone.

    The largest case scales y so that max |y| = 59: every code 2 p then stays
    within |2 y| + 3 <= 121 < 127 (no clipping, so every row is a lattice code)
    and reaches past 100 in magnitude."""
    rng = np.random.default_rng(11)
    n = O.LATTICE_DIM[lattice]
    rows, T = 5, 128
    for case in ("small", "medium", "int8_ends"):
        y = rng.standard_normal((rows, T * 3))
        y *= {"small": 0.3, "medium": 3.0}.get(case, 59.0 / np.abs(y).max())
        p = O.nearest_point(lattice, y.reshape(rows, -1, n)).reshape(rows, -1)
        c = O.point_to_codes(lattice, p.reshape(rows, -1, n)).reshape(rows, -1)
        assert np.abs(c).max() <= 127
        assert O.code_membership_ok(lattice, c.reshape(-1, n)).all()
        if case == "int8_ends":
            assert np.abs(c).max() >= 100, np.abs(c).max()
        words, offsets, total = R.encode(c.astype(np.int8), lattice, T)
        back = R.decode(words, offsets, lattice, T)
        np.testing.assert_array_equal(back, c)
        for r in range(c.shape[0]):
            for t in range(c.shape[1] // T):
                seg = R.decode_segment(words, int(offsets[r, t]), lattice, T)
                np.testing.assert_array_equal(seg, c[r, t * T:(t + 1) * T])
