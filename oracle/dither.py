"""Plain CPU oracle of the subtractive Voronoi dither of the quantizer.

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.  It shares
no code with the CUDA path.

Sources, cited by page and section:

* HyperQuant (github release page of moonmath-ai/HyperQuant), "Key algorithmic
  ingredients": two ways, usable together, to keep the cache's inner products
  unbiased -- a QJL rotation and a subtractive dither over the lattice cell;
  its file list names the cache quantizer's rotation and dither.
* Subtractive dither with a lattice (Zamir & Feder, "On lattice quantization
  noise", IEEE Trans. Inf. Theory 42, 1996): with u uniform over the Voronoi
  cell V of the lattice and independent of x, the error Q(x + u) - u - x is
  uniform over -V and independent of x (so its mean is zero and its second
  moment per coordinate is the lattice's G V^(2/n)).

Readings where the pages are silent (also in the design notes):

* One dither vector per quantized block, one value per element, from a
  counter: element (r, k) of a [rows x cols] matrix uses SplitMix64 output
  number r * cols + k (0-based) from state ``dither_seed`` -- the generator of
  the signs -- and w = (top 24 bits) / 2^24 in [0, 1).
* Uniform over V: z = box * w in a box that tiles space under a sublattice of
  the lattice (E8, D4: [0, 2)^n, as 2Z^n lies in both; A2: [0, 1) x [0, sqrt 3),
  as Z x sqrt(3) Z lies in A2; Z: [0, 1)), reduced modulo the lattice:
  u = z - Q(z).  The box is a union of whole cells' worth of volume, so the
  reduction maps its uniform law onto the uniform law of V.
* Quantize: y = w~ / s as without dither; the codes are those of p = Q(y + u);
  codes and scales keep their formats.  Reconstruction uses s (p - u).
"""
from __future__ import annotations

import numpy as np

from . import lattice_oracle as LO
from . import scale_formats as F

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_SQRT3 = np.sqrt(3.0)


def splitmix64_at(seed: int, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 output number `counters` (0-based) from state `seed` (uint64 array)."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & ((1 << 64) - 1)) + (c + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def dither_uniform(seed: int, rows: int, cols: int) -> np.ndarray:
    """w[r, k] in [0, 1): top 24 bits of SplitMix64 output r * cols + k, over 2^24."""
    idx = np.arange(rows * cols, dtype=np.uint64).reshape(rows, cols)
    return (splitmix64_at(seed, idx) >> np.uint64(40)).astype(np.float64) / float(1 << 24)


def box_of(lattice: str) -> np.ndarray:
    """Side lengths of the sampling box of one block."""
    return {"e8": np.full(8, 2.0), "d4": np.full(4, 2.0), "a2": np.array([1.0, _SQRT3]),
            "z1": np.array([1.0])}[lattice]


def dither_vectors(lattice: str, seed: int, rows: int, cols: int) -> np.ndarray:
    """u [rows, cols] (point coordinates of each block): z - Q(z), z = box * w."""
    n = LO.LATTICE_DIM[lattice]
    w = dither_uniform(seed, rows, cols).reshape(rows, cols // n, n)
    z = w * box_of(lattice)
    return (z - LO.nearest_point(lattice, z)).reshape(rows, cols)


def quantize_dithered(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, beta: float, dither_seed: int,
                      scale_format: str = "tile_f32"):
    """Quantize W with the subtractive dither; scales as in `scale_format`
    ("tile_f32" or "tile_f16").  Returns an object with codes, codes_wide,
    scales, scales_exact, y (the decoder inputs y + u), u, range_error,
    nonfinite."""
    if scale_format not in ("tile_f32", "tile_f16"):
        raise ValueError(scale_format)
    n = LO.LATTICE_DIM[lattice]
    W = np.asarray(W, dtype=np.float64)
    rows, cols = W.shape
    nt = cols // T
    finite_tile = np.all(np.isfinite(W.reshape(rows, nt, T)), axis=-1)
    Wt = LO.rht_tiles(np.where(np.isfinite(W), W, 0.0), signs, T)
    exact = LO.tile_scales(Wt, T, beta)
    stored = F.round_to_f16(exact) if scale_format == "tile_f16" else exact.astype(np.float32).astype(np.float64)
    per_tile = exact if scale_format == "tile_f32" else stored
    s_rep = np.repeat(per_tile, T, axis=1)
    ok = (s_rep > 0) & np.isfinite(s_rep)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(ok, Wt / np.where(ok, s_rep, 1.0), 0.0)
    u = dither_vectors(lattice, dither_seed, rows, cols)
    yu = np.where(ok, y + u, 0.0)
    p = LO.nearest_point(lattice, yu.reshape(rows, cols // n, n)).reshape(rows, cols)
    c = LO.point_to_codes(lattice, p.reshape(rows, cols // n, n)).reshape(rows, cols)
    c = np.where(np.repeat(~finite_tile, T, axis=1), 0, c)
    out = F.FormattedQuant(c, stored, exact, bool(np.any(np.abs(c) > 127)) or bool(np.any(np.isinf(stored))),
                           bool(np.any(~finite_tile)))
    out.y = yu
    out.u = u
    return out


def dequantize_dithered(codes, scales, signs, T: int, lattice: str, dither_seed: int) -> np.ndarray:
    """W^ = D H (s (p - u)) / sqrt(T) per tile."""
    n = LO.LATTICE_DIM[lattice]
    codes = np.asarray(codes, dtype=np.int64)
    rows, cols = codes.shape
    p = LO.codes_to_point(lattice, codes.reshape(rows, cols // n, n)).reshape(rows, cols)
    u = dither_vectors(lattice, dither_seed, rows, cols)
    s = np.repeat(np.asarray(scales, dtype=np.float64), T, axis=1)
    return LO.inverse_rht_tiles(s * (p - u), signs, T)
