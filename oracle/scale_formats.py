"""Plain CPU oracle of the quantizer's alternative scale formats.

TEST INFRASTRUCTURE ONLY: imported by tests and ``__graft_entry__.smoke()``,
never by the library.  It shares no code with the CUDA path.

Sources, cited by page and section:

* HyperQuant (github release page of moonmath-ai/HyperQuant), "mma='int8'"
  paragraph: each weight row is normalised by a per-output-channel statistic
  and the codes are stored with one bfloat16 scale per row.
* Same page, KV-cache storage table: int8 codes with 16-bit (fp16) norms.
* bfloat16: IEEE-754 binary32 cut to 8 significant bits (1 sign, 8 exponent,
  7 fraction bits); float16: IEEE-754 binary16 (5 exponent bits, 10 fraction
  bits, subnormals down to 2^-24, largest finite 65504).  Rounding to both is
  round-to-nearest, ties to even, as IEEE-754 defines it.

Readings where the pages are silent (also in the design notes):

* "row_bf16": the row's statistic is its RMS (the standard deviation about
  zero): s_r = beta * sqrt(mean over the whole row of w~^2), which equals
  beta * RMS of the raw row because each tile's Hadamard is orthonormal.  No
  mean is subtracted: the format stores no offset.  The stored scale is
  bf16(s_r), and the codes are the nearest lattice points of w~ / bf16(s_r),
  so that the stored scale is the one the reconstruction uses.
* "tile_f16": the per-tile scale of the default format, s = beta * RMS(tile),
  stored as fp16(s); codes from w~ / fp16(s).  A scale that overflows fp16 is
  a range error (codes unspecified); one that rounds to zero gives zero codes.
* "tile_f32" is the default format of ``lattice_oracle.quantize``.
"""
from __future__ import annotations

import numpy as np

from . import lattice_oracle as LO

SCALE_FORMATS = ("tile_f32", "row_bf16", "tile_f16")


def _round_binary(x: np.ndarray, frac_bits: int, min_exp: int, max_finite: float) -> np.ndarray:
    """Round to the binary format with `frac_bits` fraction bits, smallest normal
    exponent `min_exp` and largest finite value `max_finite`; ties to even."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    ax = np.abs(x)
    nz = (ax > 0) & np.isfinite(ax)
    # exponent e with 2^e <= |x| < 2^(e+1), floored at the subnormal range
    _, e2 = np.frexp(ax[nz])                   # ax = m 2^e2, m in [0.5, 1)
    e = np.maximum(e2 - 1, min_exp)
    quantum = np.ldexp(1.0, e - frac_bits)      # spacing of representable values
    q = LO.round_half_even(ax[nz] / quantum) * quantum
    # values that round past the largest finite one overflow (IEEE: beyond max + half a quantum)
    top_quantum = np.ldexp(1.0, int(np.floor(np.log2(max_finite))) - frac_bits)
    q = np.where(ax[nz] >= max_finite + top_quantum / 2, np.inf, q)
    out[nz] = np.sign(x[nz]) * q
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value (float64), ties to even."""
    return _round_binary(x, 7, -126, float.fromhex("0x1.fep127"))


def round_to_f16(x: np.ndarray) -> np.ndarray:
    """Nearest float16 value (float64), ties to even."""
    return _round_binary(x, 10, -14, 65504.0)


def codes_with_scales(Wt: np.ndarray, lattice: str, T: int, tile_scales: np.ndarray) -> np.ndarray:
    """Unclipped codes (int64 [rows, cols]) of rotated rows Wt at given per-tile scales.

    A tile whose scale is zero or not finite gets zero codes."""
    n = LO.LATTICE_DIM[lattice]
    rows, cols = Wt.shape
    s_rep = np.repeat(np.asarray(tile_scales, dtype=np.float64), T, axis=1)
    ok = (s_rep > 0) & np.isfinite(s_rep)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(ok, Wt / np.where(ok, s_rep, 1.0), 0.0)
    p = LO.nearest_point(lattice, y.reshape(rows, cols // n, n)).reshape(rows, cols)
    return LO.point_to_codes(lattice, p.reshape(rows, cols // n, n)).reshape(rows, cols)


class FormattedQuant:
    """codes int8 [rows, cols]; scales: stored values as float64 ([rows] for
    row_bf16, [rows, cols/T] otherwise); scales_exact: the unrounded float64
    scales; codes_wide: unclipped codes; range_error / nonfinite flags."""

    def __init__(self, codes_wide, scales, scales_exact, range_error, nonfinite):
        self.codes_wide = codes_wide
        self.codes = np.clip(codes_wide, -128, 127).astype(np.int8)
        self.scales = scales
        self.scales_exact = scales_exact
        self.range_error = range_error
        self.nonfinite = nonfinite


def tile_scales_of(scales: np.ndarray, scale_format: str, tiles_per_row: int) -> np.ndarray:
    """Stored scales of any format as one scale per (row, tile)."""
    s = np.asarray(scales, dtype=np.float64)
    if scale_format == "row_bf16":
        return np.repeat(s.reshape(-1, 1), tiles_per_row, axis=1)
    return s


def quantize_formatted(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, beta: float,
                       scale_format: str) -> FormattedQuant:
    """Quantize W with the scale stored in `scale_format` (see the module notes)."""
    if scale_format not in SCALE_FORMATS:
        raise ValueError(scale_format)
    W = np.asarray(W, dtype=np.float64)
    rows, cols = W.shape
    nt = cols // T
    finite_row = np.all(np.isfinite(W), axis=1)
    finite_tile = np.all(np.isfinite(W.reshape(rows, nt, T)), axis=-1)
    Wt = LO.rht_tiles(np.where(np.isfinite(W), W, 0.0), signs, T)
    if scale_format == "row_bf16":
        exact = beta * np.sqrt(np.mean(Wt * Wt, axis=1))
        stored = round_to_bf16(exact)
        bad = ~finite_row
    else:
        exact = LO.tile_scales(Wt, T, beta)
        stored = round_to_f16(exact) if scale_format == "tile_f16" else exact.astype(np.float32).astype(np.float64)
        bad = ~finite_tile
    per_tile = tile_scales_of(stored, scale_format, nt)
    if scale_format == "tile_f32":
        # the default format decodes against the unrounded scale
        c = codes_with_scales(Wt, lattice, T, exact)
    else:
        c = codes_with_scales(Wt, lattice, T, per_tile)
    bad_rep = np.repeat(bad, cols, axis=0).reshape(rows, cols) if scale_format == "row_bf16" \
        else np.repeat(bad, T, axis=1)
    c = np.where(bad_rep, 0, c)
    range_error = bool(np.any(np.abs(c) > 127)) or bool(np.any(np.isinf(per_tile)))
    return FormattedQuant(c, stored, exact, range_error, bool(np.any(bad)))


def dequantize_formatted(codes, scales, scale_format: str, signs, T: int, lattice: str) -> np.ndarray:
    """W^ = D H (s * p) / sqrt(T) per tile with the stored scales of `scale_format`."""
    nt = np.asarray(codes).shape[1] // T
    return LO.dequantize(codes, tile_scales_of(scales, scale_format, nt), signs, T, lattice)


def gemv_formatted(codes, scales, scale_format: str, signs, T: int, lattice: str, x) -> np.ndarray:
    """y[b, r] = sum_t s[r, t] sum_i p[r, t, i] x~[b, t, i] with the stored scales."""
    nt = np.asarray(codes).shape[1] // T
    return LO.gemv(codes, tile_scales_of(scales, scale_format, nt), signs, T, lattice, x)
