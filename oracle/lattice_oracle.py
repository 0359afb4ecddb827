"""Float64 CPU oracle of per-tile RHT + lattice vector quantization of weights.

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.

Sources, cited by page and section:

* HyperQuant (github release page of moonmath-ai/HyperQuant), "Key algorithmic
  ingredients": per-tile Randomized Hadamard Transform (random +-1 signs, then a
  Walsh-Hadamard transform), optimal low-dimensional lattice VQ (E8, D4, A2,
  Z1), E8's 0.65 dB granular gain over scalar quantization.
* Same page, intro paragraph: the four lattices E8, D4, A2, Z1.
* Same page, "mma='int8'" paragraph: decoded codes held as int8 ("E8int decode
  into int8"); on each forward the activation goes through the RHT first.
* Same page, "Hadamard block size" paragraph: tile sizes {256, 512, 1024, 2048},
  the largest allowed size <= the requested one that divides in_features.
* Same page, KV-cache storage table: int8 codes + 16-bit norms give ~1.97x.
* Nearest-point decoders for Z^n, D_n, E8 (via D8 and D8 + 1/2) and the
  normalised second moments: Conway & Sloane, "Sphere Packings, Lattices and
  Groups", ch. 20 (nearest-point algorithms) and ch. 2 table 2.3.

Readings where the page is silent (each also listed in the design notes):

* Tiles are 1 x T runs along the columns (in_features) of one row.
* Hadamard in Sylvester natural order, H[i, j] = (-1)^popcount(i & j),
  orthonormal scaling 1/sqrt(T); signs before the Hadamard: w~ = H D w / sqrt(T).
* One sign per global column, drawn from SplitMix64 (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014): sign k is -1
  when the top bit of the (k+1)-th output from state ``seed`` is set.
* Per-tile scale s = beta * sqrt(mean(w~^2)); y = w~ / s; s == 0 gives y = 0.
  The stored scale is float32(s).
* Rounding is half-to-even.  D_n parity fix re-rounds the coordinate with the
  largest |y_i - rint(y_i)| (lowest index on ties) the other way (+1 when the
  residual is >= 0).  E8 keeps the D8 candidate when the two coset distances tie.
* A2 is the hexagonal lattice of minimum distance 1, Z x sqrt(3)Z together with
  its coset shifted by (1/2, sqrt(3)/2); its code for point (x, y) is
  (2x, 2y/sqrt(3)).  Other lattices store the doubled coordinates 2p.
* A code vector is valid when every |c| <= 127; otherwise the range flag is set.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

LATTICES = ("e8", "d4", "a2", "z1")
LATTICE_DIM = {"e8": 8, "d4": 4, "a2": 2, "z1": 1}
_SQRT3 = np.sqrt(3.0)

# --------------------------------------------------------------------------
# a1: Rademacher signs
# --------------------------------------------------------------------------
_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1


def splitmix64(state: int, count: int) -> list[int]:
    """First ``count`` outputs of SplitMix64 started from ``state``.

    Published definition (Steele, Lea & Flood 2014, the public-domain
    ``splitmix64`` generator): the state advances by the golden-ratio increment
    and each output is the state passed through the two xor-shift-multiply
    rounds of the MurmurHash3 64-bit finaliser variant (shifts 30, 27, 31).
    Pure Python integers; no vectorisation.
    """
    out = []
    s = state & _MASK
    for _ in range(count):
        s = (s + _GAMMA) & _MASK
        z = s
        z = ((z ^ (z >> 30)) * _M1) & _MASK
        z = ((z ^ (z >> 27)) * _M2) & _MASK
        z = z ^ (z >> 31)
        out.append(z)
    return out


def splitmix64_signs(seed: int, n: int) -> np.ndarray:
    """Random +-1 diagonal of the RHT, one entry per column (int8 [n]).

    HyperQuant page, "Key algorithmic ingredients" (randomized Hadamard) and
    the KV "signs" rotation (random +-1 diagonal).  Sign k is -1 iff the top
    bit of SplitMix64 output k (0-based) from state ``seed`` is 1.
    """
    outs = splitmix64(seed, n)
    return np.array([-1 if (z >> 63) else 1 for z in outs], dtype=np.int8)


# --------------------------------------------------------------------------
# a3: per-tile randomized Hadamard transform
# --------------------------------------------------------------------------
def hadamard_matrix(T: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_T with H[i, j] = (-1)^popcount(i & j) (float64)."""
    if T <= 0 or (T & (T - 1)) != 0:
        raise ValueError("T must be a power of two")
    i = np.arange(T)
    parity = np.zeros((T, T), dtype=np.int64)
    both = i[:, None] & i[None, :]
    while both.any():
        parity ^= both & 1
        both = both >> 1
    return np.where(parity == 1, -1.0, 1.0)


def rht_tiles(A: np.ndarray, signs: np.ndarray, T: int) -> np.ndarray:
    """Per-tile RHT of each row of A: tile t of row r maps to H_T (d_t * a_t) / sqrt(T).

    HyperQuant page, "Key algorithmic ingredients" (per-tile RHT).  A is
    [rows x cols], cols % T == 0; computed as an explicit dense product with
    H_T in float64 (no butterfly), tile by tile.
    """
    A = np.asarray(A, dtype=np.float64)
    rows, cols = A.shape
    if cols % T:
        raise ValueError("cols must be a multiple of T")
    H = hadamard_matrix(T)
    d = np.asarray(signs, dtype=np.float64)
    out = np.empty_like(A)
    for t in range(cols // T):
        sl = slice(t * T, (t + 1) * T)
        v = A[:, sl] * d[sl][None, :]
        out[:, sl] = (v @ H.T) / np.sqrt(T)
    return out


def inverse_rht_tiles(B: np.ndarray, signs: np.ndarray, T: int) -> np.ndarray:
    """Inverse of :func:`rht_tiles`: tile b_t maps back to D_t H_T b_t / sqrt(T)."""
    B = np.asarray(B, dtype=np.float64)
    rows, cols = B.shape
    H = hadamard_matrix(T)
    d = np.asarray(signs, dtype=np.float64)
    out = np.empty_like(B)
    for t in range(cols // T):
        sl = slice(t * T, (t + 1) * T)
        out[:, sl] = d[sl][None, :] * ((B[:, sl] @ H.T) / np.sqrt(T))
    return out


# --------------------------------------------------------------------------
# a5: nearest lattice points (Conway & Sloane, ch. 20)
# --------------------------------------------------------------------------
def round_half_even(y: np.ndarray) -> np.ndarray:
    """Nearest integer, ties to even (IEEE default rounding)."""
    return np.rint(y)


def nearest_z1(y: np.ndarray) -> np.ndarray:
    """Nearest point of Z^n: coordinate-wise rounding."""
    return round_half_even(y)


def nearest_dn(y: np.ndarray) -> np.ndarray:
    """Nearest point of D_n = {x in Z^n : sum(x) even} for blocks y [..., n].

    Round every coordinate; if the rounded sum is odd, round the worst
    coordinate (largest |y_i - f_i|, first index on ties) the other way.
    """
    y = np.asarray(y, dtype=np.float64)
    f = round_half_even(y)
    delta = y - f
    odd = (np.sum(f, axis=-1) % 2) != 0
    if np.any(odd):
        k = np.argmax(np.abs(delta), axis=-1)
        idx = np.nonzero(odd)
        kk = k[idx]
        step = np.where(delta[idx + (kk,)] >= 0.0, 1.0, -1.0)
        f[idx + (kk,)] += step
    return f


def nearest_e8(y: np.ndarray) -> np.ndarray:
    """Nearest point of E8 = D8 u (D8 + 1/2) for blocks y [..., 8].

    Decode each coset with the D8 decoder and keep the closer one; on equal
    squared distances keep the D8 candidate.
    """
    y = np.asarray(y, dtype=np.float64)
    a = nearest_dn(y)
    b = nearest_dn(y - 0.5) + 0.5
    da = np.sum((y - a) ** 2, axis=-1)
    db = np.sum((y - b) ** 2, axis=-1)
    take_b = db < da
    return np.where(take_b[..., None], b, a)


def nearest_a2(y: np.ndarray) -> np.ndarray:
    """Nearest point of the hexagonal lattice A2 (minimum distance 1), blocks [..., 2].

    A2 = R u (R + (1/2, sqrt(3)/2)) with R = Z x sqrt(3) Z; each coset is a
    rectangular lattice decoded by coordinate rounding; keep the closer one
    (the R candidate on ties).
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.stack([round_half_even(y[..., 0]),
                  _SQRT3 * round_half_even(y[..., 1] / _SQRT3)], axis=-1)
    b = np.stack([round_half_even(y[..., 0] - 0.5) + 0.5,
                  _SQRT3 * (round_half_even(y[..., 1] / _SQRT3 - 0.5) + 0.5)], axis=-1)
    da = np.sum((y - a) ** 2, axis=-1)
    db = np.sum((y - b) ** 2, axis=-1)
    return np.where((db < da)[..., None], b, a)


def nearest_point(lattice: str, y: np.ndarray) -> np.ndarray:
    """Dispatch to the nearest-point decoder of ``lattice`` (blocks in the last axis)."""
    if lattice == "e8":
        return nearest_e8(y)
    if lattice == "d4":
        return nearest_dn(y)
    if lattice == "a2":
        return nearest_a2(y)
    if lattice == "z1":
        return nearest_z1(y)
    raise ValueError(f"unknown lattice {lattice!r}")


def point_to_codes(lattice: str, p: np.ndarray) -> np.ndarray:
    """Lattice point -> integer code (int64): 2p, or (2x, 2y/sqrt(3)) for A2."""
    p = np.asarray(p, dtype=np.float64)
    if lattice == "a2":
        c = np.stack([2.0 * p[..., 0], 2.0 * p[..., 1] / _SQRT3], axis=-1)
    else:
        c = 2.0 * p
    return np.rint(c).astype(np.int64)


def codes_to_point(lattice: str, c: np.ndarray) -> np.ndarray:
    """Integer code -> lattice point (float64); inverse of :func:`point_to_codes`."""
    c = np.asarray(c, dtype=np.float64)
    if lattice == "a2":
        return np.stack([0.5 * c[..., 0], 0.5 * _SQRT3 * c[..., 1]], axis=-1)
    return 0.5 * c


def code_membership_ok(lattice: str, c: np.ndarray) -> np.ndarray:
    """True where a code block [..., n] is the code of a lattice point.

    E8: all coordinates of one parity and sum = 0 mod 4.  D4: all even and
    sum = 0 mod 4.  A2: both of one parity.  Z1: even.
    """
    c = np.asarray(c, dtype=np.int64)
    par = c & 1
    same = np.all(par == par[..., :1], axis=-1)
    if lattice == "e8":
        return same & (np.sum(c, axis=-1) % 4 == 0)
    if lattice == "d4":
        return np.all(par == 0, axis=-1) & (np.sum(c, axis=-1) % 4 == 0)
    if lattice == "a2":
        return same
    if lattice == "z1":
        return np.all(par == 0, axis=-1)
    raise ValueError(lattice)


def block_sqdist(lattice: str, y: np.ndarray, c: np.ndarray) -> np.ndarray:
    """Squared distance ||y - point(c)||^2 per block, float64."""
    p = codes_to_point(lattice, c)
    return np.sum((np.asarray(y, dtype=np.float64) - p) ** 2, axis=-1)


def _brute_axis_candidates(lattice: str, y: np.ndarray, radius: float, parity: int):
    """Per coordinate, the integer codes of the given parity whose point lies within ``radius``."""
    n = LATTICE_DIM[lattice]
    cands = []
    for i in range(n):
        unit = 0.5 * _SQRT3 if (lattice == "a2" and i == 1) else 0.5
        lo = int(np.ceil((y[i] - radius) / unit - 1e-12))
        hi = int(np.floor((y[i] + radius) / unit + 1e-12))
        k = np.arange(lo, hi + 1, dtype=np.int64)
        cands.append(k[(k & 1) == parity])
    return cands


# Covering radii (lattice units): a nearest point is never farther than this,
# so per coordinate it lies within the radius of y.
_COVERING_RADIUS = {"e8": 1.0, "d4": 1.0, "a2": 1.0 / np.sqrt(3.0), "z1": 0.5}
# Code parity classes: E8 and A2 codes are all even or all odd; D4 and Z1 are even.
_PARITIES = {"e8": (0, 1), "d4": (0,), "a2": (0, 1), "z1": (0,)}


def brute_nearest(lattice: str, y_block: np.ndarray, tol: float = 1e-12):
    """Exhaustive nearest point of one block by enumeration of codes.

    Enumerates every integer code, one parity class at a time, whose point lies
    coordinate by coordinate within the covering radius of y (for E8 that is
    the +-2 doubled-coordinate neighbourhood of 2y), keeps those that pass
    :func:`code_membership_ok`, and returns (best_distance, array of every code
    within ``tol`` of it).
    """
    y = np.asarray(y_block, dtype=np.float64)
    r = _COVERING_RADIUS[lattice] + 1e-9
    grids = []
    for par in _PARITIES[lattice]:
        cands = _brute_axis_candidates(lattice, y, r, par)
        if any(len(c) == 0 for c in cands):
            continue
        mesh = np.meshgrid(*cands, indexing="ij")
        grids.append(np.stack([m.ravel() for m in mesh], axis=1))
    grid = np.concatenate(grids, axis=0)
    grid = grid[code_membership_ok(lattice, grid)]
    d = block_sqdist(lattice, y[None, :], grid)
    best = d.min()
    return best, grid[d <= best + tol]


# --------------------------------------------------------------------------
# a4-a6: quantize
# --------------------------------------------------------------------------
def tile_scales(Wt: np.ndarray, T: int, beta: float) -> np.ndarray:
    """s = beta * sqrt(mean(w~^2)) per tile of the rotated rows (float64 [rows, cols/T])."""
    rows, cols = Wt.shape
    sq = (np.asarray(Wt, dtype=np.float64) ** 2).reshape(rows, cols // T, T)
    return beta * np.sqrt(np.mean(sq, axis=-1))


@dataclass
class QuantResult:
    codes: np.ndarray        # int8 [rows, cols] (int64 values clipped into int8 when out of range)
    scales: np.ndarray       # float32 [rows, cols / T]
    y: np.ndarray            # float64 [rows, cols]: w~ / s, the points handed to the decoder
    codes_wide: np.ndarray   # int64 [rows, cols]: the unclipped codes
    nonfinite: bool          # a tile held NaN or Inf
    range_error: bool        # some |code| > 127


def quantize(W: np.ndarray, lattice: str, T: int, signs: np.ndarray, beta: float) -> QuantResult:
    """Quantize W [rows x cols]: per-tile RHT, RMS*beta scale, nearest lattice point.

    Steps a2-a6 of the hot path, float64 throughout, in the order: sign flip,
    Hadamard (explicit matrix), scale, divide, decode, doubled-coordinate codes.
    """
    n = LATTICE_DIM[lattice]
    if T % n:
        raise ValueError("tile must be a multiple of the lattice dimension")
    W = np.asarray(W, dtype=np.float64)
    rows, cols = W.shape
    nt = cols // T
    finite_tile = np.all(np.isfinite(W.reshape(rows, nt, T)), axis=-1)
    Wc = np.where(np.isfinite(W), W, 0.0)
    Wt = rht_tiles(Wc, signs, T)
    s = tile_scales(Wt, T, beta)                           # float64
    s_rep = np.repeat(s, T, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(s_rep > 0.0, Wt / s_rep, 0.0)
    p = nearest_point(lattice, y.reshape(rows, cols // n, n)).reshape(rows, cols)
    c = point_to_codes(lattice, p.reshape(rows, cols // n, n)).reshape(rows, cols)
    nonfinite_rep = np.repeat(~finite_tile, T, axis=1)
    c = np.where(nonfinite_rep, 0, c)
    range_error = bool(np.any(np.abs(c) > 127))
    return QuantResult(
        codes=np.clip(c, -128, 127).astype(np.int8),
        scales=s.astype(np.float32),
        y=y,
        codes_wide=c,
        nonfinite=bool(np.any(~finite_tile)),
        range_error=range_error,
    )


# --------------------------------------------------------------------------
# a11: dequantize
# --------------------------------------------------------------------------
def dequantize(codes: np.ndarray, scales: np.ndarray, signs: np.ndarray, T: int,
               lattice: str) -> np.ndarray:
    """W^ = D H (s32 * p) / sqrt(T) per tile (float64 [rows, cols])."""
    n = LATTICE_DIM[lattice]
    codes = np.asarray(codes, dtype=np.int64)
    rows, cols = codes.shape
    p = codes_to_point(lattice, codes.reshape(rows, cols // n, n)).reshape(rows, cols)
    s = np.repeat(np.asarray(scales, dtype=np.float64), T, axis=1)
    return inverse_rht_tiles(s * p, signs, T)


# --------------------------------------------------------------------------
# a7-a10: products from the codes
# --------------------------------------------------------------------------
def rht_activations(x: np.ndarray, signs: np.ndarray, T: int) -> np.ndarray:
    """x~ = H D x / sqrt(T) per tile of each activation row (float64)."""
    return rht_tiles(np.atleast_2d(np.asarray(x, dtype=np.float64)), signs, T)


def _tile_sum_product(codes, scales, signs, T, lattice, X):
    n = LATTICE_DIM[lattice]
    codes = np.asarray(codes, dtype=np.int64)
    R, C = codes.shape
    nt = C // T
    P = codes_to_point(lattice, codes.reshape(R, C // n, n)).reshape(R, nt, T)
    Xt = rht_activations(X, signs, T).reshape(-1, nt, T)
    partial = np.einsum("rtj,btj->brt", P, Xt)          # per (row, tile) inner products
    return np.sum(partial * np.asarray(scales, dtype=np.float64)[None, :, :], axis=-1)


def gemv(codes, scales, signs, T, lattice, x) -> np.ndarray:
    """y[b, r] = sum_t s32[r, t] * sum_i p[r, t, i] * x~[b, t, i]  (float64 [batch, rows]).

    The decode-side product computed from the codes, never materialising W^
    (HyperQuant page, "mma='bf16'" paragraph: the product is accumulated from
    the codes; no decoded weight is stored).
    """
    return _tile_sum_product(codes, scales, signs, T, lattice, x)


def gemm(codes, scales, signs, T, lattice, X) -> np.ndarray:
    """Y[m, n] = sum_t s32[n, t] * (X~_t[m] . p[n, t])  (float64 [M, N]); same form as gemv."""
    return _tile_sum_product(codes, scales, signs, T, lattice, X)


def dense_reconstruction_matmul(codes, scales, signs, T, lattice, X) -> np.ndarray:
    """Y = X @ W^T with W^ from :func:`dequantize` -- the plain definition of the product."""
    What = dequantize(codes, scales, signs, T, lattice)
    return np.atleast_2d(np.asarray(X, dtype=np.float64)) @ What.T


# --------------------------------------------------------------------------
# statistics and layout helpers
# --------------------------------------------------------------------------
def covolume(lattice: str) -> float:
    """Volume of a fundamental cell at the scale used here."""
    return {"e8": 1.0, "d4": 2.0, "a2": np.sqrt(3.0) / 2.0, "z1": 1.0}[lattice]


def normalized_second_moment(lattice: str, mean_sq_error_per_block: float) -> float:
    """G = E||y - p||^2 / (n V^(2/n)) from the mean squared error per block."""
    n = LATTICE_DIM[lattice]
    return mean_sq_error_per_block / (n * covolume(lattice) ** (2.0 / n))


def compression_ratio(T: int, source_bits: int = 16, code_bits: int = 8,
                      scale_bits: int = 32) -> float:
    """Bits of the source weight over stored bits per weight (code + scale share)."""
    return source_bits / (code_bits + scale_bits / T)


def pick_tile(cols: int, requested: int, allowed=(256, 512, 1024, 2048)) -> int:
    """Largest allowed tile <= requested that divides cols; 0 when none does.

    HyperQuant page, "Hadamard block size" paragraph.
    """
    best = 0
    for t in allowed:
        if t <= requested and cols % t == 0 and t > best:
            best = t
    return best


def code_entropy_bits(codes: np.ndarray) -> float:
    """Empirical zeroth-order entropy of the code values (bits per scalar):
    H = -sum_v p(v) log2 p(v) over the relative counts p(v) of each value
    (Shannon 1948).  Pinned to hand-worked cases (tests/golden/
    entropy_hand_cases.json) and to the bounds 0 <= H <= log2(#values)."""
    vals, counts = np.unique(np.asarray(codes).ravel(), return_counts=True)
    p = counts / counts.sum()
    return float(-(p * np.log2(p)).sum())
