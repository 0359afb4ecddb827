"""Plain CPU oracle of the bit-stripped Rice format of lattice codes.

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.  Pure Python integers and lists; meant for small cases.

Source: HyperQuant (github release page of moonmath-ai/HyperQuant), "Key
algorithmic ingredients": lossless bit-stripping removes the bits that the
lattice pins deterministically, then Rice codes (variable length, no fixed
codebook, any integer) store what is left; the mma="bf16" paragraph stores the
weight as such a bitstream (~4 bps) and decodes it inside the GEMV.  Rice
codes: R. F. Rice, "Some practical universal noiseless coding techniques",
JPL Publication 79-22 (1979) -- the Golomb code with divisor 2^K.

The pages fix neither the symbol set nor the bit layout; the readings below are
the plainest ones consistent with them (each is listed in the design notes):

* Bit-stripping, per block of n doubled-coordinate codes c (int8):
  - E8 and A2: every code of a block has the same parity (D8 points / A2 first
    coset give even codes, the shifted coset odd ones).  That parity k is stored
    once, as one raw bit, and the codes are halved: u_i = floor(c_i / 2).
  - D4 and Z1: every code is even; u_i = c_i / 2 and no parity bit is stored.
  - E8 and D4: the sum of the halved codes is even (sum of a D_n point; for the
    shifted E8 coset c = 2d + 1 with d in D8).  The last one's low bit is then
    implied and only floor(u_{n-1} / 2) is stored.
* Symbols are signed integers mapped to unsigned by zigzag: z = 2u (u >= 0),
  z = -2u - 1 (u < 0).
* Rice code of z with parameter K: floor(z / 2^K) one-bits, one zero-bit, then
  the K low bits of z, least significant first.
* One segment per (row, tile): K in 3 bits (least significant first), then per
  block in column order: [parity bit k] and the Rice codes of its symbols in
  coordinate order.  K is the value in 0..7 with the shortest segment (the
  smallest K on equal length).
* Segments follow each other in row-major (row, tile) order with no padding.
  Stream bit b is bit (b mod 32) of 32-bit word floor(b / 32).  The offset of
  every segment (bits from the stream start) is kept in an array [rows, tiles].
"""
from __future__ import annotations

import numpy as np

K_BITS = 3
K_MAX = 7
LATTICE_DIM = {"e8": 8, "d4": 4, "a2": 2, "z1": 1}
_HAS_PARITY_BIT = {"e8": True, "a2": True, "d4": False, "z1": False}
_EVEN_SUM = {"e8": True, "d4": True, "a2": False, "z1": False}


def zigzag(u: int) -> int:
    return 2 * u if u >= 0 else -2 * u - 1


def unzigzag(z: int) -> int:
    return z // 2 if z % 2 == 0 else -(z + 1) // 2


def rice_bits(z: int, K: int) -> list[int]:
    """Rice codeword of z >= 0 as a bit list in stream order."""
    q = z >> K
    return [1] * q + [0] + [(z >> i) & 1 for i in range(K)]


def rice_length(z: int, K: int) -> int:
    return (z >> K) + 1 + K


def strip_block(lattice: str, c) -> tuple[int | None, list[int]]:
    """Codes of one block -> (parity bit or None, symbols before zigzag)."""
    c = [int(v) for v in c]
    n = LATTICE_DIM[lattice]
    assert len(c) == n
    k = None
    if _HAS_PARITY_BIT[lattice]:
        k = c[0] & 1
        assert all((v & 1) == k for v in c), "codes of a block must share one parity"
    else:
        assert all((v & 1) == 0 for v in c), "codes must be even"
    u = [v >> 1 for v in c]                    # floor(c / 2)
    if _EVEN_SUM[lattice]:
        assert sum(u) % 2 == 0, "halved codes must have an even sum"
        u[-1] = u[-1] >> 1                     # low bit implied by the others
    return k, u


def unstrip_block(lattice: str, k: int | None, s: list[int]) -> list[int]:
    """Inverse of :func:`strip_block`."""
    u = list(s)
    if _EVEN_SUM[lattice]:
        u[-1] = 2 * u[-1] + (sum(u[:-1]) & 1)
    kk = k if k is not None else 0
    return [2 * v + kk for v in u]


def _segment_symbols(lattice: str, codes_tile):
    n = LATTICE_DIM[lattice]
    out = []
    for j in range(0, len(codes_tile), n):
        k, u = strip_block(lattice, codes_tile[j:j + n])
        out.append((k, [zigzag(v) for v in u]))
    return out


def best_k(lattice: str, codes_tile) -> int:
    """K in 0..7 giving the shortest segment (smallest K on ties)."""
    syms = _segment_symbols(lattice, codes_tile)
    lengths = [sum(rice_length(z, K) for _, zs in syms for z in zs) for K in range(K_MAX + 1)]
    return int(np.argmin(lengths))


def segment_bits(lattice: str, codes_tile, K: int | None = None) -> list[int]:
    """Bits of one (row, tile) segment in stream order."""
    if K is None:
        K = best_k(lattice, codes_tile)
    bits = [(K >> i) & 1 for i in range(K_BITS)]
    for k, zs in _segment_symbols(lattice, codes_tile):
        if k is not None:
            bits.append(k)
        for z in zs:
            bits += rice_bits(z, K)
    return bits


def pack_bits(bits: list[int]) -> np.ndarray:
    words = np.zeros((len(bits) + 31) // 32, dtype=np.uint32)
    for b, v in enumerate(bits):
        if v:
            words[b >> 5] |= np.uint32(1 << (b & 31))
    return words


def encode(codes: np.ndarray, lattice: str, T: int):
    """codes int [rows, cols] -> (words uint32, offsets uint32 [rows, cols/T], total_bits)."""
    rows, cols = codes.shape
    assert cols % T == 0 and T % LATTICE_DIM[lattice] == 0
    tiles = cols // T
    bits: list[int] = []
    offsets = np.zeros((rows, tiles), dtype=np.uint32)
    for r in range(rows):
        for t in range(tiles):
            offsets[r, t] = len(bits)
            bits += segment_bits(lattice, codes[r, t * T:(t + 1) * T].tolist())
    return pack_bits(bits), offsets, len(bits)


class _Reader:
    def __init__(self, words: np.ndarray, pos: int):
        self.words = words
        self.pos = pos

    def bit(self) -> int:
        b = (int(self.words[self.pos >> 5]) >> (self.pos & 31)) & 1
        self.pos += 1
        return b

    def uint(self, nbits: int) -> int:
        return sum(self.bit() << i for i in range(nbits))

    def rice(self, K: int) -> int:
        q = 0
        while self.bit() == 1:
            q += 1
        return (q << K) | self.uint(K)


def decode_segment(words: np.ndarray, offset: int, lattice: str, T: int) -> list[int]:
    n = LATTICE_DIM[lattice]
    rd = _Reader(words, int(offset))
    K = rd.uint(K_BITS)
    out: list[int] = []
    for _ in range(T // n):
        k = rd.bit() if _HAS_PARITY_BIT[lattice] else None
        s = [unzigzag(rd.rice(K)) for _ in range(n)]
        out += unstrip_block(lattice, k, s)
    return out


def decode(words: np.ndarray, offsets: np.ndarray, lattice: str, T: int) -> np.ndarray:
    rows, tiles = offsets.shape
    out = np.zeros((rows, tiles * T), dtype=np.int64)
    for r in range(rows):
        for t in range(tiles):
            out[r, t * T:(t + 1) * T] = decode_segment(words, offsets[r, t], lattice, T)
    return out


def bits_per_weight(total_bits: int, rows: int, cols: int) -> float:
    return total_bits / float(rows * cols)
