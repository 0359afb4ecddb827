"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module holds no arithmetic of the quantization method: it only draws
random matrices and vectors of the shapes and value distributions of the
workloads (Llama-shaped linear layers, N(0, sigma^2) entries, 0.1 % of entries
scaled x20 as outliers) and rounds them to the storage dtype.

Host arrays come from numpy's PCG64 ``default_rng`` so that the same seed gives
the same values on x86 and Arm hosts.  The helpers return float32 arrays whose
values are exactly representable in the requested storage dtype (bf16 values
are rounded to nearest-even, as a bf16 cast does) together with the raw 16-bit
patterns when the dtype is bf16.
"""
from __future__ import annotations

import numpy as np

# Llama-3-8B decoder layer linear shapes (rows = out_features, cols = in_features)
LLAMA3_8B_LAYER = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)

# Llama-3-70B MLP shapes used by the prefill GEMM workload (rows x cols)
LLAMA3_70B_MLP = (("up_like", 8192, 28672), ("down_like", 28672, 8192))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bit patterns.

    Non-finite values keep their class (NaN stays a quiet NaN, +-inf stays inf).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_to_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    """Return float32 values exactly representable in ``dtype`` ('bf16' or 'fp32')."""
    if dtype == "fp32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(a))
    raise ValueError(f"unknown dtype {dtype!r}")


def gaussian_matrix(rows: int, cols: int, std: float, seed: int, *,
                    outlier_frac: float = 0.0, outlier_mult: float = 20.0,
                    dtype: str = "bf16") -> np.ndarray:
    """N(0, std^2) matrix [rows x cols] from seed; a Bernoulli(outlier_frac) mask
    drawn from the same generator multiplies the masked entries by outlier_mult.

    Returns float32 values representable in ``dtype``.
    """
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(std)
    if outlier_frac > 0.0:
        mask = rng.random((rows, cols), dtype=np.float32) < outlier_frac
        w[mask] *= np.float32(outlier_mult)
    return round_to_dtype(w, dtype)


def gaussian_vectors(batch: int, cols: int, seed: int, *, std: float = 1.0,
                     dtype: str = "bf16") -> np.ndarray:
    """N(0, std^2) activations [batch x cols] from seed, representable in ``dtype``."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, cols), dtype=np.float32) * np.float32(std)
    return round_to_dtype(x, dtype)


def small_fp32_case(seed: int = 0):
    """The small correctness workload: W fp32 256 x 1024, N(0, 0.02^2) with 0.1 %
    of entries x20, and one activation row x ~ N(0, 1) of length 1024, both from
    ``seed``.  Returns (W, x)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((256, 1024), dtype=np.float32) * np.float32(0.02)
    mask = rng.random((256, 1024), dtype=np.float32) < 0.001
    w[mask] *= np.float32(20.0)
    x = rng.standard_normal((1, 1024), dtype=np.float32)
    return w, x


def layer_seed(matrix_index: int, base: int = 1000) -> int:
    """Seed of matrix ``matrix_index`` (q, k, v, o, gate, up, down = 0..6) of a layer."""
    return base + matrix_index


def stack_seed(layer: int, matrix_index: int) -> int:
    """Seed of one matrix of the 32-layer stack."""
    return 2000 + 7 * layer + matrix_index


def torch_gaussian_matrix(rows: int, cols: int, std: float, seed: int, *, device,
                          outlier_frac: float = 0.0, outlier_mult: float = 20.0,
                          dtype=None):
    """Device-side variant for workloads too large to draw on the host.

    Uses a seeded ``torch.Generator`` on ``device``; the values differ from
    :func:`gaussian_matrix` for the same seed.  Returns a torch tensor of
    ``dtype`` (default bfloat16).
    """
    import torch
    dtype = torch.bfloat16 if dtype is None else dtype
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.empty((rows, cols), device=device, dtype=torch.float32)
    w.normal_(0.0, std, generator=g)
    if outlier_frac > 0.0:
        u = torch.empty_like(w)
        u.uniform_(0.0, 1.0, generator=g)
        w = torch.where(u < outlier_frac, w * outlier_mult, w)
        del u
    return w.to(dtype)
