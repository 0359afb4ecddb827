"""The seeded input module shared by the oracle tests and the GPU tests: bf16
rounding against torch's own float32 -> bfloat16 conversion (round to nearest,
ties to even), determinism per seed, and the workload recipes (Llama-3-8B layer
shapes, N(0, std^2) with a Bernoulli mask of x20 outliers)."""
import numpy as np
import torch

from synthetic import (LLAMA3_70B_MLP, LLAMA3_8B_LAYER, bf16_bits_to_f32, f32_to_bf16_bits, gaussian_matrix,
                       gaussian_vectors, small_fp32_case)


def _torch_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000)]
    # exact ties between two bf16 neighbours (low 16 bits 0x8000) at both parities of
    # the last kept bit, over finite exponents and both signs
    sign = rng.integers(0, 2, 4000).astype(np.uint32) << 31
    expo = rng.integers(1, 254, 4000).astype(np.uint32) << 23
    mant = rng.integers(0, 128, 4000).astype(np.uint32) << 16
    vals.append((sign | expo | mant | 0x8000).view(np.float32))
    # subnormals, zeros, the largest finite values (which round to inf), infinities
    special = np.array([0.0, -0.0, 1e-40, -1e-40, 1.1754942e-38, 3.4028235e38, -3.4028235e38,
                        3.3961776e38, np.inf, -np.inf], dtype=np.float32)
    vals.append(special)
    a = np.concatenate(vals).astype(np.float32)
    np.testing.assert_array_equal(f32_to_bf16_bits(a), _torch_bf16_bits(a))
    nan = f32_to_bf16_bits(np.array([np.nan], dtype=np.float32))
    assert np.isnan(bf16_bits_to_f32(nan))[0]


def test_bf16_widening_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f32(bits)
    finite = np.isfinite(f)
    np.testing.assert_array_equal(f32_to_bf16_bits(f[finite]), bits[finite])


def test_seeded_draws_are_deterministic():
    a = gaussian_matrix(64, 512, 0.02, 7, outlier_frac=0.01)
    b = gaussian_matrix(64, 512, 0.02, 7, outlier_frac=0.01)
    c = gaussian_matrix(64, 512, 0.02, 8, outlier_frac=0.01)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)
    np.testing.assert_array_equal(gaussian_vectors(4, 256, 3), gaussian_vectors(4, 256, 3))


def test_outlier_mask_scales_entries_by_twenty():
    rows, cols, frac = 512, 1024, 0.001
    plain = gaussian_matrix(rows, cols, 0.02, 11, dtype="fp32")
    spiked = gaussian_matrix(rows, cols, 0.02, 11, outlier_frac=frac, dtype="fp32")
    nz = plain != 0
    ratio = spiked[nz] / plain[nz]
    assert np.all((ratio == 1.0) | (np.abs(ratio - 20.0) < 1e-5))
    n = rows * cols
    k = int(np.sum(np.abs(ratio - 20.0) < 1e-5))
    # Bernoulli(frac) count: within 5 standard deviations of n * frac
    assert abs(k - n * frac) < 5 * np.sqrt(n * frac * (1 - frac))
    assert abs(float(plain.std()) - 0.02) < 0.001


def test_small_case_recipe():
    W, x = small_fp32_case(0)
    assert W.shape == (256, 1024) and W.dtype == np.float32
    assert x.shape == (1, 1024) and x.dtype == np.float32
    big = np.abs(W) > 0.02 * 6     # essentially only the x20 entries
    assert 0.0003 < big.mean() < 0.002


def test_workload_shapes():
    assert [n for n, _, _ in LLAMA3_8B_LAYER] == ["q", "k", "v", "o", "gate", "up", "down"]
    assert sum(r * c for _, r, c in LLAMA3_8B_LAYER) == 218_103_808
    assert dict((n, (r, c)) for n, r, c in LLAMA3_70B_MLP) == {"up_like": (8192, 28672),
                                                             "down_like": (28672, 8192)}
