"""Plain CPU oracle of lattice-quantized KV-cache attention (decode step).

TEST INFRASTRUCTURE ONLY: imported by tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.

Source: HyperQuant (github release page of moonmath-ai/HyperQuant), KV-cache
section: the cache stores lattice codes plus one norm per vector (int8 codes
~1.97x, Rice ~3.8x against bf16), the vectors are rotated first ("signs": a
random +-1 diagonal, O(n)), and attention runs on the quantized K/V.  The
readings taken (also listed in the design notes):

* A K or V cache is a matrix [tokens x kv_heads * head_dim]; every (token,
  head) vector is one tile of head_dim columns of the weight quantizer (the
  "signs" rotation = the per-tile RHT, one sign per column, the norm = the
  per-tile scale).  So quantizing a cache is ``lattice_oracle.quantize`` with
  T = head_dim.
* Decode attention of query head h (kv head h // group, group = q_heads /
  kv_heads): o_h = softmax(K^_h q_h / sqrt(head_dim)) V^_h over all tokens,
  with K^, V^ the dequantized caches -- the textbook definition, float64.
* The "qjl" rotation (a Haar-uniform rotation whose inner products are
  unbiased on average, per the page): a Haar orthogonal matrix Q [d x d] drawn as the Q factor of a
  Gaussian matrix with the signs of R's diagonal folded in (Mezzadri, "How to
  generate random matrices from the classical compact groups", Notices AMS
  2007), applied to every head vector (x -> Q x) before the quantizer's own
  sign rotation; queries are rotated by the same Q and the attention output is
  rotated back by Q^T (inner products are unchanged by an orthogonal Q).
"""
from __future__ import annotations

import numpy as np

from . import lattice_oracle as LO


def kv_quantize(X: np.ndarray, lattice: str, head_dim: int, signs: np.ndarray, beta: float):
    """Cache [tokens x kv_heads * head_dim] -> QuantResult (codes, per-vector scales)."""
    return LO.quantize(X, lattice, head_dim, signs, beta)


def attention_decode(q: np.ndarray, K_hat: np.ndarray, V_hat: np.ndarray, kv_heads: int,
                     head_dim: int) -> np.ndarray:
    """q [q_heads x head_dim]; K_hat, V_hat [tokens x kv_heads * head_dim] -> [q_heads x head_dim]."""
    q = np.asarray(q, dtype=np.float64)
    q_heads = q.shape[0]
    group = q_heads // kv_heads
    out = np.zeros((q_heads, head_dim))
    for h in range(q_heads):
        kv = h // group
        Kh = np.asarray(K_hat[:, kv * head_dim:(kv + 1) * head_dim], dtype=np.float64)
        Vh = np.asarray(V_hat[:, kv * head_dim:(kv + 1) * head_dim], dtype=np.float64)
        s = Kh @ q[h] / np.sqrt(head_dim)
        p = np.exp(s - s.max())
        out[h] = (p @ Vh) / p.sum()
    return out


def attention_from_codes(q, k_codes, k_scales, k_signs, v_codes, v_scales, v_signs, kv_heads, head_dim,
                         lattice):
    """Decode attention over caches held as codes: dequantize, then the definition."""
    K_hat = LO.dequantize(k_codes, k_scales, k_signs, head_dim, lattice)
    V_hat = LO.dequantize(v_codes, v_scales, v_signs, head_dim, lattice)
    return attention_decode(q, K_hat, V_hat, kv_heads, head_dim)


def haar_rotation(d: int, seed: int) -> np.ndarray:
    """Haar-distributed orthogonal d x d matrix from a seeded Gaussian matrix."""
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((d, d))
    Q, R = np.linalg.qr(A)
    return Q * np.sign(np.diag(R))[None, :]


def rotate_blocks(X: np.ndarray, Q: np.ndarray, transpose: bool = False) -> np.ndarray:
    """Every d-column block x of every row of X -> Q x (Q^T x with transpose)."""
    X = np.asarray(X, dtype=np.float64)
    d = Q.shape[0]
    M = Q.T if transpose else Q
    rows, cols = X.shape
    return (X.reshape(rows, cols // d, d) @ M.T).reshape(rows, cols)
