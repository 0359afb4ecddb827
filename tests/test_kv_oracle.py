"""Pins of the KV-cache attention oracle (CPU only): closed forms of softmax
attention that do not retype the oracle."""
import numpy as np

import oracle as O
import oracle.kv_oracle as KV
from synthetic import gaussian_matrix


def test_equal_keys_average_the_values():
    """All keys equal -> uniform weights -> the output is the mean of V."""
    rng = np.random.default_rng(0)
    K = np.tile(rng.standard_normal((1, 128)), (50, 1))
    V = rng.standard_normal((50, 128))
    q = rng.standard_normal((1, 128))
    np.testing.assert_allclose(KV.attention_decode(q, K, V, 1, 128)[0], V.mean(axis=0), rtol=1e-12, atol=1e-12)


def test_dominant_key_selects_its_value():
    """One key aligned with q and 1e3 times larger -> the output is that row of V."""
    rng = np.random.default_rng(1)
    K = rng.standard_normal((40, 128))
    q = rng.standard_normal((1, 128))
    K[17] = 1e3 * q[0] / np.linalg.norm(q[0])
    V = rng.standard_normal((40, 128))
    np.testing.assert_allclose(KV.attention_decode(q, K, V, 1, 128)[0], V[17], rtol=1e-9, atol=1e-9)


def test_two_tokens_closed_form():
    """Two tokens: weight of token 0 is the logistic of (s0 - s1)."""
    rng = np.random.default_rng(2)
    K = rng.standard_normal((2, 128))
    V = rng.standard_normal((2, 128))
    q = rng.standard_normal((1, 128))
    s = K @ q[0] / np.sqrt(128)
    w0 = 1.0 / (1.0 + np.exp(s[1] - s[0]))
    np.testing.assert_allclose(KV.attention_decode(q, K, V, 1, 128)[0], w0 * V[0] + (1 - w0) * V[1], rtol=1e-12)


def test_group_query_heads_share_a_kv_head():
    """q heads 0..3 read kv head 0, 4..7 kv head 1; permuting tokens changes nothing."""
    rng = np.random.default_rng(3)
    K = rng.standard_normal((30, 256))
    V = rng.standard_normal((30, 256))
    q = rng.standard_normal((8, 128))
    o = KV.attention_decode(q, K, V, 2, 128)
    o1 = KV.attention_decode(q[4:5], K[:, 128:], V[:, 128:], 1, 128)
    np.testing.assert_allclose(o[4], o1[0], rtol=1e-12)
    perm = rng.permutation(30)
    np.testing.assert_allclose(KV.attention_decode(q, K[perm], V[perm], 2, 128), o, rtol=1e-12, atol=1e-14)


def test_quantized_attention_tracks_exact_attention():
    """E8 at beta 1/8 on Gaussian K/V: attention from the codes is close to exact
    attention (relative error of order the quantizer's, ~sqrt(beta^2 G) ~ 3 %)."""
    X = gaussian_matrix(64, 256, 1.0, 11)
    Y = gaussian_matrix(64, 256, 1.0, 12)
    q = gaussian_matrix(8, 128, 1.0, 13)
    d = O.splitmix64_signs(5, 256)
    kq = KV.kv_quantize(X, "e8", 128, d, 0.125)
    vq = KV.kv_quantize(Y, "e8", 128, d, 0.125)
    o = KV.attention_from_codes(q, kq.codes, kq.scales, d, vq.codes, vq.scales, d, 2, 128, "e8")
    ref = KV.attention_decode(q, X, Y, 2, 128)
    rel = np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert rel < 0.06, rel


def test_haar_rotation_is_orthogonal_and_haar_like():
    Q = KV.haar_rotation(128, 3)
    np.testing.assert_allclose(Q.T @ Q, np.eye(128), atol=1e-12)
    assert abs(abs(np.linalg.det(Q)) - 1) < 1e-9
    # Haar: every entry has mean 0 and variance 1/d (checked over many draws)
    Qs = np.stack([KV.haar_rotation(16, s) for s in range(400)])
    assert abs(Qs.mean()) < 0.01 and abs((Qs ** 2).mean() - 1 / 16) < 0.002
    # the sign fix matters: diag(R) > 0 convention gives E[Q_00] = 0, not a biased sign
    assert abs(Qs[:, 0, 0].mean()) < 0.05


def test_rotated_attention_is_unchanged_without_quantization():
    """Rotating K, V and q by the same orthogonal Q and the output back by Q^T leaves
    exact attention unchanged (scores are inner products)."""
    rng = np.random.default_rng(4)
    K = rng.standard_normal((40, 256))
    V = rng.standard_normal((40, 256))
    q = rng.standard_normal((4, 128))
    Q = KV.haar_rotation(128, 9)
    o = KV.attention_decode(q, K, V, 2, 128)
    o_rot = KV.attention_decode(KV.rotate_blocks(q, Q), KV.rotate_blocks(K, Q), KV.rotate_blocks(V, Q), 2, 128)
    np.testing.assert_allclose(KV.rotate_blocks(o_rot, Q, transpose=True), o, rtol=1e-10, atol=1e-12)
