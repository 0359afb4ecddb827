"""GPU quantize / dequantize / KV decode attention with the subtractive Voronoi
dither against the dither oracle (oracle/dither.py)."""
import types

import numpy as np
import pytest

import oracle as O
import oracle.kv_oracle as KV
from oracle import dither as D
from oracle import scale_formats as F
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import compare_codes, normwise_rel
from tests.gpu_util import cuda, to_dev_bf16
from tests.test_gpu_scale_formats import check_scales

pytestmark = pytest.mark.gpu


def dithered_reference(W, lattice, T, d, dseed, got_scales, fmt):
    """Oracle decoder inputs y + u and codes at the scales the GPU stored."""
    Wt = O.rht_tiles(np.asarray(W, dtype=np.float64), d, T)
    s_rep = np.repeat(np.asarray(got_scales, dtype=np.float64), T, axis=1)
    ok = s_rep > 0
    y = np.where(ok, Wt / np.where(ok, s_rep, 1.0), 0.0)
    u = D.dither_vectors(lattice, dseed, *W.shape)
    yu = np.where(ok, y + u, 0.0)
    n = O.LATTICE_DIM[lattice]
    p = O.nearest_point(lattice, yu.reshape(W.shape[0], -1, n)).reshape(W.shape)
    c = O.point_to_codes(lattice, p.reshape(W.shape[0], -1, n)).reshape(W.shape)
    return types.SimpleNamespace(codes_wide=c, y=yu)


def gpu_quantize_dithered(torch, L, W, lattice, T, seed, dseed, fmt):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, signs = L.quantize_dithered(to_dev_bf16(torch, W), lattice=lattice, tile=T, seed=seed,
                                               dither_seed=dseed, beta=0.25, scale_format=fmt, dev_status=st)
    torch.cuda.synchronize()
    return codes, scales, signs, int(st.item())


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("T,fmt", [(128, "tile_f32"), (256, "tile_f16"), (1024, "tile_f32")])
def test_quantize_dequantize_dithered(lattice, T, fmt):
    torch, L = cuda()
    rows, cols = 29, {128: 5 * 128, 256: 5 * 256, 1024: 3 * 1024}[T]
    W = gaussian_matrix(rows, cols, 0.02, 500 + T, outlier_frac=0.002, dtype="bf16")
    codes, scales, signs, st = gpu_quantize_dithered(torch, L, W, lattice, T, 61, 0xABCDEF12345, fmt)
    d = O.splitmix64_signs(61, cols)
    np.testing.assert_array_equal(signs.cpu().numpy(), d)
    q = D.quantize_dithered(W, lattice, T, d, 0.25, 0xABCDEF12345, fmt)
    got_s = scales.float().cpu().numpy()
    if fmt == "tile_f32":
        np.testing.assert_allclose(got_s, q.scales, rtol=1e-6, atol=0)
    else:
        check_scales(got_s, q, fmt)
    assert st == (2 if q.range_error else 0)
    compare_codes(codes.cpu().numpy(), dithered_reference(W, lattice, T, d, 0xABCDEF12345, got_s, fmt), lattice)
    What = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    L.lq_dequantize_dithered(lattice, codes, scales, fmt, signs, 0xABCDEF12345, T, What)
    torch.cuda.synchronize()
    ref = D.dequantize_dithered(codes.cpu().numpy(), got_s, d, T, lattice, 0xABCDEF12345)
    assert normwise_rel(What.cpu().numpy(), ref) < 1e-6


def test_dithered_reconstruction_is_unbiased_on_gpu():
    """Averaging the GPU reconstructions over 24 dither seeds shrinks the error
    like 1/sqrt(24); each single error has the E8 cell's second moment."""
    torch, L = cuda()
    W = gaussian_matrix(64, 1024, 0.02, 520, dtype="bf16")
    Wd = to_dev_bf16(torch, W)
    errs = []
    for k in range(24):
        c, s, g = L.quantize_dithered(Wd, lattice="e8", tile=128, seed=3, dither_seed=900 + k, beta=0.5)
        R = torch.empty((64, 1024), dtype=torch.float32, device="cuda")
        L.lq_dequantize_dithered("e8", c, s, "tile_f32", g, 900 + k, 128, R)
        errs.append(R.cpu().numpy() - W)
    E = np.stack(errs)
    single = np.sqrt((E ** 2).mean())
    assert np.sqrt((E.mean(axis=0) ** 2).mean()) < 0.3 * single
    s2 = np.repeat(s.cpu().numpy(), 128, axis=1) ** 2
    assert abs((E ** 2).mean() / (929.0 / 12960.0 * s2.mean()) - 1.0) < 0.05


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tokens,kv_heads,group,fmt", [(1500, 2, 4, "tile_f32"), (300, 1, 8, "tile_f16"),
                                                       (37, 2, 1, "tile_f32"), (1000, 2, 2, "tile_f16")])
def test_attention_dithered(lattice, tokens, kv_heads, group, fmt):
    torch, L = cuda()
    cols = kv_heads * 128
    X = gaussian_matrix(tokens, cols, 1.0, 830 + tokens, dtype="bf16")
    Y = gaussian_matrix(tokens, cols, 1.0, 831 + tokens, dtype="bf16")
    kc, ks, kg, st1 = gpu_quantize_dithered(torch, L, X, lattice, 128, 71, 1111, fmt)
    vc, vs, vg, st2 = gpu_quantize_dithered(torch, L, Y, lattice, 128, 72, 2222, fmt)
    assert st1 == 0 and st2 == 0
    q = gaussian_vectors(kv_heads * group, 128, 832, dtype="bf16")
    out = torch.empty((kv_heads * group, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kv_heads, kv_heads * group, 128), dtype=torch.uint8,
                     device="cuda")
    L.lq_attention_decode_dithered(lattice, kc, ks, kg, 1111, vc, vs, vg, 2222, fmt, to_dev_bf16(torch, q), out, ws)
    torch.cuda.synchronize()
    dk, dv = O.splitmix64_signs(71, cols), O.splitmix64_signs(72, cols)
    Kh = D.dequantize_dithered(kc.cpu().numpy(), ks.float().cpu().numpy(), dk, 128, lattice, 1111)
    Vh = D.dequantize_dithered(vc.cpu().numpy(), vs.float().cpu().numpy(), dv, 128, lattice, 2222)
    ref = KV.attention_decode(q, Kh, Vh, kv_heads, 128)
    assert normwise_rel(out.cpu().numpy(), ref) < 2e-3


def test_quantize_dithered_fp32_input():
    """fp32 weights (the fp32 load path) with the dither, tile 256, E8 and D4."""
    torch, L = cuda()
    from tests.gpu_util import to_dev
    W = gaussian_matrix(21, 1280, 0.02, 540, outlier_frac=0.002, dtype="fp32")
    d = O.splitmix64_signs(63, 1280)
    for lattice in ("e8", "d4"):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        codes, scales, signs = L.quantize_dithered(to_dev(torch, W.astype(np.float32)), lattice=lattice, tile=256,
                                                   seed=63, dither_seed=77, beta=0.25, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got_s = scales.cpu().numpy()
        q = D.quantize_dithered(W, lattice, 256, d, 0.25, 77)
        np.testing.assert_allclose(got_s, q.scales, rtol=1e-6, atol=0)
        compare_codes(codes.cpu().numpy(), dithered_reference(W, lattice, 256, d, 77, got_s, "tile_f32"), lattice)
