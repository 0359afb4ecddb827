"""GPU quantize / dequantize / GEMV / GEMM / KV attention with the 16-bit scale
formats (per-row bf16, per-tile fp16) against the scale-format oracle."""
import types

import numpy as np
import pytest

import oracle as O
import oracle.kv_oracle as KV
from oracle import scale_formats as F
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import compare_codes, normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
SCALE_TIE = 1e-5      # relative distance of the exact scale to a rounding midpoint


def _round_fn(fmt):
    return F.round_to_bf16 if fmt == "row_bf16" else F.round_to_f16


def check_scales(got, q, fmt):
    """Stored scales equal the oracle's except where the exact scale lies within
    SCALE_TIE (relative) of the midpoint between the two candidates; returns the
    mask of such certified differences."""
    got = np.asarray(got, dtype=np.float64)
    diff = got != q.scales
    if diff.any():
        mid = 0.5 * (got[diff] + q.scales[diff])
        ex = q.scales_exact[diff]
        near = np.abs(ex - mid) <= SCALE_TIE * np.abs(ex)
        neighbour = _round_fn(fmt)(ex * (1 + 2 * SCALE_TIE)) == got[diff]
        neighbour |= _round_fn(fmt)(ex * (1 - 2 * SCALE_TIE)) == got[diff]
        assert np.all(near & neighbour), f"{int((~(near & neighbour)).sum())} scales differ beyond the tie band"
    return diff


def codes_reference(W, lattice, T, d, got_scales, fmt):
    """Oracle codes and decoder inputs at the scales the GPU stored."""
    Wt = O.rht_tiles(np.asarray(W, dtype=np.float64), d, T)
    per_tile = F.tile_scales_of(got_scales, fmt, W.shape[1] // T)
    s_rep = np.repeat(per_tile, T, axis=1)
    y = np.where(s_rep > 0, Wt / np.where(s_rep > 0, s_rep, 1.0), 0.0)
    c = F.codes_with_scales(Wt, lattice, T, per_tile)
    return types.SimpleNamespace(codes_wide=c, y=y)


def run_ex(torch, L, Wd, lattice, tile, seed, beta, fmt):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, signs = L.quantize_ex(Wd, lattice=lattice, tile=tile, seed=seed, beta=beta, scale_format=fmt,
                                         dev_status=st)
    torch.cuda.synchronize()
    return codes, scales, signs, int(st.item())


@pytest.mark.parametrize("fmt", ["row_bf16", "tile_f16"])
@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile,dtype", [(256, "bf16"), (128, "fp32"), (1024, "bf16")])
def test_quantize_dequantize_gemv_formats(fmt, lattice, tile, dtype):
    torch, L = cuda()
    rows, cols = 37, {128: 5 * 128, 256: 5 * 256, 1024: 3 * 1024}[tile]
    W = gaussian_matrix(rows, cols, 0.02, 300 + tile, outlier_frac=0.002, dtype="bf16")
    Wd = to_dev_bf16(torch, W) if dtype == "bf16" else to_dev(torch, W.astype(np.float32))
    codes, scales, signs, st = run_ex(torch, L, Wd, lattice, tile, 41, 0.25, fmt)
    d = O.splitmix64_signs(41, cols)
    np.testing.assert_array_equal(signs.cpu().numpy(), d)
    q = F.quantize_formatted(W, lattice, tile, d, 0.25, fmt)
    got_s = scales.float().cpu().numpy()
    check_scales(got_s, q, fmt)
    assert st == (2 if q.range_error else 0)
    compare_codes(codes.cpu().numpy(), codes_reference(W, lattice, tile, d, got_s, fmt), lattice)
    # dequantize and the GEMV with the GPU's codes and scales
    c_np = codes.cpu().numpy()
    What = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    L.lq_dequantize_ex(lattice, codes, scales, fmt, signs, tile, What)
    ref = F.dequantize_formatted(c_np, got_s, fmt, d, tile, lattice)
    assert normwise_rel(What.cpu().numpy(), ref) < 1e-6
    for b in (1, 5, 16):
        x = gaussian_vectors(b, cols, 60 + b, dtype="bf16")
        y = torch.empty((b, rows), dtype=torch.float32, device="cuda")
        ws = torch.empty(L.lq_gemv_workspace_size(b, cols, tile), dtype=torch.uint8, device="cuda")
        L.lq_gemv_ex(lattice, codes, scales, fmt, signs, tile, to_dev_bf16(torch, x), y, ws)
        torch.cuda.synchronize()
        assert normwise_rel(y.cpu().numpy(), F.gemv_formatted(c_np, got_s, fmt, d, tile, lattice, x)) < 2e-3


@pytest.mark.parametrize("fmt", ["row_bf16", "tile_f16"])
@pytest.mark.parametrize("lattice", ["e8", "a2"])
def test_gemm_formats(fmt, lattice):
    torch, L = cuda()
    N, K, M, tile = 256, 1536, 70, 256
    W = gaussian_matrix(N, K, 0.02, 310, dtype="bf16")
    codes, scales, signs, st = run_ex(torch, L, to_dev_bf16(torch, W), lattice, tile, 43, 0.25, fmt)
    assert st == 0
    X = gaussian_vectors(M, K, 311, dtype="bf16")
    Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    L.lq_gemm_ex(lattice, codes, scales, fmt, signs, tile, to_dev_bf16(torch, X), Y, ws)
    torch.cuda.synchronize()
    d = O.splitmix64_signs(43, K)
    ref = F.gemv_formatted(codes.cpu().numpy(), scales.float().cpu().numpy(), fmt, d, tile, lattice, X)
    assert normwise_rel(Y.cpu().numpy(), ref) < 2e-3


def test_row_bf16_full_size_gate_matrix_sampled():
    """Llama-3-8B gate_proj 14336 x 4096 bf16 with per-row bf16 scales (three
    40 MB row blocks, each read twice): oracle on sampled rows, GEMV b = 4."""
    torch, L = cuda()
    from synthetic import torch_gaussian_matrix
    Wd = torch_gaussian_matrix(14336, 4096, 0.02, 1004, device="cuda")
    codes, scales, signs, st = run_ex(torch, L, Wd, "e8", 256, 1004, 0.25, "row_bf16")
    assert st == 0
    rng = np.random.default_rng(3)
    rows = np.sort(np.concatenate([[0, 5119, 5120, 14335], rng.choice(14336, 60, replace=False)]))
    W = Wd[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    d = O.splitmix64_signs(1004, 4096)
    q = F.quantize_formatted(W, "e8", 256, d, 0.25, "row_bf16")
    got_s = scales.float().cpu().numpy()[rows]
    check_scales(got_s, q, "row_bf16")
    compare_codes(codes.cpu().numpy()[rows], codes_reference(W, "e8", 256, d, got_s, "row_bf16"), "e8")
    x = gaussian_vectors(4, 4096, 64, dtype="bf16")
    y = torch.empty((4, 14336), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_gemv_workspace_size(4, 4096, 256), dtype=torch.uint8, device="cuda")
    L.lq_gemv_ex("e8", codes, scales, "row_bf16", signs, 256, to_dev_bf16(torch, x), y, ws)
    torch.cuda.synchronize()
    ref = F.gemv_formatted(codes.cpu().numpy()[rows], got_s, "row_bf16", d, 256, "e8", x)
    assert normwise_rel(y.cpu().numpy()[:, rows], ref) < 2e-3


def test_kv_cache_with_fp16_norms():
    """K and V caches quantized with fp16 per-vector scales (T = head_dim = 128),
    decode attention from the codes against the oracle on the same codes."""
    torch, L = cuda()
    tokens, kv_heads, group = 1500, 2, 4
    cols = kv_heads * 128
    X = gaussian_matrix(tokens, cols, 1.0, 820, dtype="bf16")
    Y = gaussian_matrix(tokens, cols, 1.0, 821, dtype="bf16")
    kc, ks, kg, st1 = run_ex(torch, L, to_dev_bf16(torch, X), "e8", 128, 51, 0.25, "tile_f16")
    vc, vs, vg, st2 = run_ex(torch, L, to_dev_bf16(torch, Y), "e8", 128, 52, 0.25, "tile_f16")
    assert st1 == 0 and st2 == 0 and ks.dtype == torch.float16
    dk, dv = O.splitmix64_signs(51, cols), O.splitmix64_signs(52, cols)
    qk = F.quantize_formatted(X, "e8", 128, dk, 0.25, "tile_f16")
    check_scales(ks.float().cpu().numpy(), qk, "tile_f16")
    q = gaussian_vectors(kv_heads * group, 128, 822, dtype="bf16")
    out = torch.empty((kv_heads * group, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kv_heads, kv_heads * group, 128), dtype=torch.uint8,
                     device="cuda")
    L.lq_attention_decode_ex("e8", kc, ks, kg, vc, vs, vg, "tile_f16", to_dev_bf16(torch, q), out, ws)
    torch.cuda.synchronize()
    ref = KV.attention_from_codes(q, kc.cpu().numpy(), ks.float().cpu().numpy(), dk, vc.cpu().numpy(),
                                  vs.float().cpu().numpy(), dv, kv_heads, 128, "e8")
    assert normwise_rel(out.cpu().numpy(), ref) < 2e-3


def test_format_flags():
    """A tile whose fp16 scale overflows raises the range flag; a row holding a
    NaN gets a zero bf16 scale and the non-finite flag."""
    torch, L = cuda()
    W = gaussian_matrix(4, 512, 1.0, 330, dtype="bf16")
    W[2, :256] *= 1e6
    _, s16, _, st = run_ex(torch, L, to_dev(torch, W.astype(np.float32)), "z1", 256, 1, 0.25, "tile_f16")
    assert st & 2 and np.isinf(s16.float().cpu().numpy()[2, 0])
    W2 = gaussian_matrix(3, 256, 0.02, 331, dtype="bf16")
    W2[1, 7] = np.nan
    _, sb, _, st = run_ex(torch, L, to_dev(torch, W2.astype(np.float32)), "e8", 128, 2, 0.25, "row_bf16")
    assert st & 1 and sb.float().cpu().numpy()[1] == 0.0
