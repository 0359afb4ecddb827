"""GPU quantize / dequantize / signs against the float64 oracle (through the C ABI)."""
import numpy as np
import pytest

import oracle as O
from synthetic import gaussian_matrix, gaussian_vectors, small_fp32_case
from tests._parity import compare_codes, normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def run_quantize(torch, L, W_np, dtype, lattice, tile, seed, beta, ldw_pad=0):
    rows, cols = W_np.shape
    if dtype == "bf16":
        full = np.zeros((rows, cols + ldw_pad), dtype=np.float32)
        full[:, :cols] = W_np
        Wd = to_dev_bf16(torch, full)[:, :cols]
    else:
        full = np.zeros((rows, cols + ldw_pad), dtype=np.float32)
        full[:, :cols] = W_np
        Wd = to_dev(torch, full)[:, :cols]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, signs = L.quantize(Wd, lattice=lattice, tile=tile, seed=seed, beta=beta, dev_status=status)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), signs.cpu().numpy(), int(status.item())


def test_signs_match_oracle():
    torch, L = cuda()
    for seed, n in ((0, 1024), (12345, 14336), (2**63 + 7, 4096)):
        s = torch.empty(n, dtype=torch.int8, device="cuda")
        L.lq_make_signs(seed, s)
        np.testing.assert_array_equal(s.cpu().numpy(), O.splitmix64_signs(seed, n))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 256, 512, 1024, 2048])
def test_quantize_parity_ragged(lattice, tile):
    torch, L = cuda()
    # not a multiple of the 2048-column chunk (tiles up to 1024)
    rows, cols = 37, {512: 3 * 512, 1024: 3 * 1024, 2048: 3 * 2048}.get(tile, 5 * tile)
    W = gaussian_matrix(rows, cols, 0.02, 100 + tile, outlier_frac=0.002, dtype="bf16")
    for beta in (0.125, 0.25, 0.5):
        codes, scales, signs, st = run_quantize(torch, L, W, "bf16", lattice, tile, 77, beta)
        d = O.splitmix64_signs(77, cols)
        np.testing.assert_array_equal(signs, d)
        q = O.quantize(W, lattice, tile, d, beta)
        assert st == (2 if q.range_error else 0), st
        np.testing.assert_allclose(scales, q.scales, rtol=1e-6, atol=0)
        compare_codes(codes, q, lattice)


def test_small_fp32_case_e8():
    """256 x 1024 fp32 with 0.1 % x20 outliers, tile 256, beta 0.25, seed 0."""
    torch, L = cuda()
    W, _ = small_fp32_case(0)
    codes, scales, signs, st = run_quantize(torch, L, W, "fp32", "e8", 256, 0, 0.25)
    d = O.splitmix64_signs(0, 1024)
    q = O.quantize(W, "e8", 256, d, 0.25)
    assert st == (2 if q.range_error else 0)
    np.testing.assert_allclose(scales, q.scales, rtol=1e-6)
    compare_codes(codes, q, "e8")


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_fp32_multi_chunk(lattice):
    torch, L = cuda()
    W = gaussian_matrix(24, 6144, 0.05, 9, outlier_frac=0.001, dtype="fp32")
    codes, scales, _, st = run_quantize(torch, L, W, "fp32", lattice, 256, 5, 0.25)
    q = O.quantize(W, lattice, 256, O.splitmix64_signs(5, 6144), 0.25)
    np.testing.assert_allclose(scales, q.scales, rtol=1e-6)
    compare_codes(codes, q, lattice)


def test_strided_rows():
    torch, L = cuda()
    W = gaussian_matrix(19, 2048, 0.02, 3, dtype="bf16")
    codes, scales, _, _ = run_quantize(torch, L, W, "bf16", "e8", 256, 1, 0.25, ldw_pad=8 * 5)
    q = O.quantize(W, "e8", 256, O.splitmix64_signs(1, 2048), 0.25)
    np.testing.assert_allclose(scales, q.scales, rtol=1e-6)
    compare_codes(codes, q, "e8")


def test_exact_lattice_points_and_zero_tiles():
    """Unit spikes give y = +-1/beta exactly (codes +-8 at beta 1/4); zero tiles give zeros."""
    torch, L = cuda()
    T, C = 256, 1024
    W = np.zeros((6, C), dtype=np.float32)
    W[0, 5] = 1.0
    W[1, 300] = -2.0
    W[2, 0] = 0.5
    W[2, 1023] = 0.5
    W[4, 700] = 3.0
    codes, scales, signs, st = run_quantize(torch, L, W, "bf16", "e8", T, 9, 0.25)
    q = O.quantize(W, "e8", T, O.splitmix64_signs(9, C), 0.25)
    assert st == 0
    np.testing.assert_array_equal(codes, q.codes)
    np.testing.assert_array_equal(scales, q.scales)
    assert np.all(codes[3] == 0) and np.all(scales[3] == 0)


def test_nonfinite_and_range_flags():
    torch, L = cuda()
    W = gaussian_matrix(4, 512, 0.02, 1, dtype="fp32")
    W[1, 7] = np.nan
    W[2, 300] = np.inf
    _, _, _, st = run_quantize(torch, L, W, "fp32", "e8", 256, 0, 0.25)
    assert st & L.LQ_DEV_NONFINITE
    S = np.zeros((2, 256), dtype=np.float32)
    S[0, 3] = 1.0           # spike: code 2/beta = 200 at beta 0.01
    _, _, _, st = run_quantize(torch, L, S, "fp32", "e8", 256, 0, 0.01)
    assert st == L.LQ_DEV_RANGE
    q = O.quantize(S, "e8", 256, O.splitmix64_signs(0, 256), 0.01)
    assert q.range_error
    _, _, _, st = run_quantize(torch, L, S, "fp32", "e8", 256, 0, 0.05)   # code 40: in range
    assert st == 0


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_large_values_take_the_checked_decoder(lattice):
    """bf16 unit spikes at beta = 1/63 give |y| = 63 at every coordinate of their
    tile: every lane leaves the packed fast decoders for the range-checked scalar
    ones, the codes still fit int8 and equal the oracle's; at beta = 1/64 the
    codes would be 128 and the range flag is raised."""
    torch, L = cuda()
    S = np.zeros((4, 512), dtype=np.float32)      # one spike per tile; row 3 stays zero
    S[0, 3] = 1.0
    S[1, 300] = -1.0
    S[2, 17] = 1.0
    S[2, 400] = 1.0
    d = O.splitmix64_signs(0, 512)
    codes, scales, signs, st = run_quantize(torch, L, S, "bf16", lattice, 256, 0, 1.0 / 63.0)
    assert st == 0
    q = O.quantize(S, lattice, 256, d, 1.0 / 63.0)
    assert not q.range_error
    assert np.abs(q.codes).max() >= 120
    np.testing.assert_allclose(scales, q.scales, rtol=1e-6, atol=0)
    # these tiles are exactly symmetric (every |y| equal), so A2 meets exact
    # ties in many blocks: each differing block must be a certified tie
    compare_codes(codes, q, lattice, max_fraction=1.0)
    _, _, _, st = run_quantize(torch, L, S, "bf16", lattice, 256, 0, 1.0 / 64.0)
    assert st & L.LQ_DEV_RANGE


@pytest.mark.parametrize("lattice", ["e8", "z1", "d4"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("tile", [128, 512, 1024, 2048])
def test_large_value_tiles_among_zero_tiles_grouped(lattice, dtype, tile):
    """Single spikes of assorted sizes at beta = 1/63 (|y| = 63 over their tile)
    scattered among all-zero tiles of three matrices in one grouped launch, one
    with a padded row stride: the spike tiles go through the range-checked
    decoders, the zero tiles do not, and every matrix equals the oracle with no
    range flag."""
    torch, L = cuda()
    rng = np.random.default_rng(tile)
    shapes = [(9, 3 * tile), (3, 2048 + 2 * tile), (17, 4 * tile)]
    seeds = [5, 6, 7]
    beta = 1.0 / 63.0
    Ws, Wn = [], []
    for i, (r, c) in enumerate(shapes):
        W = np.zeros((r, c), dtype=np.float32)
        nt = c // tile
        for row in range(r):
            for t in range(nt):
                if rng.random() < 0.4:
                    W[row, t * tile + rng.integers(tile)] = rng.choice([1.0, -1.0, 3.0, -0.5, 96.0])
        pad = 16 if i == 1 else 0
        full = np.zeros((r, c + pad), dtype=np.float32)
        full[:, :c] = W
        Wd = to_dev_bf16(torch, full) if dtype == "bf16" else to_dev(torch, full)
        Ws.append(Wd[:, :c])
        Wn.append(W)
    codes, scales, signs, st = _grouped(torch, L, Ws, tile, seeds, beta, lattice)
    assert st == 0
    for m, W in enumerate(Wn):
        d = O.splitmix64_signs(seeds[m], W.shape[1])
        q = O.quantize(W, lattice, tile, d, beta)
        assert not q.range_error
        np.testing.assert_allclose(scales[m].cpu().numpy(), q.scales, rtol=1e-6, atol=0)
        compare_codes(codes[m].cpu().numpy(), q, lattice, max_fraction=1.0)
        assert np.abs(codes[m].cpu().numpy()).max() >= 120


def test_empty_rows_is_noop():
    torch, L = cuda()
    W = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    codes, scales, signs = L.quantize(W, tile=256)
    torch.cuda.synchronize()
    assert codes.shape == (0, 512)
    np.testing.assert_array_equal(signs.cpu().numpy(), O.splitmix64_signs(0, 512))


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 256, 512, 1024, 2048])
def test_dequantize_parity(lattice, tile):
    torch, L = cuda()
    rows, cols = 21, 2 * 2048 + 2 * tile
    W = gaussian_matrix(rows, cols, 0.02, 200 + tile, dtype="bf16")
    d = O.splitmix64_signs(3, cols)
    q = O.quantize(W, lattice, tile, d, 0.25)
    What = L.dequantize(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d),
                        lattice=lattice, tile=tile)
    ref = O.dequantize(q.codes, q.scales, d, tile, lattice)
    got = What.cpu().numpy()
    assert normwise_rel(got, ref) < 1e-6
    bf = L.dequantize(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d),
                      lattice=lattice, tile=tile, dtype=torch.bfloat16).float().cpu().numpy()
    assert normwise_rel(bf, ref) < 4e-3     # bf16 output rounding (2^-9 relative)


def test_full_size_gate_matrix_sampled():
    """Llama-3-8B gate_proj 14336 x 4096 bf16, E8, tile 256, beta 0.25, in one launch;
    oracle on 96 sampled rows; lattice membership of every block."""
    torch, L = cuda()
    W = gaussian_matrix(14336, 4096, 0.02, 1004, dtype="bf16")
    codes, scales, signs, st = run_quantize(torch, L, W, "bf16", "e8", 256, 1004, 0.25)
    assert st == 0
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, 14335], rng.choice(14336, 94, replace=False)]))
    q = O.quantize(W[rows], "e8", 256, O.splitmix64_signs(1004, 4096), 0.25)
    np.testing.assert_allclose(scales[rows], q.scales, rtol=1e-6)
    compare_codes(codes[rows], q, "e8")
    assert np.all(O.code_membership_ok("e8", codes.reshape(-1, 8).astype(np.int64)))


def test_stack_recipe_down_matrix_with_outliers_sampled():
    """down_proj 4096 x 14336 drawn on the device as in the 32-layer stack workload
    (N(0, 0.02^2), 0.1 % x20 outliers, bf16), E8, tile 256, beta 0.25, one launch;
    oracle on 64 sampled rows of the same bf16 values, then the batch-8 GEMV of the
    stack workload on the same rows."""
    torch, L = cuda()
    from synthetic import stack_seed, torch_gaussian_matrix
    seed = stack_seed(31, 6)
    Wd = torch_gaussian_matrix(4096, 14336, 0.02, seed, device="cuda", outlier_frac=0.001)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, signs = L.quantize(Wd, lattice="e8", tile=256, seed=seed, beta=0.25, dev_status=st)
    x = gaussian_vectors(8, 14336, 6008, dtype="bf16")
    y = L.gemv(codes, scales, signs, to_dev_bf16(torch, x), lattice="e8", tile=256, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([[0, 4095], rng.choice(4096, 62, replace=False)]))
    W = Wd[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert np.abs(W).max() > 0.2          # the sample holds outliers
    d = O.splitmix64_signs(seed, 14336)
    q = O.quantize(W, "e8", 256, d, 0.25)
    np.testing.assert_allclose(scales.cpu().numpy()[rows], q.scales, rtol=1e-6)
    compare_codes(codes.cpu().numpy()[rows], q, "e8")
    ref = O.gemv(q.codes, q.scales, d, 256, "e8", x)
    assert normwise_rel(y.cpu().numpy()[:, rows], ref) < 2e-3


def _grouped(torch, L, Ws, tile, seeds, beta, lattice):
    codes = [torch.empty(W.shape, dtype=torch.int8, device="cuda") for W in Ws]
    scales = [torch.empty((W.shape[0], W.shape[1] // tile), dtype=torch.float32, device="cuda") for W in Ws]
    signs = [torch.empty(W.shape[1], dtype=torch.int8, device="cuda") for W in Ws]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_quantize_grouped(lattice, Ws, tile, seeds, beta, codes, scales, signs, dev_status=st)
    torch.cuda.synchronize()
    return codes, scales, signs, int(st.item())


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_quantize_grouped_parity(lattice, dtype):
    """One grouped launch over matrices of different shapes (a ragged last chunk,
    several chunks per row, an empty matrix, a padded row stride): every matrix
    equals the oracle with its own seed, and the single-matrix call bit for bit."""
    torch, L = cuda()
    tile = 256
    shapes = [(37, 768), (0, 512), (64, 2304), (5, 256), (130, 4352), (19, 4096)]
    seeds = [11, 12, 2**63 + 5, 14, 15, 16]
    Ws, Wn = [], []
    for i, (r, c) in enumerate(shapes):
        W = gaussian_matrix(r, c, 0.02, 200 + i, outlier_frac=0.002, dtype="bf16")
        pad = 8 if i == 2 else 0
        full = np.zeros((r, c + pad), dtype=np.float32)
        full[:, :c] = W
        Wd = to_dev_bf16(torch, full) if dtype == "bf16" else to_dev(torch, full)
        Ws.append(Wd[:, :c])
        Wn.append(W)
    codes, scales, signs, st = _grouped(torch, L, Ws, tile, seeds, 0.25, lattice)
    any_range = False
    for m, W in enumerate(Wn):
        d = O.splitmix64_signs(seeds[m], W.shape[1])
        np.testing.assert_array_equal(signs[m].cpu().numpy(), d)
        if W.shape[0] == 0:
            continue
        q = O.quantize(W, lattice, tile, d, 0.25)
        any_range |= q.range_error
        np.testing.assert_allclose(scales[m].cpu().numpy(), q.scales, rtol=1e-6, atol=0)
        compare_codes(codes[m].cpu().numpy(), q, lattice)
        c1, s1, g1 = L.quantize(Ws[m], lattice=lattice, tile=tile, seed=seeds[m], beta=0.25)
        torch.cuda.synchronize()
        assert torch.equal(c1, codes[m]) and torch.equal(s1, scales[m]) and torch.equal(g1, signs[m])
    assert st == (2 if any_range else 0)


def test_quantize_grouped_layer_matches_single_calls():
    """The seven Llama-3-8B layer matrices (bf16, seeds 1000 + index) in one grouped
    launch equal seven single-matrix launches bit for bit; oracle on sampled rows
    of the down projection (the group's only 7-chunk rows)."""
    torch, L = cuda()
    from synthetic import LLAMA3_8B_LAYER, torch_gaussian_matrix
    Ws = [torch_gaussian_matrix(r, c, 0.02, 1000 + i, device="cuda") for i, (_, r, c) in enumerate(LLAMA3_8B_LAYER)]
    seeds = [1000 + i for i in range(len(Ws))]
    codes, scales, signs, st = _grouped(torch, L, Ws, 256, seeds, 0.25, "e8")
    assert st == 0
    for m, W in enumerate(Ws):
        c1, s1, g1 = L.quantize(W, lattice="e8", tile=256, seed=seeds[m], beta=0.25)
        torch.cuda.synchronize()
        assert torch.equal(c1, codes[m]) and torch.equal(s1, scales[m]) and torch.equal(g1, signs[m])
        del c1, s1, g1
    rng = np.random.default_rng(2)
    rows = np.sort(np.concatenate([[0, 4095], rng.choice(4096, 30, replace=False)]))
    Wd = Ws[6][torch.from_numpy(rows).cuda()].float().cpu().numpy()
    q = O.quantize(Wd, "e8", 256, O.splitmix64_signs(seeds[6], 14336), 0.25)
    np.testing.assert_allclose(scales[6].cpu().numpy()[rows], q.scales, rtol=1e-6)
    compare_codes(codes[6].cpu().numpy()[rows], q, "e8")


@pytest.mark.parametrize("tile", [256, 2048])
def test_maximum_width_rows(tile):
    """cols = 2^20, the widest row the ABI takes (512 chunks per row): quantize,
    dequantize and the batch-16 GEMV against the oracle on the whole matrix."""
    torch, L = cuda()
    rows, cols = 3, 1 << 20
    W = gaussian_matrix(rows, cols, 0.02, 610 + tile, outlier_frac=0.001, dtype="bf16")
    codes, scales, signs, st = run_quantize(torch, L, W, "bf16", "e8", tile, 611, 0.25)
    d = O.splitmix64_signs(611, cols)
    q = O.quantize(W, "e8", tile, d, 0.25)
    assert st == 0
    np.testing.assert_allclose(scales, q.scales, rtol=1e-6)
    compare_codes(codes, q, "e8")
    What = L.dequantize(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d), lattice="e8", tile=tile)
    assert normwise_rel(What.cpu().numpy(), O.dequantize(q.codes, q.scales, d, tile, "e8")) < 1e-6
    x = gaussian_vectors(16, cols, 612, dtype="bf16")
    y = L.gemv(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d), to_dev_bf16(torch, x),
               lattice="e8", tile=tile)
    torch.cuda.synchronize()
    assert normwise_rel(y.cpu().numpy(), O.gemv(q.codes, q.scales, d, tile, "e8", x)) < 2e-3


def test_quantize_grouped_with_a_maximum_width_matrix():
    """A group whose chunks-per-row counts (512 and 2) have a least common
    multiple above 64: the warps then change chunk from unit to unit (the
    signs are reloaded); every matrix still equals the oracle."""
    torch, L = cuda()
    shapes = [(3, 1 << 20), (5, 4096), (2, 2048 * 3 + 256)]
    seeds = [21, 22, 23]
    Wn = [gaussian_matrix(r, c, 0.02, 620 + i, dtype="bf16") for i, (r, c) in enumerate(shapes)]
    Ws = [to_dev_bf16(torch, W) for W in Wn]
    codes, scales, signs, st = _grouped(torch, L, Ws, 256, seeds, 0.25, "e8")
    assert st == 0
    for m, W in enumerate(Wn):
        d = O.splitmix64_signs(seeds[m], W.shape[1])
        q = O.quantize(W, "e8", 256, d, 0.25)
        np.testing.assert_array_equal(signs[m].cpu().numpy(), d)
        np.testing.assert_allclose(scales[m].cpu().numpy(), q.scales, rtol=1e-6)
        compare_codes(codes[m].cpu().numpy(), q, "e8")
