"""GPU GEMV from lattice codes against the float64 oracle (codes from the oracle)."""
import numpy as np
import pytest

import oracle as O
from synthetic import gaussian_matrix, gaussian_vectors, small_fp32_case
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3   # normwise relative error of y against the float64 oracle on the same codes


def gpu_gemv(torch, L, q, d, x, lattice, tile, xdtype):
    xd = to_dev_bf16(torch, x) if xdtype == "bf16" else to_dev(torch, x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = L.gemv(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d), xd,
               lattice=lattice, tile=tile, dev_status=status)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(status.item())


def test_small_fp32_case_gemv():
    torch, L = cuda()
    W, x = small_fp32_case(0)
    d = O.splitmix64_signs(0, 1024)
    q = O.quantize(W, "e8", 256, d, 0.25)
    y, st = gpu_gemv(torch, L, q, d, x, "e8", 256, "fp32")
    ref = O.gemv(q.codes, q.scales, d, 256, "e8", x)
    assert st == 0
    assert normwise_rel(y, ref) < TOL
    # fp16 activation: 2^-11 relative per element, about 3e-4 normwise on y
    assert normwise_rel(y, ref) < 1e-3


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 256, 512, 1024, 2048])
@pytest.mark.parametrize("batch", [1, 3, 8, 16])
def test_gemv_parity(lattice, tile, batch):
    torch, L = cuda()
    # ragged rows and (tiles up to 1024) a partial 2048-column chunk
    rows, cols = 75, (2048 + 2 * tile) if tile <= 512 else 3 * tile
    W = gaussian_matrix(rows, cols, 0.02, 300 + tile, dtype="bf16")
    d = O.splitmix64_signs(11, cols)
    q = O.quantize(W, lattice, tile, d, 0.25)
    x = gaussian_vectors(batch, cols, 400 + batch, dtype="bf16")
    y, st = gpu_gemv(torch, L, q, d, x, lattice, tile, "bf16")
    ref = O.gemv(q.codes, q.scales, d, tile, lattice, x)
    assert st == 0
    rel = normwise_rel(y, ref)
    assert rel < TOL, rel
    assert np.max(np.abs(y - ref)) <= TOL * np.max(np.abs(ref)) + 1e-12


def test_gemv_extreme_activation_scales():
    """Per-tile power-of-two scaling keeps the fp16 activation accurate for tiny and huge x."""
    torch, L = cuda()
    W = gaussian_matrix(64, 1024, 0.02, 5, dtype="bf16")
    d = O.splitmix64_signs(2, 1024)
    q = O.quantize(W, "e8", 256, d, 0.25)
    x = gaussian_vectors(4, 1024, 6, dtype="fp32")
    x[1] *= 1e-12
    x[2] *= 1e12
    x[3, :256] = 0.0
    y, st = gpu_gemv(torch, L, q, d, x, "e8", 256, "fp32")
    ref = O.gemv(q.codes, q.scales, d, 256, "e8", x)
    assert st == 0
    for b in range(4):
        assert normwise_rel(y[b], ref[b]) < 1e-3


def test_gemv_nonfinite_activation_flag():
    torch, L = cuda()
    W = gaussian_matrix(16, 512, 0.02, 5, dtype="bf16")
    d = O.splitmix64_signs(2, 512)
    q = O.quantize(W, "e8", 256, d, 0.25)
    x = gaussian_vectors(1, 512, 6, dtype="fp32")
    x[0, 10] = np.inf
    _, st = gpu_gemv(torch, L, q, d, x, "e8", 256, "fp32")
    assert st & L.LQ_DEV_NONFINITE


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_full_size_down_matrix_sampled_rows(batch):
    """down_proj 4096 x 14336 (E8, tile 256) in the launch shape the bench times: the
    codes of 64 sampled rows come from the oracle, the rest from the GPU quantizer."""
    torch, L = cuda()
    R, C = 4096, 14336
    W = gaussian_matrix(R, C, 0.02, 1006, dtype="bf16")
    Wd = to_dev_bf16(torch, W)
    codes, scales, signs = L.quantize(Wd, lattice="e8", tile=256, seed=1006, beta=0.25)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(R, 64, replace=False))
    d = O.splitmix64_signs(1006, C)
    q = O.quantize(W[rows], "e8", 256, d, 0.25)
    ridx = torch.from_numpy(rows).to("cuda")
    codes[ridx] = to_dev(torch, q.codes)
    scales[ridx] = to_dev(torch, q.scales)
    x = gaussian_vectors(batch, C, 2000 + batch, dtype="bf16")
    y = L.gemv(codes, scales, signs, to_dev_bf16(torch, x), lattice="e8", tile=256)
    torch.cuda.synchronize()
    ref = O.gemv(q.codes, q.scales, d, 256, "e8", x)
    assert normwise_rel(y.cpu().numpy()[:, rows], ref) < TOL


@pytest.mark.parametrize("tile", [128, 256, 2048])
@pytest.mark.parametrize("batch", [1, 5, 16])
def test_grouped_gemv_parity(tile, batch):
    """Three matrices of different heights (one without rows) sharing x, each with
    its own signs and scales, in one grouped call: each y against the oracle."""
    torch, L = cuda()
    cols = 2 * tile if tile >= 1024 else 2048 + tile
    heights = [75, 0, 130, 33]
    mats, refs = [], []
    x = gaussian_vectors(batch, cols, 900 + batch, dtype="bf16")
    for k, rows in enumerate(heights):
        W = gaussian_matrix(max(rows, 1), cols, 0.02, 910 + k, dtype="bf16")[:rows]
        d = O.splitmix64_signs(920 + k, cols)
        q = O.quantize(W, "e8", tile, d, 0.25)
        mats.append((to_dev(torch, q.codes.reshape(rows, cols)), to_dev(torch, q.scales.reshape(rows, cols // tile)),
                     to_dev(torch, d)))
        refs.append(O.gemv(q.codes, q.scales, d, tile, "e8", x) if rows else None)
    ys = [torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda") for rows in heights]
    ws = torch.empty(L.lq_gemv_grouped_workspace_size(len(mats), batch, cols, tile), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_gemv_grouped("e8", [m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], tile,
                      to_dev_bf16(torch, x), ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for y, ref in zip(ys, refs):
        if ref is not None:
            assert normwise_rel(y.cpu().numpy(), ref) < TOL


def test_grouped_gemv_matches_single_calls():
    """Grouping merges launches only: q/k/v-shaped matrices (4096, 1024, 1024 rows x
    4096) give the results of three lq_gemv calls (to fp32 summation order)."""
    torch, L = cuda()
    from synthetic import torch_gaussian_matrix
    cols, tile = 4096, 256
    mats = []
    for k, rows in enumerate((4096, 1024, 1024)):
        W = torch_gaussian_matrix(rows, cols, 0.02, 930 + k, device="cuda")
        mats.append(L.quantize(W, lattice="e8", tile=tile, seed=930 + k, beta=0.25))
    x = torch.randn((4, cols), device="cuda").to(torch.bfloat16)
    singles = [L.gemv(c, s, g, x, lattice="e8", tile=tile) for c, s, g in mats]
    ys = [torch.empty((4, c.shape[0]), dtype=torch.float32, device="cuda") for c, _, _ in mats]
    ws = torch.empty(L.lq_gemv_grouped_workspace_size(3, 4, cols, tile), dtype=torch.uint8, device="cuda")
    L.lq_gemv_grouped("e8", [m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], tile, x, ys, ws)
    torch.cuda.synchronize()
    for y, y1 in zip(ys, singles):
        assert normwise_rel(y.cpu().numpy(), y1.cpu().numpy()) < 1e-6


@pytest.mark.parametrize("batch", [1, 5, 16])
def test_chained_calls_read_the_previous_results(batch):
    """Back-to-back calls on one stream, no synchronisation between them: the
    weights of the second product are quantized right before it, and its
    activation is the first product's output (fp32).  The activation rotation
    of each call waits for the grid before it, so the second product sees the
    finished y1 and codes; checked over repeated chains against the float64
    oracle on the codes and y1 the GPU produced."""
    torch, L = cuda()
    tile = 256
    WA = gaussian_matrix(1024, 2048, 0.02, 61, dtype="bf16")
    dA = O.splitmix64_signs(61, 2048)
    qA = O.quantize(WA, "e8", tile, dA, 0.25)
    cA, sA, gA = to_dev(torch, qA.codes), to_dev(torch, qA.scales), to_dev(torch, dA)
    WB = to_dev_bf16(torch, gaussian_matrix(768, 1024, 0.02, 62, dtype="bf16"))
    x0 = gaussian_vectors(batch, 2048, 63, dtype="bf16")
    x0d = to_dev_bf16(torch, x0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    runs = []
    for it in range(6):
        y1 = L.gemv(cA, sA, gA, x0d, lattice="e8", tile=tile, dev_status=status)
        cB, sB, gB = L.quantize(WB, lattice="e8", tile=tile, seed=64 + it, beta=0.25, dev_status=status)
        y2 = L.gemv(cB, sB, gB, y1, lattice="e8", tile=tile, dev_status=status)
        runs.append((y1, cB, sB, gB, y2))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref1 = O.gemv(qA.codes, qA.scales, dA, tile, "e8", x0)
    for it, (y1, cB, sB, gB, y2) in enumerate(runs):
        y1h = y1.cpu().numpy()
        assert normwise_rel(y1h, ref1) < TOL
        np.testing.assert_array_equal(gB.cpu().numpy(), O.splitmix64_signs(64 + it, 1024))
        ref2 = O.gemv(cB.cpu().numpy(), sB.cpu().numpy(), gB.cpu().numpy(), tile, "e8", y1h)
        rel = normwise_rel(y2.cpu().numpy(), ref2)
        assert rel < TOL, (it, rel)
