"""GPU prefill GEMM (tcgen05) from lattice codes against the float64 oracle.

Codes and scales come from the oracle; X is bf16.  The GEMM rounds X~ and the
decoded weights to fp16 (each scaled by a power of two), so the normwise error
budget is well inside the 2e-3 tolerance."""
import numpy as np
import pytest

import oracle as O
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

TOL = 2e-3


def gpu_gemm(torch, L, q, d, X, lattice, tile):
    Xd = to_dev_bf16(torch, X)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = L.gemm(to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d), Xd,
               lattice=lattice, tile=tile, dev_status=status)
    torch.cuda.synchronize()
    return Y.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("M,N,K", [(37, 256, 256), (300, 256, 1024), (256, 384, 2048), (1, 128, 512)])
def test_gemm_parity_e8(M, N, K):
    """K = 256 runs one K split; longer K splits across CTAs (atomic accumulation)."""
    torch, L = cuda()
    W = gaussian_matrix(N, K, 0.015, 50 + M, dtype="bf16")
    d = O.splitmix64_signs(21, K)
    q = O.quantize(W, "e8", 256, d, 0.25)
    X = gaussian_vectors(M, K, 60 + M, dtype="bf16")
    Y, st = gpu_gemm(torch, L, q, d, X, "e8", 256)
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    assert st == 0
    rel = normwise_rel(Y, ref)
    assert rel < TOL, rel
    assert rel < 1e-3


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 512, 1024, 2048])
def test_gemm_parity_lattices_tiles(lattice, tile):
    torch, L = cuda()
    M, N, K = 70, 128, max(1024, 2 * tile)
    W = gaussian_matrix(N, K, 0.02, 7, dtype="bf16")
    d = O.splitmix64_signs(8, K)
    q = O.quantize(W, lattice, tile, d, 0.25)
    X = gaussian_vectors(M, K, 9, dtype="bf16")
    Y, st = gpu_gemm(torch, L, q, d, X, lattice, tile)
    ref = O.gemm(q.codes, q.scales, d, tile, lattice, X)
    assert st == 0
    assert normwise_rel(Y, ref) < TOL


def test_gemm_activation_scales_and_zero_rows():
    torch, L = cuda()
    M, N, K = 8, 128, 512
    W = gaussian_matrix(N, K, 0.02, 3, dtype="bf16")
    d = O.splitmix64_signs(4, K)
    q = O.quantize(W, "e8", 256, d, 0.25)
    X = gaussian_vectors(M, K, 5, dtype="bf16")
    X[1] = 0.0
    X[2] *= 1e-20
    X[3] *= 1e15
    Y, st = gpu_gemm(torch, L, q, d, X, "e8", 256)
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    assert st == 0
    assert np.all(Y[1] == 0.0)
    for m in (0, 2, 3, 4):
        assert normwise_rel(Y[m], ref[m]) < TOL


def test_gemm_full_size_sampled_rows():
    """Llama-3-70B up-like shape: W 8192 x 28672 (E8, tile 256), X 256 x 28672 bf16.
    Codes of 32 sampled weight rows come from the oracle; the rest from the GPU quantizer."""
    torch, L = cuda()
    N, K, M = 8192, 28672, 256
    g = torch.Generator(device="cuda").manual_seed(4000)
    Wd = (torch.randn((N, K), device="cuda", generator=g) * 0.015).to(torch.bfloat16)
    codes, scales, signs = L.quantize(Wd, lattice="e8", tile=256, seed=4000, beta=0.25)
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(N, 32, replace=False))
    Wrows = Wd[torch.from_numpy(rows).to("cuda")].float().cpu().numpy()
    del Wd
    d = O.splitmix64_signs(4000, K)
    q = O.quantize(Wrows, "e8", 256, d, 0.25)
    ridx = torch.from_numpy(rows).to("cuda")
    codes[ridx] = to_dev(torch, q.codes)
    scales[ridx] = to_dev(torch, q.scales)
    X = gaussian_vectors(M, K, 4100 + M, dtype="bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = L.gemm(codes, scales, signs, to_dev_bf16(torch, X), lattice="e8", tile=256, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    assert normwise_rel(Y.cpu().numpy()[:, rows], ref) < TOL
