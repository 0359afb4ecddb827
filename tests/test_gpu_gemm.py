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


@pytest.mark.parametrize("N,K,M", [(8192, 28672, 256), (8192, 28672, 2048), (28672, 8192, 256),
                                   (28672, 8192, 2048)])
def test_gemm_full_size_sampled_rows(N, K, M):
    """The Llama-3-70B MLP shapes the benchmark times: up-like W 8192 x 28672 and
    down-like W 28672 x 8192 (E8, tile 256), X M x K bf16 at M = 256 and 2048 --
    each in the launch configuration the benchmark uses (K split and tile
    counts follow from the shape).  Codes of 32 sampled weight rows come from
    the oracle, the rest from the GPU quantizer; Y is compared on those rows."""
    torch, L = cuda()
    seed = 4000 if N == 8192 else 4001
    g = torch.Generator(device="cuda").manual_seed(seed)
    Wd = (torch.randn((N, K), device="cuda", generator=g) * 0.015).to(torch.bfloat16)
    codes, scales, signs = L.quantize(Wd, lattice="e8", tile=256, seed=seed, beta=0.25)
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(N, 32, replace=False))
    Wrows = Wd[torch.from_numpy(rows).to("cuda")].float().cpu().numpy()
    del Wd
    d = O.splitmix64_signs(seed, K)
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
    got = Y[:, ridx].cpu().numpy()
    assert normwise_rel(got, ref) < TOL
    # every output is finite and the unsampled rows are of the same size
    assert bool(torch.isfinite(Y).all())


@pytest.mark.parametrize("N,K,M", [(200, 1024, 37), (4100, 512, 300), (130, 2048, 1), (1, 256, 5)])
def test_gemm_ragged_weight_rows(N, K, M):
    """N that is not a multiple of the 128-row weight tile: the last tile's
    missing rows are the TMA's zero fill and write nothing."""
    torch, L = cuda()
    W = gaussian_matrix(N, K, 0.02, 90 + N, dtype="bf16")
    d = O.splitmix64_signs(91, K)
    q = O.quantize(W, "e8", 256, d, 0.25)
    X = gaussian_vectors(M, K, 92 + M, dtype="bf16")
    Xd = to_dev_bf16(torch, X)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(L.lq_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    # Y inside a larger buffer: nothing may land past its M x N floats
    buf = torch.full((M * N + 4096,), 7.0, dtype=torch.float32, device="cuda")
    Y = buf[:M * N].view(M, N)
    L.lq_gemm("e8", to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d), 256, Xd, Y, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool((buf[M * N:] == 7.0).all())
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    assert normwise_rel(Y.cpu().numpy(), ref) < TOL


def _bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), np.float32(1e-30))
    return np.exp2(np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("N,K,M", [(256, 1024, 37), (200, 4096, 300), (8192, 28672, 256)])
def test_gemm_bf16_output(N, K, M):
    """bf16 Y (the page's output type): the float32 result rounded to nearest
    even.  Bound against the fp64 oracle: 2e-3 (the float32 path's bar) plus
    2^-8, the unit roundoff of bf16, normwise.  Against the float32 output of
    the same call: equal after rounding, or one bf16 step apart where a
    K-split launch added its float32 partial sums in another order."""
    torch, L = cuda()
    if N == 8192:
        g = torch.Generator(device="cuda").manual_seed(4000)
        Wd = (torch.randn((N, K), device="cuda", generator=g) * 0.015).to(torch.bfloat16)
        codes, scales, signs = L.quantize(Wd, lattice="e8", tile=256, seed=4000, beta=0.25)
        rows = np.sort(np.random.default_rng(5).choice(N, 16, replace=False))
        Wrows = Wd[torch.from_numpy(rows).to("cuda")].float().cpu().numpy()
        del Wd
        d = O.splitmix64_signs(4000, K)
        q = O.quantize(Wrows, "e8", 256, d, 0.25)
        ridx = torch.from_numpy(rows).to("cuda")
        codes[ridx] = to_dev(torch, q.codes)
        scales[ridx] = to_dev(torch, q.scales)
    else:
        W = gaussian_matrix(N, K, 0.02, 95, dtype="bf16")
        d = O.splitmix64_signs(96, K)
        q = O.quantize(W, "e8", 256, d, 0.25)
        codes, scales, signs = to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d)
        rows = np.arange(N)
        ridx = torch.arange(N, device="cuda")
    X = gaussian_vectors(M, K, 97 + M, dtype="bf16")
    Xd = to_dev_bf16(torch, X)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Yb = L.gemm(codes, scales, signs, Xd, lattice="e8", tile=256, dev_status=status, out_dtype=torch.bfloat16)
    Yf = L.gemm(codes, scales, signs, Xd, lattice="e8", tile=256, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert Yb.dtype == torch.bfloat16
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    gb = Yb[:, ridx].float().cpu().numpy()
    assert normwise_rel(gb, ref) < TOL + 2.0 ** -8
    yf = Yf.cpu().numpy()
    yb = Yb.float().cpu().numpy()
    rounded = Yf.to(torch.bfloat16).float().cpu().numpy()
    diff = np.abs(yb - rounded)
    # one bf16 step, measured in the larger binade where the two straddle a power of two;
    # plus the float32 summation-order noise of a K-split launch (its partial sums are
    # added by atomics in any order), which near a cancellation can exceed the bf16 step
    # of a tiny result: 2^-20 of the output's scale bounds it with room to spare
    step = _bf16_ulp(np.maximum(np.abs(yb), np.abs(rounded)))
    noise = 2.0 ** -20 * np.max(np.abs(yf))
    excess = diff - (step * 1.0001 + noise)
    assert np.all(excess <= 0), (float(excess.max()), float(diff.max()))


def test_gemm_wait_expiry_reports_timeout_and_recovers():
    """A bounded wait that runs out: the self-test variant of the GEMM kernel has
    an activation producer that never fills its ring and a ~0.1 ms wait limit.
    The call must come back with LQ_DEV_TIMEOUT in the status word (not hang),
    and an ordinary GEMM on the same stream afterwards must still match the
    oracle (tensor memory released, context usable)."""
    torch, L = cuda()
    M, N, K = 70, 256, 1024
    W = gaussian_matrix(N, K, 0.02, 31, dtype="bf16")
    d = O.splitmix64_signs(32, K)
    q = O.quantize(W, "e8", 256, d, 0.25)
    X = gaussian_vectors(M, K, 33, dtype="bf16")
    codes, scales, signs = to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d)
    Xd = to_dev_bf16(torch, X)
    ws = torch.empty(L.lq_gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    for _ in range(2):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        L.lq_gemm_wait_expiry_test("e8", codes, scales, signs, 256, Xd, Y, ws, status)
        torch.cuda.synchronize()
        assert int(status.item()) & L.LQ_DEV_TIMEOUT
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_gemm("e8", codes, scales, signs, 256, Xd, Y, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.gemm(q.codes, q.scales, d, 256, "e8", X)
    assert normwise_rel(Y.cpu().numpy(), ref) < TOL
