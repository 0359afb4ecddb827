"""GPU Rice format (encoder, decoder, GEMV from the stream) against the CPU oracle."""
import numpy as np
import pytest

import oracle as O
import oracle.rice_oracle as R
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def gpu_encode(torch, L, codes_dev, lattice, tile, status=None):
    rows, cols = codes_dev.shape
    nbytes = L.lq_rice_stream_bound(lattice, rows, cols, tile)
    words = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    offs = torch.empty((rows, cols // tile), dtype=torch.int32, device="cuda")
    total = torch.empty(1, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(1, L.lq_rice_workspace_size(rows, cols, tile)), dtype=torch.uint8, device="cuda")
    L.lq_rice_encode(lattice, codes_dev, tile, words, offs, total, ws, status)
    torch.cuda.synchronize()
    return words, offs, int(total.item())


def u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 256, 2048])
def test_encode_matches_oracle_bit_exact(lattice, tile):
    torch, L = cuda()
    rows, cols = 9, 2 * tile if tile == 2048 else 3 * tile
    W = gaussian_matrix(rows, cols, 0.02, 500 + tile, outlier_frac=0.005, dtype="bf16")
    q = O.quantize(W, lattice, tile, O.splitmix64_signs(9, cols), 0.25)
    codes = q.codes.astype(np.int8)
    ref_words, ref_offs, ref_total = R.encode(q.codes, lattice, tile)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    words, offs, total = gpu_encode(torch, L, to_dev(torch, codes), lattice, tile, st)
    assert int(st.item()) == 0
    assert total == ref_total
    assert np.array_equal(u32(offs), ref_offs)
    w = u32(words)
    nw = len(ref_words)
    assert np.array_equal(w[:nw], ref_words)
    assert not w[nw:].any()
    # decode of the GPU stream and of the oracle stream give the codes back
    out = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    L.lq_rice_decode(lattice, words, offs, tile, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), codes)
    ow = torch.from_numpy(np.concatenate([ref_words, np.zeros(4, np.uint32)]).view(np.int32)).cuda()
    oo = torch.from_numpy(ref_offs.view(np.int32)).cuda()
    out.zero_()
    L.lq_rice_decode(lattice, ow, oo, tile, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), codes)


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile", [128, 256, 1024])
@pytest.mark.parametrize("batch", [1, 5, 16])
def test_gemv_rice_parity(lattice, tile, batch):
    torch, L = cuda()
    rows, cols = 75, 2048 + tile
    W = gaussian_matrix(rows, cols, 0.02, 600 + tile, dtype="bf16")
    d = O.splitmix64_signs(11, cols)
    q = O.quantize(W, lattice, tile, d, 0.25)
    words, offs, _ = gpu_encode(torch, L, to_dev(torch, q.codes.astype(np.int8)), lattice, tile)
    x = gaussian_vectors(batch, cols, 700 + batch, dtype="bf16")
    y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_gemv_workspace_size(batch, cols, tile), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_gemv_rice(lattice, words, offs, to_dev(torch, q.scales), to_dev(torch, d), tile, to_dev_bf16(torch, x),
                   y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.gemv(q.codes, q.scales, d, tile, lattice, x)
    assert normwise_rel(y.cpu().numpy(), ref) < 2e-3


def _crafted_codes(lattice, rows, cols, seed):
    """Codes with the pinned bits of the lattice: most blocks in {-1, 0, 1}
    halves (a small Rice parameter), 5 % of the blocks with halves up to +-62
    (unary runs far longer than a 32-bit word), and every fourth row made only
    of the large blocks, so that rows advance through the stream at very
    different rates."""
    n = {"e8": 8, "d4": 4, "a2": 2, "z1": 1}[lattice]
    parity = lattice in ("e8", "a2")
    even = lattice in ("e8", "d4")
    rng = np.random.default_rng(seed)
    C = np.zeros((rows, cols), np.int64)
    for r in range(rows):
        frac = 1.0 if r % 4 == 3 else 0.05
        for b0 in range(0, cols, n):
            k = int(rng.integers(0, 2)) if parity else 0
            if rng.random() < frac:
                u = rng.integers(-62, 62, n)
            else:
                u = rng.integers(-1, 2, n)
            if even and u.sum() % 2:
                u[-1] += 1 if u[-1] < 60 else -1
            C[r, b0:b0 + n] = 2 * u + k
    return C


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tile,batch", [(128, 1), (256, 9), (512, 3)])
def test_gemv_rice_long_runs_and_uneven_rows(lattice, tile, batch):
    """Unary runs longer than the decoder's 32-bit window and rows of very
    different stream rates: the stream decodes back to the codes and the GEMV
    from the stream matches the oracle's GEMV of the codes."""
    torch, L = cuda()
    rows, cols = 70, 3 * tile
    codes = _crafted_codes(lattice, rows, cols, 900 + tile)
    assert np.abs(codes).max() >= 100
    rng = np.random.default_rng(901)
    scales = rng.uniform(0.5, 2.0, (rows, cols // tile)).astype(np.float32)
    d = O.splitmix64_signs(13, cols)
    words, offs, _ = gpu_encode(torch, L, to_dev(torch, codes.astype(np.int8)), lattice, tile)
    out = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    L.lq_rice_decode(lattice, words, offs, tile, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), codes.astype(np.int8))
    x = gaussian_vectors(batch, cols, 902 + batch, dtype="bf16")
    y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_gemv_workspace_size(batch, cols, tile), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_gemv_rice(lattice, words, offs, to_dev(torch, scales), to_dev(torch, d), tile,
                   to_dev_bf16(torch, x), y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.gemv(codes, scales, d, tile, lattice, x)
    assert normwise_rel(y.cpu().numpy(), ref) < 2e-3


def test_format_flag_on_codes_without_pinned_bits():
    """E8 blocks of mixed parity cannot be stripped: the encoder flags them."""
    torch, L = cuda()
    codes = np.zeros((2, 256), dtype=np.int8)
    codes[1, 8:16] = [1, 2, 1, 1, 1, 1, 1, 0]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_encode(torch, L, to_dev(torch, codes), "e8", 256, st)
    assert int(st.item()) & L.LQ_DEV_FORMAT


def test_full_size_gate_round_trip_and_rate():
    """gate_proj 14336 x 4096 (E8, tile 256, beta 0.25): quantize, encode, decode gives
    the codes back bit for bit; sampled segments equal the oracle's bits; the rate is
    near 4 bits per weight; the GEMV from the stream equals the GEMV from the codes."""
    torch, L = cuda()
    from synthetic import torch_gaussian_matrix
    rows, cols, tile = 14336, 4096, 256
    Wd = torch_gaussian_matrix(rows, cols, 0.02, 1004, device="cuda")
    codes, scales, signs = L.quantize(Wd, lattice="e8", tile=tile, seed=1004, beta=0.25)
    words, offs, total = gpu_encode(torch, L, codes, "e8", tile)
    bps = total / (rows * cols)
    assert 3.7 < bps < 4.7, bps
    out = torch.empty_like(codes)
    L.lq_rice_decode("e8", words, offs, tile, out)
    torch.cuda.synchronize()
    assert torch.equal(out, codes)
    w = u32(words)
    o = u32(offs)
    rng = np.random.default_rng(2)
    for r in rng.choice(rows, 24, replace=False):
        t = int(rng.integers(0, cols // tile))
        ref = R.segment_bits("e8", codes[r, t * tile:(t + 1) * tile].cpu().numpy().astype(np.int64).tolist())
        pos = int(o[r, t])
        got = [(int(w[(pos + i) >> 5]) >> ((pos + i) & 31)) & 1 for i in range(len(ref))]
        assert got == ref
    for batch in (1, 16):
        x = torch.randn((batch, cols), device="cuda").to(torch.bfloat16)
        y8 = L.gemv(codes, scales, signs, x, lattice="e8", tile=tile)
        yr = torch.empty_like(y8)
        ws = torch.empty(L.lq_gemv_workspace_size(batch, cols, tile), dtype=torch.uint8, device="cuda")
        L.lq_gemv_rice("e8", words, offs, scales, signs, tile, x, yr, ws)
        torch.cuda.synchronize()
        assert normwise_rel(yr.cpu().numpy(), y8.cpu().numpy()) < 1e-6
