"""Guard bytes around every output and workspace buffer: no entry point writes
outside the sizes include/lq.h gives it."""
import numpy as np
import pytest

import oracle as O
import oracle.kv_oracle as KV
from synthetic import gaussian_matrix, gaussian_vectors
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
GUARD = 512           # bytes on each side (keeps 256-byte alignment)
CANARY = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer whose edges are canaries."""

    def __init__(self, torch, shape, dtype, nbytes=None):
        elem = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if shape else 1
        self.nbytes = nbytes if nbytes is not None else n * elem
        self.raw = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n * elem].view(dtype).view(shape) if shape else None
        self.bytes_view = self.raw[GUARD:GUARD + self.nbytes]

    def intact(self):
        lo = self.raw[:GUARD].cpu().numpy()
        hi = self.raw[GUARD + self.nbytes:].cpu().numpy()
        return bool((lo == CANARY).all() and (hi == CANARY).all())


def test_quantize_dequantize_gemv_gemm_stay_in_bounds():
    torch, L = cuda()
    rows, cols, T = 37, 1536, 512
    W = to_dev_bf16(torch, gaussian_matrix(rows, cols, 0.02, 1, dtype="bf16"))
    codes = Guarded(torch, (rows, cols), torch.int8)
    scales = Guarded(torch, (rows, cols // T), torch.float32)
    signs = Guarded(torch, (cols,), torch.int8)
    L.lq_quantize("e8", W, T, 5, 0.25, codes.t, scales.t, signs.t)
    Wh = Guarded(torch, (rows, cols), torch.float32)
    L.lq_dequantize("e8", codes.t, scales.t, signs.t, T, Wh.t)
    x = to_dev_bf16(torch, gaussian_vectors(3, cols, 2, dtype="bf16"))
    y = Guarded(torch, (3, rows), torch.float32)
    wsz = L.lq_gemv_workspace_size(3, cols, T)
    ws = Guarded(torch, (wsz,), torch.uint8)
    L.lq_gemv("e8", codes.t, scales.t, signs.t, T, x, y.t, ws.t)
    ys = [Guarded(torch, (3, rows), torch.float32) for _ in range(2)]
    gws = Guarded(torch, (L.lq_gemv_grouped_workspace_size(2, 3, cols, T),), torch.uint8)
    L.lq_gemv_grouped("e8", [codes.t, codes.t], [scales.t, scales.t], [signs.t, signs.t], T, x, [g.t for g in ys],
                      gws.t)
    # GEMM needs N % 128 == 0
    Wg = to_dev_bf16(torch, gaussian_matrix(256, 1024, 0.02, 3, dtype="bf16"))
    gc, gs, gsg = L.quantize(Wg, lattice="e8", tile=256, seed=6, beta=0.25)
    X = to_dev_bf16(torch, gaussian_vectors(37, 1024, 4, dtype="bf16"))
    Y = Guarded(torch, (37, 256), torch.float32)
    gw = Guarded(torch, (L.lq_gemm_workspace_size(37, 256, 1024),), torch.uint8)
    L.lq_gemm("e8", gc, gs, gsg, 256, X, Y.t, gw.t)
    torch.cuda.synchronize()
    for g in [codes, scales, signs, Wh, y, ws, *ys, gws, Y, gw]:
        assert g.intact()


def test_rice_attention_rotation_stay_in_bounds():
    torch, L = cuda()
    rows, cols, T = 33, 1024, 256
    W = to_dev_bf16(torch, gaussian_matrix(rows, cols, 0.02, 7, dtype="bf16"))
    codes, scales, signs = L.quantize(W, lattice="e8", tile=T, seed=8, beta=0.25)
    nb = L.lq_rice_stream_bound("e8", rows, cols, T)
    words = Guarded(torch, (nb // 4,), torch.int32)
    offs = Guarded(torch, (rows, cols // T), torch.int32)
    total = Guarded(torch, (1,), torch.int64)
    rws = Guarded(torch, (L.lq_rice_workspace_size(rows, cols, T),), torch.uint8)
    L.lq_rice_encode("e8", codes, T, words.t, offs.t, total.t, rws.t)
    dec = Guarded(torch, (rows, cols), torch.int8)
    L.lq_rice_decode("e8", words.t, offs.t, T, dec.t)
    x = to_dev_bf16(torch, gaussian_vectors(2, cols, 9, dtype="bf16"))
    y = Guarded(torch, (2, rows), torch.float32)
    ws = Guarded(torch, (L.lq_gemv_workspace_size(2, cols, T),), torch.uint8)
    L.lq_gemv_rice("e8", words.t, offs.t, scales, signs, T, x, y.t, ws.t)
    # attention and the block rotation
    tokens, kvh, qh = 300, 2, 8
    Kc, Ks, Kd = L.quantize(to_dev_bf16(torch, gaussian_matrix(tokens, kvh * 128, 1.0, 10, dtype="bf16")),
                            lattice="e8", tile=128, seed=11, beta=0.25)
    Vc, Vs, Vd = L.quantize(to_dev_bf16(torch, gaussian_matrix(tokens, kvh * 128, 1.0, 12, dtype="bf16")),
                            lattice="e8", tile=128, seed=13, beta=0.25)
    q = to_dev_bf16(torch, gaussian_matrix(qh, 128, 1.0, 14, dtype="bf16"))
    out = Guarded(torch, (qh, 128), torch.float32)
    aws = Guarded(torch, (L.lq_attention_workspace_size(tokens, kvh, qh, 128),), torch.uint8)
    L.lq_attention_decode("e8", Kc, Ks, Kd, Vc, Vs, Vd, q, out.t, aws.t)
    R = to_dev(torch, KV.haar_rotation(128, 15).astype(np.float32))
    Yr = Guarded(torch, (tokens, kvh * 128), torch.float32)
    L.lq_rotate_blocks(R, to_dev_bf16(torch, gaussian_matrix(tokens, kvh * 128, 1.0, 16, dtype="bf16")), Yr.t)
    torch.cuda.synchronize()
    assert torch.equal(dec.t, codes)
    for g in [words, offs, total, rws, dec, y, ws, out, aws, Yr]:
        assert g.intact()
