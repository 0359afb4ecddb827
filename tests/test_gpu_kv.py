"""GPU decode attention over quantized KV caches against the CPU oracle."""
import numpy as np
import pytest

import oracle as O
import oracle.kv_oracle as KV
from synthetic import gaussian_matrix
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
TOL = 2e-3


def run(torch, L, lattice, kq, vq, dk, dv, q_np, kv_heads, qdtype):
    tokens = kq.codes.shape[0]
    q_heads = q_np.shape[0]
    q = to_dev_bf16(torch, q_np) if qdtype == "bf16" else to_dev(torch, q_np.astype(np.float32))
    out = torch.full((q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kv_heads, q_heads, 128) // 4 + 1, dtype=torch.float32,
                     device="cuda")
    L.lq_attention_decode(lattice, to_dev(torch, kq.codes), to_dev(torch, kq.scales), to_dev(torch, dk),
                          to_dev(torch, vq.codes), to_dev(torch, vq.scales), to_dev(torch, dv), q, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tokens,kv_heads,group", [(1, 1, 1), (37, 2, 4), (300, 1, 8), (1000, 2, 2), (4097, 1, 4)])
def test_attention_parity(lattice, tokens, kv_heads, group):
    torch, L = cuda()
    cols = kv_heads * 128
    X = gaussian_matrix(tokens, cols, 1.0, 800 + tokens, dtype="bf16")
    Y = gaussian_matrix(tokens, cols, 1.0, 900 + tokens, dtype="bf16")
    dk, dv = O.splitmix64_signs(31, cols), O.splitmix64_signs(32, cols)
    kq = KV.kv_quantize(X, lattice, 128, dk, 0.25)
    vq = KV.kv_quantize(Y, lattice, 128, dv, 0.25)
    q = gaussian_matrix(kv_heads * group, 128, 1.0, 1000 + tokens, dtype="bf16")
    ref = KV.attention_from_codes(q, kq.codes, kq.scales, dk, vq.codes, vq.scales, dv, kv_heads, 128, lattice)
    got = run(torch, L, lattice, kq, vq, dk, dv, q, kv_heads, "bf16")
    assert normwise_rel(got, ref) < TOL


def test_attention_fp32_query_and_peaked_scores():
    """fp32 queries scaled x8 (a peaked softmax) still match."""
    torch, L = cuda()
    X = gaussian_matrix(700, 256, 1.0, 71, dtype="bf16")
    Y = gaussian_matrix(700, 256, 1.0, 72, dtype="bf16")
    dk, dv = O.splitmix64_signs(41, 256), O.splitmix64_signs(42, 256)
    kq = KV.kv_quantize(X, "e8", 128, dk, 0.125)
    vq = KV.kv_quantize(Y, "e8", 128, dv, 0.125)
    q = 8.0 * gaussian_matrix(8, 128, 1.0, 73)
    ref = KV.attention_from_codes(q, kq.codes, kq.scales, dk, vq.codes, vq.scales, dv, 2, 128, "e8")
    got = run(torch, L, "e8", kq, vq, dk, dv, q, 2, "fp32")
    assert normwise_rel(got, ref) < TOL


def test_llama3_8b_cache_32k_tokens():
    """Llama-3-8B decode shape: 8 kv heads, 32 query heads, 32 768 cached tokens, quantized
    on the GPU (E8, T = 128, beta 1/4); attention from the device codes against the
    oracle's attention on the same codes."""
    torch, L = cuda()
    from synthetic import torch_gaussian_matrix
    tokens, kvh, qh = 32768, 8, 32
    K = torch_gaussian_matrix(tokens, kvh * 128, 1.0, 5100, device="cuda")
    V = torch_gaussian_matrix(tokens, kvh * 128, 1.0, 5101, device="cuda")
    kc, ks, kd = L.quantize(K, lattice="e8", tile=128, seed=5102, beta=0.25)
    vc, vs, vd = L.quantize(V, lattice="e8", tile=128, seed=5103, beta=0.25)
    q = torch.randn((qh, 128), device="cuda").to(torch.bfloat16)
    out = torch.empty((qh, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kvh, qh, 128), dtype=torch.uint8, device="cuda")
    L.lq_attention_decode("e8", kc, ks, kd, vc, vs, vd, q, out, ws)
    torch.cuda.synchronize()
    ref = KV.attention_from_codes(q.float().cpu().numpy(), kc.cpu().numpy(), ks.cpu().numpy(), kd.cpu().numpy(),
                                  vc.cpu().numpy(), vs.cpu().numpy(), vd.cpu().numpy(), kvh, 128, "e8")
    assert normwise_rel(out.cpu().numpy(), ref) < TOL


@pytest.mark.parametrize("xdtype", ["bf16", "fp32"])
def test_rotate_blocks_matches_oracle(xdtype):
    torch, L = cuda()
    X = gaussian_matrix(333, 384, 1.0, 61, dtype="bf16")
    Q = KV.haar_rotation(128, 62)
    Xd = to_dev_bf16(torch, X) if xdtype == "bf16" else to_dev(torch, X.astype(np.float32))
    Rd = to_dev(torch, Q.astype(np.float32))
    for transpose in (False, True):
        Y = torch.empty((333, 384), dtype=torch.float32, device="cuda")
        L.lq_rotate_blocks(Rd, Xd, Y, transpose=transpose)
        torch.cuda.synchronize()
        ref = KV.rotate_blocks(X, Q.astype(np.float32).astype(np.float64), transpose=transpose)
        assert normwise_rel(Y.cpu().numpy(), ref) < 1e-6


def test_qjl_rotated_cache_attention():
    """K, V and q rotated by a Haar matrix before quantization, the output rotated back:
    matches the oracle applied to the same rotated inputs."""
    torch, L = cuda()
    tokens, kvh, qh = 900, 2, 8
    X = gaussian_matrix(tokens, kvh * 128, 1.0, 63, dtype="bf16")
    Y = gaussian_matrix(tokens, kvh * 128, 1.0, 64, dtype="bf16")
    q = gaussian_matrix(qh, 128, 1.0, 65, dtype="bf16")
    Q = KV.haar_rotation(128, 66)
    Rd = to_dev(torch, Q.astype(np.float32))
    rot = lambda A: (lambda out: (L.lq_rotate_blocks(Rd, A, out), out)[1])(
        torch.empty(A.shape, dtype=torch.float32, device="cuda"))
    Kr, Vr, qr = rot(to_dev_bf16(torch, X)), rot(to_dev_bf16(torch, Y)), rot(to_dev_bf16(torch, q))
    kc, ks, kd = L.quantize(Kr, lattice="e8", tile=128, seed=67, beta=0.25)
    vc, vs, vd = L.quantize(Vr, lattice="e8", tile=128, seed=68, beta=0.25)
    out_r = torch.empty((qh, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kvh, qh, 128), dtype=torch.uint8, device="cuda")
    L.lq_attention_decode("e8", kc, ks, kd, vc, vs, vd, qr, out_r, ws)
    out = torch.empty_like(out_r)
    L.lq_rotate_blocks(Rd, out_r, out, transpose=True)
    torch.cuda.synchronize()
    # oracle on the same rotated fp32 inputs
    kq = KV.kv_quantize(Kr.cpu().numpy(), "e8", 128, kd.cpu().numpy(), 0.25)
    vq = KV.kv_quantize(Vr.cpu().numpy(), "e8", 128, vd.cpu().numpy(), 0.25)
    o_r = KV.attention_from_codes(qr.cpu().numpy(), kq.codes, kq.scales, kd.cpu().numpy(), vq.codes, vq.scales,
                                  vd.cpu().numpy(), kvh, 128, "e8")
    ref = KV.rotate_blocks(o_r, Q.astype(np.float32).astype(np.float64), transpose=True)
    assert normwise_rel(out.cpu().numpy(), ref) < TOL
