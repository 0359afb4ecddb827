"""GPU decode attention over Rice-coded K and V caches (decoded on chip)
against the oracle, and against the int8-code attention on the same codes."""
import numpy as np
import pytest

import oracle as O
import oracle.kv_oracle as KV
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev_bf16

pytestmark = pytest.mark.gpu


def rice_cache(torch, L, lattice, codes):
    rows, cols = codes.shape
    words = torch.empty(L.lq_rice_stream_bound(lattice, rows, cols, 128) // 4, dtype=torch.int32, device="cuda")
    offs = torch.empty((rows, cols // 128), dtype=torch.int32, device="cuda")
    tot = torch.empty(1, dtype=torch.int64, device="cuda")
    ws = torch.empty(L.lq_rice_workspace_size(rows, cols, 128), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.lq_rice_encode(lattice, codes, 128, words, offs, tot, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return words, offs, int(tot.item())


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
@pytest.mark.parametrize("tokens,kv_heads,group,fmt", [(1500, 2, 4, "tile_f16"), (37, 2, 1, "tile_f32"),
                                                       (300, 1, 8, "tile_f16"), (4097, 1, 2, "tile_f32")])
def test_attention_rice(lattice, tokens, kv_heads, group, fmt):
    torch, L = cuda()
    cols = kv_heads * 128
    X = gaussian_matrix(tokens, cols, 1.0, 840 + tokens, dtype="bf16")
    Y = gaussian_matrix(tokens, cols, 1.0, 841 + tokens, dtype="bf16")
    kc, ks, kg = L.quantize_ex(to_dev_bf16(torch, X), lattice=lattice, tile=128, seed=81, beta=0.25,
                               scale_format=fmt)
    vc, vs, vg = L.quantize_ex(to_dev_bf16(torch, Y), lattice=lattice, tile=128, seed=82, beta=0.25,
                               scale_format=fmt)
    kw, ko, kbits = rice_cache(torch, L, lattice, kc)
    vw, vo, vbits = rice_cache(torch, L, lattice, vc)
    q = to_dev_bf16(torch, gaussian_vectors(kv_heads * group, 128, 842, dtype="bf16"))
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kv_heads, kv_heads * group, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((kv_heads * group, 128), dtype=torch.float32, device="cuda")
    L.lq_attention_decode_rice(lattice, kw, ko, ks, kg, vw, vo, vs, vg, fmt, q, out, ws)
    ref8 = torch.empty_like(out)
    L.lq_attention_decode_ex(lattice, kc, ks, kg, vc, vs, vg, fmt, q, ref8, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    # the same arithmetic on the same codes
    assert normwise_rel(got, ref8.cpu().numpy()) < 1e-6
    dk, dv = O.splitmix64_signs(81, cols), O.splitmix64_signs(82, cols)
    ref = KV.attention_from_codes(q.float().cpu().numpy(), kc.cpu().numpy(), ks.float().cpu().numpy(), dk,
                                  vc.cpu().numpy(), vs.float().cpu().numpy(), dv, kv_heads, 128, lattice)
    assert normwise_rel(got, ref) < 2e-3
    if lattice == "e8" and fmt == "tile_f16":
        # stream + 16-bit norms: about 4 bits per cached value, ~3.8x against bf16 on the pages
        bits = (kbits + vbits + 2 * 16 * tokens * kv_heads) / (2 * tokens * cols)
        assert 3.5 < 16.0 / bits < 4.5


@pytest.mark.parametrize("lattice", ["e8", "d4", "a2", "z1"])
def test_attention_rice_long_runs(lattice):
    """Codes whose Rice segments have unary runs longer than the decoder's
    32-bit window and segments longer than the 32 stream words each token
    stages (every fourth token made only of large blocks): the attention from
    the stream equals the attention from the same int8 codes."""
    from tests.test_gpu_rice import _crafted_codes
    torch, L = cuda()
    tokens, kv_heads, group = 300, 2, 4
    cols = kv_heads * 128
    kc_np = _crafted_codes(lattice, tokens, cols, 950).astype(np.int8)
    vc_np = _crafted_codes(lattice, tokens, cols, 951).astype(np.int8)
    assert np.abs(kc_np.astype(np.int64)).max() >= 100
    rng = np.random.default_rng(952)
    ks = torch.from_numpy(rng.uniform(0.002, 0.004, (tokens, kv_heads)).astype(np.float32)).cuda()
    vs = torch.from_numpy(rng.uniform(0.002, 0.004, (tokens, kv_heads)).astype(np.float32)).cuda()
    kg = torch.from_numpy(O.splitmix64_signs(81, cols)).cuda()
    vg = torch.from_numpy(O.splitmix64_signs(82, cols)).cuda()
    kc, vc = torch.from_numpy(kc_np).cuda(), torch.from_numpy(vc_np).cuda()
    kw, ko, _ = rice_cache(torch, L, lattice, kc)
    vw, vo, _ = rice_cache(torch, L, lattice, vc)
    q = to_dev_bf16(torch, gaussian_vectors(kv_heads * group, 128, 953, dtype="bf16"))
    ws = torch.empty(L.lq_attention_workspace_size(tokens, kv_heads, kv_heads * group, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((kv_heads * group, 128), dtype=torch.float32, device="cuda")
    L.lq_attention_decode_rice(lattice, kw, ko, ks, kg, vw, vo, vs, vg, "tile_f32", q, out, ws)
    ref8 = torch.empty_like(out)
    L.lq_attention_decode_ex(lattice, kc, ks, kg, vc, vs, vg, "tile_f32", q, ref8, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    assert normwise_rel(got, ref8.cpu().numpy()) < 1e-6
    ref = KV.attention_from_codes(q.float().cpu().numpy(), kc_np, ks.cpu().numpy(), kg.cpu().numpy(), vc_np,
                                  vs.cpu().numpy(), vg.cpu().numpy(), kv_heads, 128, lattice)
    assert normwise_rel(got, ref) < 2e-3
