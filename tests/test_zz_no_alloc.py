"""lq_gemv_noalloc against lq_gemv, through the C ABI.

lq_gemv_noalloc serves callers that cannot allocate device memory (engine
plug-ins whose host owns all device memory, latency-critical loops that must
not synchronise on an allocation): it runs the same GEMV with the library's
fixed device scratch.  This file is collected last so that a run stopping at
its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
from synthetic import gaussian_matrix, gaussian_vectors
from tests._parity import normwise_rel
from tests.gpu_util import cuda, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _call(L, fn, *args):
    status = fn(*args)
    assert status == L.LQ_OK, L.status_string(status)


@pytest.mark.parametrize("batch,tile", [(1, 256), (16, 128)])
def test_noalloc_matches_gemv_twice(batch, tile):
    torch, L = cuda()
    lib = L.lib
    R, C = 300, 4096
    W = gaussian_matrix(R, C, 0.02, 77, dtype="bf16")
    d = O.splitmix64_signs(5, C)
    q = O.quantize(W, "e8", tile, d, 0.25)
    codes, scales, signs = to_dev(torch, q.codes), to_dev(torch, q.scales), to_dev(torch, d)
    x = to_dev_bf16(torch, gaussian_vectors(batch, C, 78, dtype="bf16"))
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    y_ref = torch.empty((batch, R), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.lq_gemv_workspace_size(batch, C, tile), dtype=torch.uint8, device="cuda")
    _call(L, lib.lq_gemv, L.LQ_E8, P(codes.data_ptr()), P(scales.data_ptr()), P(signs.data_ptr()), R, C, tile,
          P(x.data_ptr()), L.LQ_BF16, batch, P(y_ref.data_ptr()), P(ws.data_ptr()), None, stream)
    outs = []
    for _ in range(2):
        y = torch.full((batch, R), float("nan"), dtype=torch.float32, device="cuda")
        _call(L, lib.lq_gemv_noalloc, L.LQ_E8, P(codes.data_ptr()), P(scales.data_ptr()), P(signs.data_ptr()),
              R, C, tile, P(x.data_ptr()), L.LQ_BF16, batch, P(y.data_ptr()), None, stream)
        outs.append(y)
    torch.cuda.synchronize()
    ref = y_ref.cpu().numpy()
    oracle_y = O.gemv(q.codes, q.scales, d, tile, "e8", x.float().cpu().numpy())
    for y in outs:
        # the same kernels on the same inputs.  The GEMV adds the partial sums
        # of a row that several warps share with fp32 atomics, whose order
        # varies from run to run, so two runs agree to rounding only: a few
        # float32 ulps, far below anything stale scratch contents would cause.
        got = y.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref))
        assert normwise_rel(got, ref) < 1e-6
        assert normwise_rel(got, oracle_y) < 2e-3
    assert normwise_rel(ref, oracle_y) < 2e-3


def test_noalloc_rejects_oversized_request():
    torch, L = cuda()
    lib = L.lib
    P = ctypes.c_void_p
    cols = 1 << 20
    assert L.lq_gemv_workspace_size(16, cols, 256) > L.LQ_GEMV_NOALLOC_MAX_WORKSPACE
    # null pointers throughout: the size check comes first and returns
    # LQ_ERR_SHAPE; were it ever skipped, the pointer checks would still stop
    # the call before any launch (LQ_ERR_ARG) and the assertion would fail
    st = lib.lq_gemv_noalloc(L.LQ_E8, None, None, None, 4, cols, 256, None, L.LQ_BF16, 16, None, None, None)
    assert st == L.LQ_ERR_SHAPE
    # the largest request that fits (batch 16, 131072 columns, tile 128) is accepted
    assert L.lq_gemv_workspace_size(16, 1 << 17, 128) == L.LQ_GEMV_NOALLOC_MAX_WORKSPACE
