"""CPU-side checks of the C-ABI library: it builds, loads, exports every
symbol declared in include/lq.h, and rejects bad arguments before launching
anything (these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from lattice_vq_weight_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol():
    import lattice_vq_weight_gb300 as L
    assert set(declared_functions()) == set(L.SIGNATURES)


def test_pick_tile_matches_oracle_rule(golden_dir):
    import json
    import lattice_vq_weight_gb300 as L
    f = json.load(open(os.path.join(golden_dir, "pages_figures.json")))["hadamard_tile_sizes"]
    for c in f["cases"]:
        assert L.lq_pick_tile(c["cols"], c["requested"]) == c["expect"]
    for cols in (128, 256, 768, 1000, 3584, 4096, 14336, 28672, 8192, 5120, 2048 * 3):
        for req in (128, 256, 512, 1024, 2048, 4096):
            assert L.lq_pick_tile(cols, req) == O.pick_tile(cols, req), (cols, req)


def test_status_strings_and_version():
    import lattice_vq_weight_gb300 as L
    assert L.status_string(0) == "ok"
    for s in range(1, 6):
        assert len(L.status_string(s)) > 5
    assert L.status_string(99) == "unknown status"
    assert L.lq_version() >= 100


def test_argument_errors_are_synchronous():
    import lattice_vq_weight_gb300 as L
    lib = L.lib
    P = ctypes.c_void_p
    good = P(0x10000)        # aligned stand-in pointer, never dereferenced
    odd = P(0x10004)
    nul = P(0)
    s = P(0)
    q = lambda lat, W, wdt, rows, cols, ldw, tile, beta, codes, scales, signs: lib.lq_quantize(
        lat, W, wdt, rows, cols, ldw, tile, 0, beta, codes, scales, signs, nul, s)
    assert q(3, good, 1, 4, 256, 256, 256, 0.25, good, good, good) == L.LQ_ERR_ARG        # lattice
    assert q(8, good, 1, 4, 256, 256, 100, 0.25, good, good, good) == L.LQ_ERR_UNSUPPORTED  # tile
    assert q(8, good, 1, 4, 384, 384, 256, 0.25, good, good, good) == L.LQ_ERR_SHAPE   # cols % tile
    assert q(8, good, 7, 4, 256, 256, 256, 0.25, good, good, good) == L.LQ_ERR_DTYPE
    assert q(8, good, 1, 4, 256, 256, 256, -1.0, good, good, good) == L.LQ_ERR_ARG     # beta
    assert q(8, good, 1, 4, 256, 128, 256, 0.25, good, good, good) == L.LQ_ERR_SHAPE   # ldw < cols
    assert q(8, good, 1, 4, 256, 260, 256, 0.25, good, good, good) == L.LQ_ERR_SHAPE   # ldw*2 % 16
    assert q(8, nul, 1, 4, 256, 256, 256, 0.25, good, good, good) == L.LQ_ERR_ARG
    assert q(8, odd, 1, 4, 256, 256, 256, 0.25, good, good, good) == L.LQ_ERR_ARG
    assert q(8, good, 1, -1, 256, 256, 256, 0.25, good, good, good) == L.LQ_ERR_SHAPE
    g = lambda batch, tile=256, cols=256: lib.lq_gemv(
        8, good, good, good, 4, cols, tile, good, 1, batch, good, good, nul, s)
    assert g(0) == L.LQ_ERR_SHAPE and g(17) == L.LQ_ERR_SHAPE
    assert g(1, tile=64) == L.LQ_ERR_UNSUPPORTED
    assert g(1, tile=4096, cols=4096) == L.LQ_ERR_UNSUPPORTED   # tiles stop at 2048
    assert g(1, tile=2048, cols=3072) == L.LQ_ERR_SHAPE         # cols % tile
    assert lib.lq_dequantize(8, good, good, good, 4, 256, 256, good, 5, s) == L.LQ_ERR_DTYPE
    assert lib.lq_make_signs(0, -1, good, s) == L.LQ_ERR_SHAPE
    arr = (ctypes.c_void_p * 9)(*([0x10000] * 9))
    rows = (ctypes.c_int64 * 9)(*([4] * 9))
    gg = lambda n: lib.lq_gemv_grouped(8, n, arr, arr, arr, rows, 256, 256, good, 1, 1, arr, good, nul, s)
    assert gg(0) == L.LQ_ERR_ARG and gg(9) == L.LQ_ERR_ARG      # group size 1 .. 8
    # one fp16 plane per matrix and batch row, plus one float per (batch row, tile)
    assert L.lq_gemv_grouped_workspace_size(3, 2, 4096, 256) >= 3 * 2 * (4096 * 2 + 16 * 4)
    assert L.lq_gemv_workspace_size(1, 4096, 256) >= 4096 * 2 + 16 * 4
    # grouped quantize: group size, then the per-matrix checks of lq_quantize
    I64 = ctypes.c_int64 * 9
    ones = (ctypes.c_uint64 * 9)(*([1] * 9))
    qg = lambda n, rows, cols, ldw, tile=256, beta=0.25, Ws=arr: lib.lq_quantize_grouped(
        8, n, Ws, 1, I64(*rows), I64(*cols), I64(*ldw), tile, ones, beta, arr, arr, arr, nul, s)
    r9, c9 = [4] * 9, [256] * 9
    assert qg(0, r9, c9, c9) == L.LQ_ERR_ARG and qg(9, r9, c9, c9) == L.LQ_ERR_ARG
    assert qg(2, r9, [256, 384] + c9[2:], [256, 384] + c9[2:]) == L.LQ_ERR_SHAPE        # cols % tile
    assert qg(2, r9, c9, [256, 128] + c9[2:]) == L.LQ_ERR_SHAPE                         # ldw < cols
    assert qg(2, [4, -1] + r9[2:], c9, c9) == L.LQ_ERR_SHAPE
    assert qg(2, r9, c9, c9, tile=100) == L.LQ_ERR_UNSUPPORTED
    assert qg(2, r9, c9, c9, beta=0.0) == L.LQ_ERR_ARG
    bad = (ctypes.c_void_p * 9)(*([0x10000, 0x10004] + [0x10000] * 7))
    assert qg(2, r9, c9, c9, Ws=bad) == L.LQ_ERR_ARG                                    # W alignment
    assert lib.lq_quantize_grouped(8, 2, nul, 1, I64(*r9), I64(*c9), I64(*c9), 256, ones, 0.25, arr, arr, arr,
                                   nul, s) == L.LQ_ERR_ARG
    # scale formats: unknown format -> LQ_ERR_ARG; 16-bit scales need 2-byte, float32 4-byte alignment
    two = P(0x10002)
    qx = lambda fmt, scales: lib.lq_quantize_ex(8, good, 1, 4, 256, 256, 256, 0, 0.25, fmt, good, scales, good,
                                                nul, s)
    assert qx(3, good) == L.LQ_ERR_ARG and qx(-1, good) == L.LQ_ERR_ARG
    assert qx(L.LQ_SCALE_TILE_F32, two) == L.LQ_ERR_ARG
    assert lib.lq_dequantize_ex(8, good, good, 9, good, 4, 256, 256, good, 0, s) == L.LQ_ERR_ARG
    assert lib.lq_dequantize_ex(8, good, P(0x10001), L.LQ_SCALE_TILE_F16, good, 4, 256, 256, good, 0,
                                s) == L.LQ_ERR_ARG
    assert lib.lq_gemv_ex(8, good, good, 5, good, 4, 256, 256, good, 1, 1, good, good, nul, s) == L.LQ_ERR_ARG
    assert lib.lq_gemm_ex(8, good, good, 7, good, 128, 256, 256, good, 4, good, L.LQ_F32, good, nul,
                          s) == L.LQ_ERR_ARG
    # GEMM output type: float32 or bf16; the bf16 workspace adds the float32 sums [M x N]
    assert lib.lq_gemm(8, good, good, good, 200, 256, 256, good, 4, good, 5, good, nul, s) == L.LQ_ERR_DTYPE
    assert L.lq_gemm_workspace_size(4, 200, 256, 7) == 0
    assert (L.lq_gemm_workspace_size(300, 200, 1024, L.LQ_BF16)
            >= L.lq_gemm_workspace_size(300, 200, 1024, L.LQ_F32) + 300 * 200 * 4)
    # the wait-expiry self-test needs a status word to report into
    assert lib.lq_gemm_wait_expiry_test(8, good, good, good, 128, 256, 256, good, 4, good, L.LQ_F32, good, nul,
                                        s) == L.LQ_ERR_ARG
    # lq_gemv_noalloc: a request larger than its fixed scratch is refused before any pointer is looked at
    assert lib.lq_gemv_noalloc(8, None, None, None, 4, 1 << 20, 256, None, L.LQ_BF16, 16, None, None,
                               None) == L.LQ_ERR_SHAPE
    # the KV attention takes float32 or fp16 tile scales only
    assert lib.lq_attention_decode_ex(8, good, good, good, good, good, good, L.LQ_SCALE_ROW_BF16, 16, 1, 1, 128,
                                      good, 1, good, good, ctypes.c_size_t(1 << 20), s) == L.LQ_ERR_ARG
    # dithered calls take float32 or fp16 tile scales only
    assert lib.lq_quantize_dithered(8, good, 1, 4, 256, 256, 256, 0, 1, 0.25, L.LQ_SCALE_ROW_BF16, good, good,
                                    good, nul, s) == L.LQ_ERR_ARG
    assert lib.lq_dequantize_dithered(8, good, good, L.LQ_SCALE_ROW_BF16, good, 1, 4, 256, 256, good, 0,
                                      s) == L.LQ_ERR_ARG
    assert lib.lq_attention_decode_dithered(8, good, good, good, 1, good, good, good, 2, L.LQ_SCALE_ROW_BF16, 16, 1,
                                            1, 128, good, 1, good, good, ctypes.c_size_t(1 << 20), s) == L.LQ_ERR_ARG
    # Rice-coded caches: streams and offsets required; 2^28 values per stream at most
    ar = lambda ks, tokens: lib.lq_attention_decode_rice(8, ks, ctypes.c_size_t(1024), good, good, good, good,
                                                         ctypes.c_size_t(1024), good, good, good, 0, tokens, 1, 1,
                                                         128, good, 1, good, good, ctypes.c_size_t(1 << 30), s)
    assert ar(nul, 16) == L.LQ_ERR_ARG
    assert ar(good, (1 << 21) + 1) == L.LQ_ERR_SHAPE
    # Rice format: worst case 8 bits per symbol + parity bits + 3 bits per segment, 16 bytes of padding
    assert L.lq_rice_stream_bound("e8", 2, 256, 256) == ((2 * 3 + 2 * 256 * 8 + 2 * 32 + 31) // 32) * 4 + 16
    assert L.lq_rice_stream_bound("e8", 1 << 15, 1 << 14, 256) == 0          # more than 2^28 weights
    enc = lambda rows, cols, tile, nbytes: lib.lq_rice_encode(8, good, rows, cols, tile, good, nbytes, good,
                                                             P(0x10008), good, nul, s)
    assert enc(2, 256, 256, 16) == L.LQ_ERR_SHAPE                  # stream smaller than the bound
    assert enc(2, 256, 100, 1 << 20) == L.LQ_ERR_UNSUPPORTED
    # closed-form scale for a target SNR: the library's host function against the oracle
    import oracle.calibration_oracle as C
    for lat in ("e8", "d4", "a2", "z1"):
        for snr in (10.0, 20.0, 30.0):
            assert abs(L.lq_beta_for_snr(lat, snr) / C.beta_for_snr(lat, snr) - 1) < 1e-6
    assert L.lq_beta_for_snr(3, 20.0) == 0.0
    # attention: head_dim 128 only, group sizes 1/2/4/8
    att = lambda kvh, qh, d, ws_bytes=1 << 30: lib.lq_attention_decode(
        8, good, good, good, good, good, good, 100, kvh, qh, d, good, 1, good, good, ws_bytes, s)
    assert att(2, 8, 64) == L.LQ_ERR_UNSUPPORTED
    assert att(4, 6, 128) == L.LQ_ERR_SHAPE and att(2, 6, 128) == L.LQ_ERR_UNSUPPORTED
    assert att(2, 8, 128, 16) == L.LQ_ERR_SHAPE                      # workspace too small
    assert L.lq_attention_workspace_size(100, 2, 8, 64) == 0
    assert L.lq_gemv_workspace_size(0, 4096, 256) == 0
