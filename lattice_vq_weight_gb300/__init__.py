"""Thin Python binding of liblq (include/lq.h): argument marshalling only.

Every step of quantization and of the code-based products runs in the CUDA
kernels of ``liblq.so``; this module only turns torch tensors into pointers,
sizes and the current CUDA stream, and raises :class:`LQError` on a non-OK
status.  There is no fallback: if the library is missing, importing the
binding's entry points raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblq.so")

LQ_OK, LQ_ERR_ARG, LQ_ERR_SHAPE, LQ_ERR_DTYPE, LQ_ERR_CUDA, LQ_ERR_UNSUPPORTED = range(6)
LQ_DEV_NONFINITE, LQ_DEV_RANGE, LQ_DEV_TIMEOUT, LQ_DEV_FORMAT = 1, 2, 4, 8
LQ_Z1, LQ_A2, LQ_D4, LQ_E8 = 1, 2, 4, 8
LQ_F32, LQ_BF16 = 0, 1
LATTICE_IDS = {"z1": LQ_Z1, "a2": LQ_A2, "d4": LQ_D4, "e8": LQ_E8}
LATTICE_DIM = {"z1": 1, "a2": 2, "d4": 4, "e8": 8}

# (name, restype, argtypes) of every entry point declared in include/lq.h
_P, _I64, _U64, _I32, _F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "lq_status_string": (ctypes.c_char_p, [_I32]),
    "lq_version": (_I32, []),
    "lq_pick_tile": (_I32, [_I64, _I32]),
    "lq_make_signs": (_I32, [_U64, _I64, _P, _P]),
    "lq_quantize": (_I32, [_I32, _P, _I32, _I64, _I64, _I64, _I32, _U64, _F32, _P, _P, _P, _P, _P]),
    "lq_quantize_grouped": (_I32, [_I32, _I32, _P, _I32, _P, _P, _P, _I32, _P, _F32, _P, _P, _P, _P, _P]),
    "lq_dequantize": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I32, _P, _I32, _P]),
    "lq_quantize_ex": (_I32, [_I32, _P, _I32, _I64, _I64, _I64, _I32, _U64, _F32, _I32, _P, _P, _P, _P, _P]),
    "lq_dequantize_ex": (_I32, [_I32, _P, _P, _I32, _P, _I64, _I64, _I32, _P, _I32, _P]),
    "lq_gemv_ex": (_I32, [_I32, _P, _P, _I32, _P, _I64, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P]),
    "lq_gemm_ex": (_I32, [_I32, _P, _P, _I32, _P, _I64, _I64, _I32, _P, _I64, _P, _I32, _P, _P, _P]),
    "lq_attention_decode_ex": (_I32, [_I32, _P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _P, _I32, _P,
                                      _P, ctypes.c_size_t, _P]),
    "lq_quantize_dithered": (_I32, [_I32, _P, _I32, _I64, _I64, _I64, _I32, _U64, _U64, _F32, _I32, _P, _P, _P,
                                    _P, _P]),
    "lq_dequantize_dithered": (_I32, [_I32, _P, _P, _I32, _P, _U64, _I64, _I64, _I32, _P, _I32, _P]),
    "lq_attention_decode_rice": (_I32, [_I32, _P, ctypes.c_size_t, _P, _P, _P, _P, ctypes.c_size_t, _P, _P, _P,
                                        _I32, _I64, _I32, _I32, _I32, _P, _I32, _P, _P, ctypes.c_size_t, _P]),
    "lq_attention_decode_dithered": (_I32, [_I32, _P, _P, _P, _U64, _P, _P, _P, _U64, _I32, _I64, _I32, _I32, _I32,
                                            _P, _I32, _P, _P, ctypes.c_size_t, _P]),
    "lq_gemv_workspace_size": (ctypes.c_size_t, [_I32, _I64, _I32]),
    "lq_gemv": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P]),
    "lq_gemv_noalloc": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I32, _P, _I32, _I32, _P, _P, _P]),
    "lq_gemv_grouped_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I64, _I32]),
    "lq_gemv_grouped": (_I32, [_I32, _I32, _P, _P, _P, _P, _I64, _I32, _P, _I32, _I32, _P, _P, _P, _P]),
    "lq_gemm_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I32]),
    "lq_gemm": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I32, _P, _I64, _P, _I32, _P, _P, _P]),
    "lq_gemm_wait_expiry_test": (_I32, [_I32, _P, _P, _P, _I64, _I64, _I32, _P, _I64, _P, _I32, _P, _P, _P]),
    "lq_rice_stream_bound": (ctypes.c_size_t, [_I32, _I64, _I64, _I32]),
    "lq_rice_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I32]),
    "lq_rice_encode": (_I32, [_I32, _P, _I64, _I64, _I32, _P, ctypes.c_size_t, _P, _P, _P, _P, _P]),
    "lq_rice_decode": (_I32, [_I32, _P, ctypes.c_size_t, _P, _I64, _I64, _I32, _P, _P]),
    "lq_gemv_rice": (_I32, [_I32, _P, ctypes.c_size_t, _P, _P, _P, _I64, _I64, _I32, _P, _I32, _I32, _P, _P,
                            _P, _P]),
    "lq_beta_for_snr": (ctypes.c_double, [_I32, ctypes.c_double]),
    "lq_error_sums": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _P]),
    "lq_calibrate_workspace_size": (ctypes.c_size_t, [_I32, _I64, _I64, _I32]),
    "lq_calibrate_bps": (_I32, [_I32, _I32, ctypes.c_double, _P, _I32, _I64, _I64, _I64, _U64, _P, ctypes.c_size_t,
                                _P, _P]),
    "lq_attention_workspace_size": (ctypes.c_size_t, [_I64, _I32, _I32, _I32]),
    "lq_attention_decode": (_I32, [_I32, _P, _P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _I32, _P, _P,
                                   ctypes.c_size_t, _P]),
    "lq_rotate_blocks": (_I32, [_P, _I32, _I32, _P, _I32, _I64, _I64, _I64, _P, _I64, _P]),
}


class LQError(RuntimeError):
    """A liblq entry point returned a status other than LQ_OK."""

    def __init__(self, name: str, status: int):
        super().__init__(f"{name} failed: status {status} ({status_string(status)})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"liblq.so is not built ({LIB_PATH}); run `python -m lattice_vq_weight_gb300.build` "
            "or __graft_entry__.build()")
    dll = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(dll, name)
        fn.restype = res
        fn.argtypes = args
    return dll


_LIB = None


def _get_lib():
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _get_lib()
    raise AttributeError(name)


def status_string(status: int) -> str:
    return _get_lib().lq_status_string(int(status)).decode()


def _check(name: str, status: int) -> None:
    if status != LQ_OK:
        raise LQError(name, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _lattice_id(lattice) -> int:
    return LATTICE_IDS[lattice] if isinstance(lattice, str) else int(lattice)


def _row_stride(W) -> int:
    """Row stride in elements; an empty matrix (whose stride torch may report as 0) passes its width."""
    return int(W.stride(0)) if W.shape[0] > 0 else int(W.shape[1])


def _dtype_id(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return LQ_BF16
    if t.dtype == torch.float32:
        return LQ_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ------------------------------------------------------------------ C-ABI calls
def lq_version() -> int:
    return _get_lib().lq_version()


def lq_pick_tile(cols: int, requested: int) -> int:
    return _get_lib().lq_pick_tile(int(cols), int(requested))


def lq_make_signs(seed: int, signs, stream=None) -> None:
    _check("lq_make_signs", _get_lib().lq_make_signs(int(seed), signs.numel(), _ptr(signs), _stream(stream)))


def lq_quantize(lattice, W, tile: int, seed: int, beta: float, codes, scales, signs,
                dev_status=None, stream=None) -> None:
    """W [rows x cols] (row stride W.stride(0)) -> codes, scales, signs (all preallocated)."""
    rows, cols = W.shape
    assert W.stride(1) == 1
    _check("lq_quantize", _get_lib().lq_quantize(
        _lattice_id(lattice), _ptr(W), _dtype_id(W), rows, cols, _row_stride(W), int(tile), int(seed),
        float(beta), _ptr(codes), _ptr(scales), _ptr(signs), _ptr(dev_status), _stream(stream)))


def lq_dequantize(lattice, codes, scales, signs, tile: int, W_hat, stream=None) -> None:
    rows, cols = codes.shape
    _check("lq_dequantize", _get_lib().lq_dequantize(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _ptr(signs), rows, cols, int(tile),
        _ptr(W_hat), _dtype_id(W_hat), _stream(stream)))


def lq_gemv_workspace_size(batch: int, cols: int, tile: int) -> int:
    return int(_get_lib().lq_gemv_workspace_size(int(batch), int(cols), int(tile)))


def lq_gemv(lattice, codes, scales, signs, tile: int, x, y, workspace, dev_status=None,
            stream=None) -> None:
    """y[b, r] = sum_t s[r,t] p[r,t,:] . x~[b,t,:]; x [batch x cols], y float32 [batch x rows]."""
    rows, cols = codes.shape
    batch = x.shape[0]
    _check("lq_gemv", _get_lib().lq_gemv(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _ptr(signs), rows, cols, int(tile),
        _ptr(x), _dtype_id(x), batch, _ptr(y), _ptr(workspace), _ptr(dev_status), _stream(stream)))


# Largest workspace lq_gemv_noalloc can serve (LQ_GEMV_NOALLOC_MAX_WORKSPACE in lq.h)
LQ_GEMV_NOALLOC_MAX_WORKSPACE = 4 * 1024 * 1024 + 64 * 1024


def lq_gemv_noalloc(lattice, codes, scales, signs, tile: int, x, y, dev_status=None, stream=None) -> None:
    """lq_gemv using the library's fixed device scratch instead of a caller workspace."""
    rows, cols = codes.shape
    batch = x.shape[0]
    _check("lq_gemv_noalloc", _get_lib().lq_gemv_noalloc(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _ptr(signs), rows, cols, int(tile),
        _ptr(x), _dtype_id(x), batch, _ptr(y), _ptr(dev_status), _stream(stream)))


# Largest group lq_quantize_grouped takes (LQ_QUANTIZE_MAX_GROUP in lq.h)
LQ_QUANTIZE_MAX_GROUP = 8


def lq_quantize_grouped(lattice, Ws, tile: int, seeds, beta: float, codes, scales, signs, dev_status=None,
                        stream=None) -> None:
    """lq_quantize for n matrices in one launch pair: lists Ws[m], seeds[m], codes[m], scales[m], signs[m].

    Every W has the same dtype; rows, cols and the row stride are taken per matrix."""
    n = len(Ws)
    if any(W.dtype != Ws[0].dtype for W in Ws):
        raise TypeError("lq_quantize_grouped: every matrix of a group has the same dtype")
    rows = (ctypes.c_int64 * n)(*[int(W.shape[0]) for W in Ws])
    cols = (ctypes.c_int64 * n)(*[int(W.shape[1]) for W in Ws])
    ldw = (ctypes.c_int64 * n)(*[_row_stride(W) for W in Ws])
    sd = (ctypes.c_uint64 * n)(*[int(x) & 0xFFFFFFFFFFFFFFFF for x in seeds])
    keep = [_ptr_array(Ws), _ptr_array(codes), _ptr_array(scales), _ptr_array(signs)]
    _check("lq_quantize_grouped", _get_lib().lq_quantize_grouped(
        _lattice_id(lattice), n, keep[0][1], _dtype_id(Ws[0]), ctypes.cast(rows, ctypes.c_void_p),
        ctypes.cast(cols, ctypes.c_void_p), ctypes.cast(ldw, ctypes.c_void_p), int(tile),
        ctypes.cast(sd, ctypes.c_void_p), float(beta), keep[1][1], keep[2][1], keep[3][1], _ptr(dev_status),
        _stream(stream)))


# Largest group lq_gemv_grouped takes (LQ_GEMV_MAX_GROUP in lq.h)
LQ_GEMV_MAX_GROUP = 8


def lq_gemv_grouped_workspace_size(n: int, batch: int, cols: int, tile: int) -> int:
    return int(_get_lib().lq_gemv_grouped_workspace_size(int(n), int(batch), int(cols), int(tile)))


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[None if t is None else t.data_ptr() for t in tensors])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def lq_gemv_grouped(lattice, codes, scales, signs, tile: int, x, ys, workspace, dev_status=None,
                    stream=None) -> None:
    """lq_gemv for n matrices sharing x: lists codes[m], scales[m], signs[m], ys[m]."""
    n = len(codes)
    cols = codes[0].shape[1]
    rows = (ctypes.c_int64 * n)(*[int(c.shape[0]) for c in codes])
    keep = [_ptr_array(codes), _ptr_array(scales), _ptr_array(signs), _ptr_array(ys)]
    _check("lq_gemv_grouped", _get_lib().lq_gemv_grouped(
        _lattice_id(lattice), n, keep[0][1], keep[1][1], keep[2][1], ctypes.cast(rows, ctypes.c_void_p),
        cols, int(tile), _ptr(x), _dtype_id(x), x.shape[0], keep[3][1], _ptr(workspace), _ptr(dev_status),
        _stream(stream)))


def lq_gemm_workspace_size(M: int, N: int, K: int, ydtype=LQ_F32) -> int:
    yd = ydtype if isinstance(ydtype, int) else _dtype_id(ydtype)
    return int(_get_lib().lq_gemm_workspace_size(int(M), int(N), int(K), yd))


def lq_gemm(lattice, codes, scales, signs, tile: int, X, Y, workspace, dev_status=None,
            stream=None) -> None:
    """Y [M x N] (float32 or bf16, Y's dtype) = X~ . (s p)^T from the codes [N x K]; X bf16 [M x K]."""
    N, K = codes.shape
    M = X.shape[0]
    _check("lq_gemm", _get_lib().lq_gemm(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _ptr(signs), N, K, int(tile), _ptr(X), M,
        _ptr(Y), _dtype_id(Y), _ptr(workspace), _ptr(dev_status), _stream(stream)))


def lq_gemm_wait_expiry_test(lattice, codes, scales, signs, tile: int, X, Y, workspace, dev_status,
                             stream=None) -> None:
    """The GEMM's wait-expiry self-test (lq.h): raises LQ_DEV_TIMEOUT in dev_status."""
    N, K = codes.shape
    _check("lq_gemm_wait_expiry_test", _get_lib().lq_gemm_wait_expiry_test(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _ptr(signs), N, K, int(tile), _ptr(X), X.shape[0],
        _ptr(Y), _dtype_id(Y), _ptr(workspace), _ptr(dev_status), _stream(stream)))


def lq_rice_stream_bound(lattice, rows: int, cols: int, tile: int) -> int:
    return int(_get_lib().lq_rice_stream_bound(_lattice_id(lattice), int(rows), int(cols), int(tile)))


def lq_rice_workspace_size(rows: int, cols: int, tile: int) -> int:
    return int(_get_lib().lq_rice_workspace_size(int(rows), int(cols), int(tile)))


def lq_rice_encode(lattice, codes, tile: int, stream_words, tile_offsets, total_bits, workspace,
                   dev_status=None, stream=None) -> None:
    """codes int8 [rows x cols] -> Rice stream (uint32 words, as int32 tensor), offsets, total bits."""
    rows, cols = codes.shape
    _check("lq_rice_encode", _get_lib().lq_rice_encode(
        _lattice_id(lattice), _ptr(codes), rows, cols, int(tile), _ptr(stream_words),
        stream_words.numel() * stream_words.element_size(), _ptr(tile_offsets), _ptr(total_bits),
        _ptr(workspace), _ptr(dev_status), _stream(stream)))


def lq_rice_decode(lattice, stream_words, tile_offsets, tile: int, codes, stream=None) -> None:
    rows, cols = codes.shape
    _check("lq_rice_decode", _get_lib().lq_rice_decode(
        _lattice_id(lattice), _ptr(stream_words), stream_words.numel() * stream_words.element_size(),
        _ptr(tile_offsets), rows, cols, int(tile), _ptr(codes), _stream(stream)))


def lq_gemv_rice(lattice, stream_words, tile_offsets, scales, signs, tile: int, x, y, workspace,
                 dev_status=None, stream=None) -> None:
    """lq_gemv from the Rice stream; y float32 [batch x rows]."""
    rows = tile_offsets.shape[0]
    cols = signs.numel()
    batch = x.shape[0]
    _check("lq_gemv_rice", _get_lib().lq_gemv_rice(
        _lattice_id(lattice), _ptr(stream_words), stream_words.numel() * stream_words.element_size(),
        _ptr(tile_offsets), _ptr(scales), _ptr(signs), rows, cols, int(tile), _ptr(x), _dtype_id(x), batch,
        _ptr(y), _ptr(workspace), _ptr(dev_status), _stream(stream)))


def lq_beta_for_snr(lattice, snr_db: float) -> float:
    return float(_get_lib().lq_beta_for_snr(_lattice_id(lattice), float(snr_db)))


def lq_error_sums(W, W_hat, sums, stream=None) -> None:
    """sums (float64 device tensor of 2) = (sum w^2, sum (w - w^)^2)."""
    rows, cols = W.shape
    _check("lq_error_sums", _get_lib().lq_error_sums(
        _ptr(W), _dtype_id(W), rows, cols, _row_stride(W), _ptr(W_hat), _ptr(sums), _stream(stream)))


def lq_calibrate_workspace_size(lattice, rows: int, cols: int, tile: int) -> int:
    return int(_get_lib().lq_calibrate_workspace_size(_lattice_id(lattice), int(rows), int(cols), int(tile)))


def lq_calibrate_bps(lattice, tile: int, target_bps: float, W, seed: int, workspace, stream=None):
    """(beta, bits per weight, SNR dB) of the scale that meets target_bps on the sample W (synchronous)."""
    rows, cols = W.shape
    out = (ctypes.c_double * 3)()
    _check("lq_calibrate_bps", _get_lib().lq_calibrate_bps(
        _lattice_id(lattice), int(tile), float(target_bps), _ptr(W), _dtype_id(W), rows, cols, _row_stride(W),
        int(seed), _ptr(workspace), workspace.numel(), ctypes.cast(out, ctypes.c_void_p), _stream(stream)))
    return float(out[0]), float(out[1]), float(out[2])


def lq_attention_workspace_size(tokens: int, kv_heads: int, q_heads: int, head_dim: int) -> int:
    return int(_get_lib().lq_attention_workspace_size(int(tokens), int(kv_heads), int(q_heads), int(head_dim)))


def lq_attention_decode(lattice, k_codes, k_scales, k_signs, v_codes, v_scales, v_signs, q, out, workspace,
                        stream=None) -> None:
    """out [q_heads x d] = softmax(K^ q / sqrt d) V^ from quantized caches [tokens x kv_heads*d]."""
    tokens = k_codes.shape[0]
    kv_heads = k_scales.shape[1]
    q_heads, head_dim = q.shape
    _check("lq_attention_decode", _get_lib().lq_attention_decode(
        _lattice_id(lattice), _ptr(k_codes), _ptr(k_scales), _ptr(k_signs), _ptr(v_codes), _ptr(v_scales),
        _ptr(v_signs), tokens, kv_heads, q_heads, head_dim, _ptr(q), _dtype_id(q), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


# Scale formats (LQ_SCALE_* in lq.h)
LQ_SCALE_TILE_F32, LQ_SCALE_ROW_BF16, LQ_SCALE_TILE_F16 = 0, 1, 2
_SCALE_FORMATS = {"tile_f32": 0, "row_bf16": 1, "tile_f16": 2}


def _scale_format_id(fmt) -> int:
    return int(_SCALE_FORMATS.get(fmt, fmt))


def scales_tensor(rows: int, cols: int, tile: int, scale_format, device):
    """Empty scale tensor of the shape and dtype `scale_format` stores."""
    import torch
    f = _scale_format_id(scale_format)
    if f == LQ_SCALE_ROW_BF16:
        return torch.empty((rows,), dtype=torch.bfloat16, device=device)
    dt = torch.float16 if f == LQ_SCALE_TILE_F16 else torch.float32
    return torch.empty((rows, cols // tile), dtype=dt, device=device)


def lq_quantize_ex(lattice, W, tile: int, seed: int, beta: float, scale_format, codes, scales, signs,
                   dev_status=None, stream=None) -> None:
    """lq_quantize storing the scales in `scale_format` ("tile_f32", "row_bf16", "tile_f16")."""
    rows, cols = W.shape
    _check("lq_quantize_ex", _get_lib().lq_quantize_ex(
        _lattice_id(lattice), _ptr(W), _dtype_id(W), rows, cols, _row_stride(W), int(tile),
        int(seed) & 0xFFFFFFFFFFFFFFFF, float(beta), _scale_format_id(scale_format), _ptr(codes), _ptr(scales),
        _ptr(signs), _ptr(dev_status), _stream(stream)))


def quantize_ex(W, lattice: str = "e8", tile: int = 256, seed: int = 0, beta: float = 0.25,
                scale_format="tile_f32", dev_status=None, stream=None):
    """Allocate outputs and call :func:`lq_quantize_ex`; returns (codes, scales, signs)."""
    import torch
    rows, cols = W.shape
    codes = torch.empty((rows, cols), dtype=torch.int8, device=W.device)
    scales = scales_tensor(rows, cols, tile, scale_format, W.device)
    signs = torch.empty((cols,), dtype=torch.int8, device=W.device)
    lq_quantize_ex(lattice, W, tile, seed, beta, scale_format, codes, scales, signs, dev_status, stream)
    return codes, scales, signs


def lq_dequantize_ex(lattice, codes, scales, scale_format, signs, tile: int, W_hat, stream=None) -> None:
    rows, cols = codes.shape
    _check("lq_dequantize_ex", _get_lib().lq_dequantize_ex(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _scale_format_id(scale_format), _ptr(signs), rows, cols,
        int(tile), _ptr(W_hat), _dtype_id(W_hat), _stream(stream)))


def lq_gemv_ex(lattice, codes, scales, scale_format, signs, tile: int, x, y, workspace, dev_status=None,
               stream=None) -> None:
    rows, cols = codes.shape
    _check("lq_gemv_ex", _get_lib().lq_gemv_ex(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _scale_format_id(scale_format), _ptr(signs), rows, cols,
        int(tile), _ptr(x), _dtype_id(x), x.shape[0], _ptr(y), _ptr(workspace), _ptr(dev_status),
        _stream(stream)))


def lq_gemm_ex(lattice, codes, scales, scale_format, signs, tile: int, X, Y, workspace, dev_status=None,
               stream=None) -> None:
    N, K = codes.shape
    _check("lq_gemm_ex", _get_lib().lq_gemm_ex(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _scale_format_id(scale_format), _ptr(signs), N, K,
        int(tile), _ptr(X), X.shape[0], _ptr(Y), _dtype_id(Y), _ptr(workspace), _ptr(dev_status),
        _stream(stream)))


def lq_attention_decode_ex(lattice, k_codes, k_scales, k_signs, v_codes, v_scales, v_signs, scale_format, q, out,
                           workspace, stream=None) -> None:
    tokens = k_codes.shape[0]
    kv_heads = k_scales.shape[1]
    q_heads, head_dim = q.shape
    _check("lq_attention_decode_ex", _get_lib().lq_attention_decode_ex(
        _lattice_id(lattice), _ptr(k_codes), _ptr(k_scales), _ptr(k_signs), _ptr(v_codes), _ptr(v_scales),
        _ptr(v_signs), _scale_format_id(scale_format), tokens, kv_heads, q_heads, head_dim, _ptr(q), _dtype_id(q),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def lq_quantize_dithered(lattice, W, tile: int, seed: int, dither_seed: int, beta: float, scale_format, codes,
                         scales, signs, dev_status=None, stream=None) -> None:
    """lq_quantize with the subtractive Voronoi dither of seed `dither_seed`."""
    rows, cols = W.shape
    _check("lq_quantize_dithered", _get_lib().lq_quantize_dithered(
        _lattice_id(lattice), _ptr(W), _dtype_id(W), rows, cols, _row_stride(W), int(tile),
        int(seed) & 0xFFFFFFFFFFFFFFFF, int(dither_seed) & 0xFFFFFFFFFFFFFFFF, float(beta),
        _scale_format_id(scale_format), _ptr(codes), _ptr(scales), _ptr(signs), _ptr(dev_status), _stream(stream)))


def quantize_dithered(W, lattice: str = "e8", tile: int = 128, seed: int = 0, dither_seed: int = 1,
                      beta: float = 0.25, scale_format="tile_f32", dev_status=None, stream=None):
    """Allocate outputs and call :func:`lq_quantize_dithered`; returns (codes, scales, signs)."""
    import torch
    rows, cols = W.shape
    codes = torch.empty((rows, cols), dtype=torch.int8, device=W.device)
    scales = scales_tensor(rows, cols, tile, scale_format, W.device)
    signs = torch.empty((cols,), dtype=torch.int8, device=W.device)
    lq_quantize_dithered(lattice, W, tile, seed, dither_seed, beta, scale_format, codes, scales, signs, dev_status,
                         stream)
    return codes, scales, signs


def lq_dequantize_dithered(lattice, codes, scales, scale_format, signs, dither_seed: int, tile: int, W_hat,
                           stream=None) -> None:
    rows, cols = codes.shape
    _check("lq_dequantize_dithered", _get_lib().lq_dequantize_dithered(
        _lattice_id(lattice), _ptr(codes), _ptr(scales), _scale_format_id(scale_format), _ptr(signs),
        int(dither_seed) & 0xFFFFFFFFFFFFFFFF, rows, cols, int(tile), _ptr(W_hat), _dtype_id(W_hat),
        _stream(stream)))


def lq_attention_decode_dithered(lattice, k_codes, k_scales, k_signs, k_dither_seed: int, v_codes, v_scales,
                                 v_signs, v_dither_seed: int, scale_format, q, out, workspace, stream=None) -> None:
    tokens = k_codes.shape[0]
    kv_heads = k_scales.shape[1]
    q_heads, head_dim = q.shape
    _check("lq_attention_decode_dithered", _get_lib().lq_attention_decode_dithered(
        _lattice_id(lattice), _ptr(k_codes), _ptr(k_scales), _ptr(k_signs), int(k_dither_seed) & 0xFFFFFFFFFFFFFFFF,
        _ptr(v_codes), _ptr(v_scales), _ptr(v_signs), int(v_dither_seed) & 0xFFFFFFFFFFFFFFFF,
        _scale_format_id(scale_format), tokens, kv_heads, q_heads, head_dim, _ptr(q), _dtype_id(q), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def lq_attention_decode_rice(lattice, k_stream, k_offsets, k_scales, k_signs, v_stream, v_offsets, v_scales,
                             v_signs, scale_format, q, out, workspace, stream=None) -> None:
    """Decode attention over Rice-coded caches (streams and offsets from lq_rice_encode, tile = head_dim)."""
    tokens, kv_heads = k_offsets.shape
    q_heads, head_dim = q.shape
    _check("lq_attention_decode_rice", _get_lib().lq_attention_decode_rice(
        _lattice_id(lattice), _ptr(k_stream), k_stream.numel() * k_stream.element_size(), _ptr(k_offsets),
        _ptr(k_scales), _ptr(k_signs), _ptr(v_stream), v_stream.numel() * v_stream.element_size(), _ptr(v_offsets),
        _ptr(v_scales), _ptr(v_signs), _scale_format_id(scale_format), tokens, kv_heads, q_heads, head_dim, _ptr(q),
        _dtype_id(q), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def lq_rotate_blocks(R, X, Y, transpose: bool = False, stream=None) -> None:
    """Y (float32) = every 128-column block of X rotated by R (or R^T)."""
    rows, cols = X.shape
    _check("lq_rotate_blocks", _get_lib().lq_rotate_blocks(
        _ptr(R), int(bool(transpose)), R.shape[0], _ptr(X), _dtype_id(X), rows, cols, X.stride(0), _ptr(Y),
        Y.stride(0), _stream(stream)))


# ------------------------------------------------------------------ allocating helpers
def quantize(W, lattice: str = "e8", tile: int = 256, seed: int = 0, beta: float = 0.25,
             dev_status=None, stream=None):
    """Allocate outputs with torch on W's device and call :func:`lq_quantize`.

    Returns (codes int8 [rows x cols], scales float32 [rows x cols/tile], signs int8 [cols]).
    """
    import torch
    rows, cols = W.shape
    codes = torch.empty((rows, cols), dtype=torch.int8, device=W.device)
    scales = torch.empty((rows, cols // tile), dtype=torch.float32, device=W.device)
    signs = torch.empty((cols,), dtype=torch.int8, device=W.device)
    lq_quantize(lattice, W, tile, seed, beta, codes, scales, signs, dev_status, stream)
    return codes, scales, signs


def dequantize(codes, scales, signs, lattice: str = "e8", tile: int = 256, dtype=None, stream=None):
    import torch
    dtype = torch.float32 if dtype is None else dtype
    out = torch.empty(codes.shape, dtype=dtype, device=codes.device)
    lq_dequantize(lattice, codes, scales, signs, tile, out, stream)
    return out


def gemv(codes, scales, signs, x, lattice: str = "e8", tile: int = 256, workspace=None,
         dev_status=None, stream=None):
    import torch
    rows, cols = codes.shape
    y = torch.empty((x.shape[0], rows), dtype=torch.float32, device=codes.device)
    if workspace is None:
        workspace = torch.empty(lq_gemv_workspace_size(x.shape[0], cols, tile), dtype=torch.uint8,
                                device=codes.device)
    lq_gemv(lattice, codes, scales, signs, tile, x, y, workspace, dev_status, stream)
    return y


def gemm(codes, scales, signs, X, lattice: str = "e8", tile: int = 256, workspace=None,
         dev_status=None, stream=None, out_dtype=None):
    import torch
    N, K = codes.shape
    M = X.shape[0]
    Y = torch.empty((M, N), dtype=out_dtype or torch.float32, device=codes.device)
    if workspace is None:
        workspace = torch.empty(lq_gemm_workspace_size(M, N, K, _dtype_id(Y)), dtype=torch.uint8,
                                device=codes.device)
    lq_gemm(lattice, codes, scales, signs, tile, X, Y, workspace, dev_status, stream)
    return Y


# ------------------------------------------------------------------ checkpoint
CHECKPOINT_FORMAT = "lq-codes-v1"


def save_quantized(path, codes, scales, signs, lattice: str, tile: int, seed: int, beta: float,
                   scale_format="tile_f32", dither_seed=None) -> None:
    """Write codes, scales and signs with the header needed to use them again
    (lattice, tile, seed, beta, shape, scale format, and the dither seed of a
    dithered quantization or None) in one torch.save file."""
    import torch
    fmt = {v: k for k, v in _SCALE_FORMATS.items()}.get(_scale_format_id(scale_format))
    if fmt is None:
        raise ValueError(f"unknown scale format {scale_format!r}")
    torch.save({"format": CHECKPOINT_FORMAT, "lattice": str(lattice), "tile": int(tile), "seed": int(seed),
                "beta": float(beta), "shape": list(codes.shape), "scale_format": fmt,
                "dither_seed": None if dither_seed is None else int(dither_seed), "codes": codes.detach().cpu(),
                "scales": scales.detach().cpu(), "signs": signs.detach().cpu()}, path)


def load_quantized(path, device=None) -> dict:
    """Read a file written by :func:`save_quantized`; tensors moved to `device` when given.
    Files written before the scale formats existed read as float32 tile scales."""
    import torch
    d = torch.load(path, map_location="cpu", weights_only=True)
    if d.get("format") != CHECKPOINT_FORMAT:
        raise ValueError(f"{path}: not a {CHECKPOINT_FORMAT} file")
    d.setdefault("scale_format", "tile_f32")
    d.setdefault("dither_seed", None)
    rows, cols = d["shape"]
    want_scales = (rows,) if d["scale_format"] == "row_bf16" else (rows, cols // d["tile"])
    if tuple(d["codes"].shape) != (rows, cols) or tuple(d["scales"].shape) != want_scales \
            or tuple(d["signs"].shape) != (cols,):
        raise ValueError(f"{path}: tensor shapes do not match the header")
    if device is not None:
        for k in ("codes", "scales", "signs"):
            d[k] = d[k].to(device)
    return d

