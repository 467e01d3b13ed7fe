"""Thin Python binding over libthinmx.so (include/thinmx.h).

Each ``tt_*`` function here has the same name and argument order as the C
entry point; it only marshals torch tensors into device pointers and the
current CUDA stream, calls the library, and raises ``ThinmxError`` on a
non-OK status.  All arithmetic runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback — if the library is missing the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libthinmx.so")

STATUS = {
    0: "TT_OK", 1: "TT_ERR_NULL", 2: "TT_ERR_SHAPE", 3: "TT_ERR_ALIGN",
    4: "TT_ERR_NONFINITE", 5: "TT_ERR_UNSUPPORTED", 6: "TT_ERR_CUDA",
    7: "TT_ERR_TIMEOUT", 8: "TT_ERR_SIZE",
}
TT_OK = 0

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/thinmx.h
SIGNATURES = {
    "tt_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "tt_version": (ctypes.c_int, []),
    "tt_device_error_read": (ctypes.c_int, [_P]),
    "tt_quantize_mxfp4": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P]),
    "tt_mxfp4_dequantize": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "tt_mxfp4_swiglu_packed_bytes": (_SZ, [_I64, _I64]),
    "tt_mxfp4_pack_swiglu": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "tt_mxfp4_swiglu_matvec": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_bf16_swiglu_matvec": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_mxfp4_matvec": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_bf16_matvec": (ctypes.c_int, [_P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_mxfp4_rows_packed_bytes": (_SZ, [_I64, _I64]),
    "tt_mxfp4_pack_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _SZ, _P]),
    "tt_moe_workspace_bytes": (_SZ, [_I64, _I64, _I32, _I32]),
    "tt_moe_mxfp4_topk_mlp": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P,
                                              _P, _SZ, _P]),
    "tt_moe_mxfp4_topk_mlp_static": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _P,
                                                     _P, _P, _P]),
    "tt_quantize_fp8": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P]),
    "tt_fp8_matvec": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_fp8_swiglu_matvec": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "tt_quantize_int4_grouped": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P, _P, _P]),
    "tt_int4_grouped_matvec": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _P, _I64, _P, _P]),
    "tt_lowbit_matrix_bytes": (_SZ, [_I32, _I64, _I64]),
    "tt_quantize_lowbit": (ctypes.c_int, [_I32, _P, _I64, _I64, _P, _SZ, _P, _P]),
    "tt_moe_lowbit_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "tt_moe_lowbit_topk_mlp": (ctypes.c_int, [_I32, _P, _I64, _I64, _P, _I32, _I32, _P, _P,
                                               _P, _P, _P, _P, _SZ, _P]),
    "tt_gqa_decode_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "tt_gqa_decode_attention": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _I64, _I64,
                                                ctypes.c_float, _P, _P, _SZ, _P]),
}


class ThinmxError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:  # fast path of every call after the first
        return lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with bit_weight_only_mxfp4_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_torch = None


def _current_stream() -> int:
    """Raw handle of torch's current CUDA stream on the current device."""
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    raw = getattr(_torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(_torch._C._cuda_getDevice())
    return _torch.cuda.current_stream().cuda_stream


def _stream(stream):
    if stream is None:
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != TT_OK:
        raise ThinmxError(fn, st)


# ---------------------------------------------------------------- entry points
def tt_status_str(status: int) -> str:
    return load().tt_status_str(status).decode()


def tt_version() -> int:
    return load().tt_version()


def tt_device_error_read() -> int:
    out = ctypes.c_int32(0)
    _check("tt_device_error_read", load().tt_device_error_read(ctypes.addressof(out)))
    return out.value


def tt_quantize_mxfp4(w, n, k, codes, scales, status_dev=None, stream=None):
    _check("tt_quantize_mxfp4", load().tt_quantize_mxfp4(
        _ptr(w), n, k, _ptr(codes), _ptr(scales), _ptr(status_dev), _stream(stream)))


def tt_mxfp4_dequantize(codes, scales, n, k, out, stream=None):
    _check("tt_mxfp4_dequantize", load().tt_mxfp4_dequantize(
        _ptr(codes), _ptr(scales), n, k, _ptr(out), _stream(stream)))


def tt_mxfp4_swiglu_packed_bytes(n, k) -> int:
    return int(load().tt_mxfp4_swiglu_packed_bytes(n, k))


def tt_mxfp4_pack_swiglu(gate_codes, gate_scales, gate_postscale, up_codes, up_scales,
                         up_postscale, n, k, packed, packed_bytes, stream=None):
    _check("tt_mxfp4_pack_swiglu", load().tt_mxfp4_pack_swiglu(
        _ptr(gate_codes), _ptr(gate_scales), _ptr(gate_postscale), _ptr(up_codes),
        _ptr(up_scales), _ptr(up_postscale), n, k, _ptr(packed), packed_bytes,
        _stream(stream)))


def tt_mxfp4_swiglu_matvec(packed, n, k, x_bf16, m, h_bf16, stream=None):
    _check("tt_mxfp4_swiglu_matvec", load().tt_mxfp4_swiglu_matvec(
        _ptr(packed), n, k, _ptr(x_bf16), m, _ptr(h_bf16), _stream(stream)))


def tt_bf16_swiglu_matvec(wg, wu, n, k, x_bf16, m, h_bf16, stream=None):
    _check("tt_bf16_swiglu_matvec", load().tt_bf16_swiglu_matvec(
        _ptr(wg), _ptr(wu), n, k, _ptr(x_bf16), m, _ptr(h_bf16), _stream(stream)))


def tt_quantize_fp8(w, n, k, codes, scales, status_dev=None, stream=None):
    _check("tt_quantize_fp8", load().tt_quantize_fp8(
        _ptr(w), n, k, _ptr(codes), _ptr(scales), _ptr(status_dev), _stream(stream)))


def tt_fp8_matvec(codes, scales, n, k, x_bf16, m, y_bf16, stream=None):
    _check("tt_fp8_matvec", load().tt_fp8_matvec(
        _ptr(codes), _ptr(scales), n, k, _ptr(x_bf16), m, _ptr(y_bf16), _stream(stream)))


def tt_fp8_swiglu_matvec(gate_codes, gate_scales, up_codes, up_scales, n, k, x_bf16, m, h_bf16,
                         stream=None):
    _check("tt_fp8_swiglu_matvec", load().tt_fp8_swiglu_matvec(
        _ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes), _ptr(up_scales), n, k,
        _ptr(x_bf16), m, _ptr(h_bf16), _stream(stream)))


def tt_quantize_int4_grouped(w, n, k, group, codes, scales_f16, zp_u4, status_dev=None,
                             stream=None):
    _check("tt_quantize_int4_grouped", load().tt_quantize_int4_grouped(
        _ptr(w), n, k, group, _ptr(codes), _ptr(scales_f16), _ptr(zp_u4), _ptr(status_dev),
        _stream(stream)))


def tt_int4_grouped_matvec(codes, scales_f16, zp_u4, n, k, group, x_bf16, m, y_bf16,
                           stream=None):
    _check("tt_int4_grouped_matvec", load().tt_int4_grouped_matvec(
        _ptr(codes), _ptr(scales_f16), _ptr(zp_u4), n, k, group, _ptr(x_bf16), m, _ptr(y_bf16),
        _stream(stream)))


def tt_mxfp4_matvec(codes, scales, postscale, n, k, x_bf16, m, y_bf16, stream=None):
    _check("tt_mxfp4_matvec", load().tt_mxfp4_matvec(
        _ptr(codes), _ptr(scales), _ptr(postscale), n, k, _ptr(x_bf16), m, _ptr(y_bf16),
        _stream(stream)))


def tt_bf16_matvec(w, n, k, x_bf16, m, y_bf16, stream=None):
    _check("tt_bf16_matvec", load().tt_bf16_matvec(
        _ptr(w), n, k, _ptr(x_bf16), m, _ptr(y_bf16), _stream(stream)))


def tt_mxfp4_rows_packed_bytes(n, k) -> int:
    return int(load().tt_mxfp4_rows_packed_bytes(n, k))


def tt_mxfp4_pack_rows(codes, scales, n, k, packed, packed_bytes, stream=None):
    _check("tt_mxfp4_pack_rows", load().tt_mxfp4_pack_rows(
        _ptr(codes), _ptr(scales), n, k, _ptr(packed), packed_bytes, _stream(stream)))


def tt_moe_workspace_bytes(hidden, inter, n_experts, top_k) -> int:
    return int(load().tt_moe_workspace_bytes(hidden, inter, n_experts, top_k))


def tt_moe_mxfp4_topk_mlp(x_bf16, hidden, inter, router_w_bf16, n_experts, top_k,
                          gate_up_packed, down_packed, out_bf16, out_idx, out_prob, workspace,
                          workspace_bytes, stream=None):
    _check("tt_moe_mxfp4_topk_mlp", load().tt_moe_mxfp4_topk_mlp(
        _ptr(x_bf16), hidden, inter, _ptr(router_w_bf16), n_experts, top_k,
        _ptr(gate_up_packed), _ptr(down_packed), _ptr(out_bf16), _ptr(out_idx), _ptr(out_prob),
        _ptr(workspace), workspace_bytes, _stream(stream)))


# Largest top_k * inter the workspace-free MoE call accepts (its fixed scratch).
TT_MOE_STATIC_MAX_HIDDEN = 4096


def tt_moe_mxfp4_topk_mlp_static(x_bf16, hidden, inter, router_w_bf16, n_experts, top_k,
                                 gate_up_packed, down_packed, out_bf16, out_idx, out_prob,
                                 stream=None):
    """The MoE layer on the library's own fixed scratch: for callers that
    cannot allocate device memory (see include/thinmx.h)."""
    _check("tt_moe_mxfp4_topk_mlp_static", load().tt_moe_mxfp4_topk_mlp_static(
        _ptr(x_bf16), hidden, inter, _ptr(router_w_bf16), n_experts, top_k,
        _ptr(gate_up_packed), _ptr(down_packed), _ptr(out_bf16), _ptr(out_idx), _ptr(out_prob),
        _stream(stream)))


def tt_gqa_decode_workspace_bytes(heads, kv_heads, head_dim) -> int:
    return int(load().tt_gqa_decode_workspace_bytes(heads, kv_heads, head_dim))


def tt_gqa_decode_attention(q_bf16, k_cache, v_cache, heads, kv_heads, head_dim, cap, length,
                            scale, out_bf16, workspace, workspace_bytes, stream=None):
    _check("tt_gqa_decode_attention", load().tt_gqa_decode_attention(
        _ptr(q_bf16), _ptr(k_cache), _ptr(v_cache), heads, kv_heads, head_dim, cap, length,
        float(scale), _ptr(out_bf16), _ptr(workspace), workspace_bytes, _stream(stream)))


def tt_lowbit_matrix_bytes(bits, n, k) -> int:
    return int(load().tt_lowbit_matrix_bytes(bits, n, k))


def tt_quantize_lowbit(bits, w, n, k, buf, buf_bytes, status_dev=None, stream=None):
    _check("tt_quantize_lowbit", load().tt_quantize_lowbit(
        bits, _ptr(w), n, k, _ptr(buf), buf_bytes, _ptr(status_dev), _stream(stream)))


def tt_moe_lowbit_workspace_bytes(inter, n_experts, top_k) -> int:
    return int(load().tt_moe_lowbit_workspace_bytes(inter, n_experts, top_k))


def tt_moe_lowbit_topk_mlp(bits, x_bf16, hidden, inter, router_w_bf16, n_experts, top_k,
                           gate_up, down, out_bf16, out_idx, out_prob, workspace,
                           workspace_bytes, stream=None):
    _check("tt_moe_lowbit_topk_mlp", load().tt_moe_lowbit_topk_mlp(
        bits, _ptr(x_bf16), hidden, inter, _ptr(router_w_bf16), n_experts, top_k,
        _ptr(gate_up), _ptr(down), _ptr(out_bf16), _ptr(out_idx), _ptr(out_prob),
        _ptr(workspace), workspace_bytes, _stream(stream)))

