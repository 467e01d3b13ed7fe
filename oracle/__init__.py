"""thinmx CPU oracle — TEST INFRASTRUCTURE, not part of the product.

A ctypes front end over ``thinmx_oracle.c`` (plain C, fp64, single thread).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``bit_weight_only_mxfp4_gb300``; the two meet only on the seeded
inputs of ``bit_weight_only_mxfp4_gb300.synth``.

Every function is pinned in ``tests/test_oracle_pins.py``; the sources each
one follows are listed in ``thinmx_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "thinmx_oracle.c")
_HDR = os.path.join(_HERE, "thinmx_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_SHAPE = 2
ERR_NONFINITE = 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C99, no FP contraction, so that x86
    and Arm hosts give identical results)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            _declare(lib)
            _lib = lib
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def _declare(lib):
    sig = {
        "orc_e2m1_value": (ctypes.c_double, [ctypes.c_uint]),
        "orc_e8m0_value": (ctypes.c_double, [ctypes.c_uint]),
        "orc_e2m1_encode": (ctypes.c_uint, [ctypes.c_double]),
        "orc_floor_log2": (ctypes.c_int, [ctypes.c_float]),
        "orc_bf16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_f16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_f16_round": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_mxfp4_quantize": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
        "orc_mxfp4_dequantize": (None, [_P, _P, _I64, _I64, _P]),
        "orc_mxfp4_matvec": (None, [_P, _P, _P, _I64, _I64, _P, _I64, _P]),
        "orc_bf16_matvec": (None, [_P, _I64, _I64, _P, _I64, _P]),
        "orc_swiglu": (None, [_P, _P, _I64, _P]),
        "orc_mxfp4_swiglu_matvec": (None, [_P, _P, _P, _P, _P, _P, _I64, _I64,
                                           _P, _I64, _P]),
        "orc_bf16_swiglu_matvec": (None, [_P, _P, _I64, _I64, _P, _I64, _P]),
        "orc_router_logits": (None, [_P, _P, _I32, _I64, _P]),
        "orc_topk": (None, [_P, _I32, _I32, _P]),
        "orc_softmax_selected": (None, [_P, _P, _I32, _P]),
        "orc_moe_mlp": (ctypes.c_int, [_P, _I64, _I64, _P, _I32, _I32, _P, _P,
                                       _P, _P, _P, _P, _P, _P]),
        "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint]),
        "orc_e4m3_encode": (ctypes.c_uint, [ctypes.c_double]),
        "orc_fp8_quantize": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
        "orc_fp8_dequantize": (None, [_P, _P, _I64, _I64, _P]),
        "orc_fp8_matvec": (None, [_P, _P, _I64, _I64, _P, _I64, _P]),
        "orc_fp8_swiglu_matvec": (None, [_P, _P, _P, _P, _I64, _I64, _P, _I64, _P]),
        "orc_gqa_decode": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _I64, _I64,
                                          ctypes.c_double, _P]),
        "orc_lowbit_plane_bytes": (_I64, [_I64]),
        "orc_lowbit_scale_bytes": (_I64, [_I64]),
        "orc_lowbit_matrix_bytes": (_I64, [_I32, _I64, _I64]),
        "orc_lowbit_quantize": (ctypes.c_int, [_I32, _P, _I64, _I64, _P]),
        "orc_lowbit_dequantize": (None, [_I32, _P, _I64, _I64, _P]),
        "orc_moe_lowbit_mlp": (ctypes.c_int, [_I32, _P, _I64, _I64, _P, _I32, _I32, _P, _P,
                                              _P, _P, _P, _P, _P]),
        "orc_int4_quantize": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P]),
        "orc_int4_dequantize": (None, [_P, _P, _P, _I64, _I64, _I32, _P]),
        "orc_int4_matvec": (None, [_P, _P, _P, _I64, _I64, _I32, _P, _I64, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar formats -------------------------------------------------------
def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(int(byte))


def e2m1_encode(t: float) -> int:
    return int(_load().orc_e2m1_encode(float(t)))


def floor_log2(a: float) -> int:
    return int(_load().orc_floor_log2(float(np.float32(a))))


def bf16_value(b: int) -> float:
    return _load().orc_bf16_value(int(b))


def bf16_round(v: float) -> int:
    return int(_load().orc_bf16_round(float(v)))


def f16_value(h: int) -> float:
    return _load().orc_f16_value(int(h))


def f16_round(v: float) -> int:
    return int(_load().orc_f16_round(float(v)))


def bf16_round_array(v) -> np.ndarray:
    """fp64 array -> bf16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    flat = np.asarray(v, dtype=np.float64).ravel()
    out = np.fromiter((lib.orc_bf16_round(float(t)) for t in flat),
                      dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(v))


# ---- MXFP4 ----------------------------------------------------------------
def mxfp4_quantize(w):
    """fp32 [n, k] -> (codes u8 [n, k/2], scales u8 [n, k/32], status)."""
    w = _c(w, np.float32)
    n, k = w.shape
    codes = np.zeros((n, k // 2), np.uint8)
    scales = np.zeros((n, k // 32), np.uint8)
    st = _load().orc_mxfp4_quantize(_ptr(w), n, k, _ptr(codes), _ptr(scales))
    return codes, scales, st


def mxfp4_dequantize(codes, scales):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n = codes.shape[0]
    k = codes.shape[1] * 2
    out = np.zeros((n, k), np.float64)
    _load().orc_mxfp4_dequantize(_ptr(codes), _ptr(scales), n, k, _ptr(out))
    return out


def mxfp4_matvec(codes, scales, postscale, x_bf16):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n = codes.shape[0]
    k = codes.shape[1] * 2
    m = x.shape[0]
    ps = None if postscale is None else _c(postscale, np.float32)
    y = np.zeros((m, n), np.float64)
    _load().orc_mxfp4_matvec(_ptr(codes), _ptr(scales), _ptr(ps), n, k,
                             _ptr(x), m, _ptr(y))
    return y


def bf16_matvec(w_bf16, x_bf16):
    w = _c(w_bf16, np.uint16)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n, k = w.shape
    m = x.shape[0]
    y = np.zeros((m, n), np.float64)
    _load().orc_bf16_matvec(_ptr(w), n, k, _ptr(x), m, _ptr(y))
    return y


def swiglu(g, u):
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    h = np.zeros_like(g)
    _load().orc_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def mxfp4_swiglu_matvec(gate, up, x_bf16):
    """gate/up: (codes, scales, postscale-or-None).  Returns fp64 [m, n]."""
    gc, gs, gp = (_c(gate[0], np.uint8), _c(gate[1], np.uint8),
                  None if gate[2] is None else _c(gate[2], np.float32))
    uc, us, up_ = (_c(up[0], np.uint8), _c(up[1], np.uint8),
                   None if up[2] is None else _c(up[2], np.float32))
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n = gc.shape[0]
    k = gc.shape[1] * 2
    m = x.shape[0]
    h = np.zeros((m, n), np.float64)
    _load().orc_mxfp4_swiglu_matvec(_ptr(gc), _ptr(gs), _ptr(gp), _ptr(uc),
                                    _ptr(us), _ptr(up_), n, k, _ptr(x), m,
                                    _ptr(h))
    return h


def bf16_swiglu_matvec(wg, wu, x_bf16):
    wg = _c(wg, np.uint16)
    wu = _c(wu, np.uint16)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n, k = wg.shape
    m = x.shape[0]
    h = np.zeros((m, n), np.float64)
    _load().orc_bf16_swiglu_matvec(_ptr(wg), _ptr(wu), n, k, _ptr(x), m,
                                   _ptr(h))
    return h


# ---- MoE ------------------------------------------------------------------
def router_logits(x_bf16, wr_bf16):
    x = _c(x_bf16, np.uint16).ravel()
    wr = _c(wr_bf16, np.uint16)
    e, k = wr.shape
    out = np.zeros(e, np.float64)
    _load().orc_router_logits(_ptr(x), _ptr(wr), e, k, _ptr(out))
    return out


def topk(logits32, top_k):
    lg = _c(logits32, np.float32)
    idx = np.zeros(top_k, np.int32)
    _load().orc_topk(_ptr(lg), lg.size, top_k, _ptr(idx))
    return idx


def softmax_selected(logits32, idx):
    lg = _c(logits32, np.float32)
    idx = _c(idx, np.int32)
    p = np.zeros(idx.size, np.float64)
    _load().orc_softmax_selected(_ptr(lg), _ptr(idx), idx.size, _ptr(p))
    return p


def moe_mlp(x_bf16, wr_bf16, top_k, gu_codes, gu_scales, dn_codes, dn_scales):
    """Stacked experts: gu_codes [E, 2I, H/2], gu_scales [E, 2I, H/32],
    dn_codes [E, H, I/2], dn_scales [E, H, I/32].  Returns
    (out fp64 [H], idx [top_k], p fp64 [top_k], logits32 [E], status)."""
    x = _c(x_bf16, np.uint16).ravel()
    wr = _c(wr_bf16, np.uint16)
    gc = _c(gu_codes, np.uint8)
    gs = _c(gu_scales, np.uint8)
    dc = _c(dn_codes, np.uint8)
    ds = _c(dn_scales, np.uint8)
    e, hidden = wr.shape
    inter = gc.shape[1] // 2
    out = np.zeros(hidden, np.float64)
    idx = np.zeros(top_k, np.int32)
    p = np.zeros(top_k, np.float64)
    lg = np.zeros(e, np.float32)
    st = _load().orc_moe_mlp(_ptr(x), hidden, inter, _ptr(wr), e, top_k,
                             _ptr(gc), _ptr(gs), _ptr(dc), _ptr(ds), _ptr(out),
                             _ptr(idx), _ptr(p), _ptr(lg))
    return out, idx, p, lg, st


# ---- grouped affine INT4 --------------------------------------------------
def int4_quantize(w, group):
    w = _c(w, np.float32)
    n, k = w.shape
    ng = (k + group - 1) // group
    codes = np.zeros((n, k // 2), np.uint8)
    scales = np.zeros((n, ng), np.uint16)
    zp = np.zeros((n, (ng + 1) // 2), np.uint8)
    st = _load().orc_int4_quantize(_ptr(w), n, k, group, _ptr(codes),
                                   _ptr(scales), _ptr(zp))
    return codes, scales, zp, st


def int4_dequantize(codes, scales_f16, zp, group):
    codes = _c(codes, np.uint8)
    sc = _c(scales_f16, np.uint16)
    zp = _c(zp, np.uint8)
    n = codes.shape[0]
    k = codes.shape[1] * 2
    out = np.zeros((n, k), np.float64)
    _load().orc_int4_dequantize(_ptr(codes), _ptr(sc), _ptr(zp), n, k, group,
                                _ptr(out))
    return out


def int4_matvec(codes, scales_f16, zp, group, x_bf16):
    codes = _c(codes, np.uint8)
    sc = _c(scales_f16, np.uint16)
    zp = _c(zp, np.uint8)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n = codes.shape[0]
    k = codes.shape[1] * 2
    m = x.shape[0]
    y = np.zeros((m, n), np.float64)
    _load().orc_int4_matvec(_ptr(codes), _ptr(sc), _ptr(zp), n, k, group,
                            _ptr(x), m, _ptr(y))
    return y


# ---- FP8 (E4M3) with one fp32 scale per row [DL3] -------------------------
def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(code)


def e4m3_encode(t: float) -> int:
    return _load().orc_e4m3_encode(float(t))


def fp8_quantize(w):
    """fp32 [n, k] -> (codes uint8 [n, k], scales fp32 [n], status)."""
    w = _c(w, np.float32)
    n, k = w.shape
    codes = np.zeros((n, k), np.uint8)
    scales = np.zeros(n, np.float32)
    st = _load().orc_fp8_quantize(_ptr(w), n, k, _ptr(codes), _ptr(scales))
    return codes, scales, st


def fp8_dequantize(codes, scales):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n, k = codes.shape
    out = np.zeros((n, k), np.float64)
    _load().orc_fp8_dequantize(_ptr(codes), _ptr(scales), n, k, _ptr(out))
    return out


def fp8_matvec(codes, scales, x_bf16):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n, k = codes.shape
    m = x.shape[0]
    y = np.zeros((m, n), np.float64)
    _load().orc_fp8_matvec(_ptr(codes), _ptr(scales), n, k, _ptr(x), m, _ptr(y))
    return y


def fp8_swiglu_matvec(gate, up, x_bf16):
    """gate/up: (codes, scales).  Returns fp64 [m, n]."""
    gc, gs = _c(gate[0], np.uint8), _c(gate[1], np.float32)
    uc, us = _c(up[0], np.uint8), _c(up[1], np.float32)
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    n, k = gc.shape
    m = x.shape[0]
    h = np.zeros((m, n), np.float64)
    _load().orc_fp8_swiglu_matvec(_ptr(gc), _ptr(gs), _ptr(uc), _ptr(us), n, k,
                                  _ptr(x), m, _ptr(h))
    return h


# ---- single-token GQA attention [DL3] --------------------------------------
def gqa_decode(q_bf16, k_bf16, v_bf16, length, scale):
    """q [heads, d]; k, v [kv_heads, cap, d] bf16 bits; attends over the
    first `length` tokens.  Returns (o fp64 [heads, d], status)."""
    q = _c(q_bf16, np.uint16)
    k = _c(k_bf16, np.uint16)
    v = _c(v_bf16, np.uint16)
    heads, d = q.shape
    kvh, cap, _ = k.shape
    o = np.zeros((heads, d), np.float64)
    st = _load().orc_gqa_decode(_ptr(q), _ptr(k), _ptr(v), heads, kvh, d, cap, int(length),
                                float(scale), _ptr(o))
    return o, st


# ---- Q1 / Q2 packed low-bit experts ----------------------------------------
def lowbit_matrix_bytes(bits, n, k) -> int:
    return int(_load().orc_lowbit_matrix_bytes(bits, n, k))


def lowbit_plane_bytes(k) -> int:
    return int(_load().orc_lowbit_plane_bytes(k))


def lowbit_scale_bytes(k) -> int:
    return int(_load().orc_lowbit_scale_bytes(k))


def lowbit_quantize(bits, w):
    """fp32 [n, k] -> (buffer uint8 [lowbit_matrix_bytes], status)."""
    w = _c(w, np.float32)
    n, k = w.shape
    buf = np.zeros(lowbit_matrix_bytes(bits, n, k), np.uint8)
    st = _load().orc_lowbit_quantize(bits, _ptr(w), n, k, _ptr(buf))
    return buf, st


def lowbit_dequantize(bits, buf, n, k):
    buf = _c(buf, np.uint8)
    out = np.zeros((n, k), np.float64)
    _load().orc_lowbit_dequantize(bits, _ptr(buf), n, k, _ptr(out))
    return out


def moe_lowbit_mlp(bits, x_bf16, wr_bf16, top_k, gu, dn, inter):
    """gu [E, gate/up matrix bytes] ([2 inter][hidden] each), dn [E, down
    matrix bytes] ([hidden][inter] each).  Returns (out fp64 [hidden],
    idx [top_k], p fp64 [top_k], logits32 [E], h fp64 [top_k, inter],
    status)."""
    x = _c(x_bf16, np.uint16).ravel()
    wr = _c(wr_bf16, np.uint16)
    gu = _c(gu, np.uint8)
    dn = _c(dn, np.uint8)
    e, hidden = wr.shape
    out = np.zeros(hidden, np.float64)
    idx = np.zeros(top_k, np.int32)
    p = np.zeros(top_k, np.float64)
    lg = np.zeros(e, np.float32)
    h = np.zeros((top_k, inter), np.float64)
    st = _load().orc_moe_lowbit_mlp(bits, _ptr(x), hidden, inter, _ptr(wr), e, top_k,
                                    _ptr(gu), _ptr(dn), _ptr(out), _ptr(idx), _ptr(p),
                                    _ptr(lg), _ptr(h))
    return out, idx, p, lg, h, st

