"""Host-side checks of the C ABI: the library builds for sm_103a, loads
without a GPU, exports every entry point declared in include/thinmx.h, and
rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from bit_weight_only_mxfp4_gb300 import build as tt_build
from bit_weight_only_mxfp4_gb300 import thinmx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tt_build.build()
    return thinmx.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "thinmx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tt_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_symbols()
    for required in ["tt_quantize_mxfp4", "tt_mxfp4_swiglu_matvec"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in thinmx.SIGNATURES, f"binding lacks {name}"


def declared_arities():
    """name -> number of parameters, from the prototypes in the header."""
    text = open(os.path.join(ROOT, "include", "thinmx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(tt_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = " ".join(params.split())
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    ar = declared_arities()
    assert set(ar) == set(declared_symbols())
    for name, n in ar.items():
        assert len(thinmx.SIGNATURES[name][1]) == n, name


def test_status_strings(lib):
    assert thinmx.tt_status_str(0) == "TT_OK"
    assert thinmx.tt_status_str(7) == "TT_ERR_TIMEOUT"
    assert thinmx.tt_status_str(99) == "TT_ERR_UNKNOWN"
    assert thinmx.tt_version() >= 10000


def test_packed_bytes_host_arithmetic(lib):
    # record = gate codes + up codes + both scale rows + 8 B of postscales, 16-B padded
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(11008, 2048) == 11008 * 2192
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(2880, 2880) == 2880 * 3072
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(17920, 5120) == 17920 * 5456
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(1, 32) == 48
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(1, 48) == 0      # k % 32 != 0
    assert thinmx.tt_mxfp4_swiglu_packed_bytes(0, 64) == 0


def _st(fn, *args):
    return getattr(thinmx.load(), fn)(*args)


def test_validation_before_launch(lib):
    A = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced
    s = None
    # shapes
    assert _st("tt_mxfp4_swiglu_matvec", A, 128, 48, A, 1, A, s) == 2
    assert _st("tt_mxfp4_swiglu_matvec", A, 0, 64, A, 1, A, s) == 2
    assert _st("tt_mxfp4_swiglu_matvec", A, 128, 64, A, 0, A, s) == 2
    assert _st("tt_mxfp4_swiglu_matvec", A, 128, 64, A, 65, A, s) == 2
    assert _st("tt_mxfp4_swiglu_matvec", A, 128, 32768, A, 1, A, s) == 2
    assert _st("tt_quantize_mxfp4", A, 4, 40, A, A, None, s) == 2
    # null pointers
    assert _st("tt_mxfp4_swiglu_matvec", None, 128, 64, A, 1, A, s) == 1
    assert _st("tt_quantize_mxfp4", None, 4, 64, A, A, None, s) == 1
    # alignment
    assert _st("tt_mxfp4_swiglu_matvec", A + 8, 128, 64, A, 1, A, s) == 3
    assert _st("tt_mxfp4_swiglu_matvec", A, 128, 64, A + 2, 1, A, s) == 3
    assert _st("tt_bf16_swiglu_matvec", A, A + 4, 16, 64, A, 1, A, s) == 3
    # caller buffer too small for the packed layout
    assert _st("tt_mxfp4_pack_swiglu", A, A, None, A, A, None, 16, 64, A, 100, s) == 8
    # empty quantise is a no-op
    assert _st("tt_quantize_mxfp4", None, 0, 64, None, None, None, s) == 0


def test_moe_validation_before_launch(lib):
    A = 1 << 20  # never dereferenced: every case fails validation first
    s = None
    ws = _st("tt_moe_workspace_bytes", 2880, 2880, 32, 4)
    assert ws >= 64 + 256 * 2880 * 4  # counters + one partial vector per CTA
    assert _st("tt_moe_workspace_bytes", 8224, 2880, 32, 4) == 0  # hidden beyond 8192
    assert _st("tt_moe_workspace_bytes", 2880, 2880, 4, 8) == 0   # top_k > n_experts
    call = lambda H, I, E, K, x=A, wsp=A, wsb=ws, tg=A, td=A: _st(
        "tt_moe_mxfp4_topk_mlp", x, H, I, A, E, K, tg, td, A, A, A, wsp, wsb, s)
    assert call(2880, 2880, 32, 4, wsb=ws - 1) == 8          # workspace too small
    assert call(8224, 2880, 32, 4, wsb=1 << 30) == 2          # hidden beyond 8192
    assert call(2880, 8224, 32, 4, wsb=1 << 30) == 2          # inter beyond 8192
    assert call(2880, 2880, 32, 9) == 2                       # top_k beyond 8
    assert call(2880, 2880, 257, 4) == 2                      # more than 256 experts
    assert call(2880, 2880, 32, 0) == 2
    assert call(2880, 2880, 32, 4, x=None) == 1
    assert call(2880, 2880, 32, 4, wsp=None) == 1
    assert call(2880, 2880, 32, 4, x=A + 8) == 3              # x not 16-byte aligned
    assert call(2880, 2880, 32, 4, wsp=A + 4) == 3            # workspace not 16-byte aligned
    assert call(2880, 2880, 32, 4, tg=None) == 1              # no gate/up expert table
    assert call(2880, 2880, 32, 4, td=A + 4) == 3             # expert table not 8-byte aligned


def test_fp8_validation_before_launch(lib):
    A = 1 << 20  # never dereferenced: every case fails validation first
    s = None
    mv = lambda n, k, m, codes=A, x=A: _st("tt_fp8_matvec", codes, A, n, k, x, m, A, s)
    sw = lambda n, k, m, uc=A: _st("tt_fp8_swiglu_matvec", A, A, uc, A, n, k, A, m, A, s)
    assert mv(2048, 11008, 9) == 2        # m beyond 8
    assert mv(2048, 11000, 1) == 2        # k not a multiple of 16
    assert mv(2048, 32768, 1) == 2        # k beyond 16384
    assert mv(0, 2048, 1) == 2
    assert mv(2048, 2048, 1, codes=None) == 1
    assert mv(2048, 2048, 1, codes=A + 8) == 3
    assert mv(2048, 2048, 1, x=A + 2) == 3
    assert sw(11008, 2048, 0) == 2
    assert sw(11008, 2048, 1, uc=None) == 1
    assert sw(11008, 2048, 1, uc=A + 4) == 3
    # the quantiser: an empty matrix is a no-op, a NULL output an error
    assert _st("tt_quantize_fp8", None, 0, 64, None, None, None, s) == 0
    assert _st("tt_quantize_fp8", A, 4, 64, None, A, None, s) == 1


def test_int4_validation_before_launch(lib):
    A = 1 << 20
    s = None
    call = lambda n, k, g, m, codes=A, x=A: _st("tt_int4_grouped_matvec", codes, A, A, n, k, g,
                                                 x, m, A, s)
    assert call(5120, 2880, 128, 9) == 2      # m beyond 8
    assert call(5120, 2880, 100, 1) == 2      # group not a multiple of 32
    assert call(5120, 2890, 128, 1) == 2      # k not a multiple of 32
    assert call(5120, 16384, 128, 1) == 2     # k beyond 8192
    assert call(0, 2880, 128, 1) == 2
    assert call(5120, 2880, 128, 1, codes=None) == 1
    assert call(5120, 2880, 128, 1, x=A + 2) == 3


def test_gqa_validation_before_launch(lib):
    A = 1 << 20  # never dereferenced: every case fails validation first
    s = None
    ws = _st("tt_gqa_decode_workspace_bytes", 64, 8, 64)
    # 256 split partials of 8 heads x (64 + 2) floats per kv head
    assert ws == 8 * 256 * 8 * 66 * 4
    assert _st("tt_gqa_decode_workspace_bytes", 16, 4, 128) == 4 * 256 * 4 * 130 * 4
    assert _st("tt_gqa_decode_workspace_bytes", 12, 1, 64) == 256 * 12 * 66 * 4
    assert _st("tt_gqa_decode_workspace_bytes", 15, 4, 128) == 0   # not a group
    assert _st("tt_gqa_decode_workspace_bytes", 16, 4, 96) == 0    # head_dim
    assert _st("tt_gqa_decode_workspace_bytes", 68, 4, 64) == 0    # 17-wide groups
    assert _st("tt_gqa_decode_workspace_bytes", 65, 65, 64) == 0   # more than 64 kv heads
    call = lambda heads=64, kvh=8, d=64, cap=4096, ln=4096, scale=0.125, q=A, out=A, wsp=A, \
        wsb=ws: _st("tt_gqa_decode_attention", q, A, A, heads, kvh, d, cap, ln,
                    ctypes.c_float(scale), out, wsp, wsb, s)
    assert call(ln=0) == 2
    assert call(ln=4097) == 2                 # len beyond the cache
    assert call(heads=60) == 2                # heads not a multiple of kv_heads
    assert call(d=80) == 5                    # head_dim other than 64 / 128
    assert call(heads=136, kvh=8, wsb=1 << 30) == 5   # 17-wide groups
    assert call(heads=65, kvh=65, wsb=1 << 30) == 5   # more than 64 kv heads
    assert call(scale=float("inf")) == 4
    assert call(q=None) == 1
    assert call(wsp=None) == 1
    assert call(wsb=ws - 16) == 8
    assert call(q=A + 8) == 3
    assert call(out=A + 2) == 3
    assert call(wsp=A + 4) == 3


def test_lowbit_validation_before_launch(lib):
    A = 1 << 20  # never dereferenced: every case fails validation first
    s = None
    assert _st("tt_lowbit_matrix_bytes", 1, 5760, 2880) == 5760 * (368 + 32)
    assert _st("tt_lowbit_matrix_bytes", 2, 2880, 2880) == 2880 * (2 * 368 + 32)
    assert _st("tt_lowbit_matrix_bytes", 1, 3, 130) == 3 * (32 + 16)
    assert _st("tt_lowbit_matrix_bytes", 3, 8, 128) == 0
    q = lambda bits=1, n=8, k=128, w=A, buf=A, nb=1 << 20, st=None: _st(
        "tt_quantize_lowbit", bits, w, n, k, buf, nb, st, s)
    assert q(bits=4) == 2
    assert q(k=0) == 2
    assert q(n=0, w=None, buf=None) == 0   # empty: a no-op
    assert q(w=None) == 1
    assert q(nb=10) == 8
    assert q(buf=A + 8) == 3
    assert q(st=A + 2) == 3
    wsb = _st("tt_moe_lowbit_workspace_bytes", 2880, 32, 4)
    assert wsb == 4 * 2880 * 4 + 128
    call = lambda bits=1, H=2880, I=2880, E=32, K=4, x=A, tg=A, td=A, wsp=A, nb=wsb: _st(
        "tt_moe_lowbit_topk_mlp", bits, x, H, I, A, E, K, tg, td, A, A, A, wsp, nb, s)
    assert call(bits=3) == 2
    assert call(H=2890) == 2
    assert call(I=8224, nb=1 << 30) == 2
    assert call(K=9) == 2
    assert call(E=257) == 2
    assert call(x=None) == 1
    assert call(tg=None) == 1
    assert call(nb=wsb - 4) == 8
    assert call(x=A + 8) == 3
    assert call(td=A + 4) == 3
    assert call(wsp=A + 8) == 3
