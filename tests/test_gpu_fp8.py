"""GPU parity of the FP8 (E4M3, one fp32 scale per row) quantiser, matvec
and gate/up SwiGLU matvec against the CPU oracle: codes and scales bit for
bit, float outputs at the tolerance of tests/parity.py."""
import os

import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _quantize(w_np):
    import torch
    n, k = w_np.shape
    codes = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
    scales = torch.zeros(n, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    thinmx.tt_quantize_fp8(gu.dev(w_np.astype(np.float32)), n, k, codes, scales, status)
    return codes, scales, status


def _check_quantize(w):
    codes, scales, status = _quantize(w)
    rc, rs, rst = oracle.fp8_quantize(w)
    got_s = gu.host(scales)
    assert np.array_equal(np.isnan(got_s), np.isnan(rs))
    ok = ~np.isnan(rs)
    assert np.array_equal(got_s[ok].view(np.uint32), rs[ok].view(np.uint32))
    assert np.array_equal(gu.host(codes), rc)
    assert int(gu.host(status)[0]) == rst
    return codes, scales


def test_quantize_random_and_special_rows():
    g = synth.rng(120)
    k = 200
    rows = [g.standard_normal(k) * 0.02, np.zeros(k), -np.zeros(k),
            g.standard_normal(k) * 1e-40,                   # amax / 448 underflows fp32
            g.standard_normal(k) * 1e30,
            np.ldexp(1.0, g.integers(-40, 40, k)) * g.choice([-1, 1], k),
            np.full(k, 3.4e38)]
    _check_quantize(np.array(rows, np.float32))


def test_quantize_nonfinite_rows_flag_status():
    g = synth.rng(121)
    w = (g.standard_normal((4, 64)) * 0.02).astype(np.float32)
    w[1, 5] = np.nan
    w[3, 63] = -np.inf
    codes, scales = _check_quantize(w)
    s = gu.host(scales)
    assert np.isnan(s[1]) and np.isnan(s[3]) and not np.isnan(s[0])


def test_quantize_rounds_the_hand_derived_ties():
    """A row whose max is 448 gets scale 1 exactly, so its other values are
    encoded as they stand: the hand-derived midpoints of the golden file."""
    vals, want = [448.0], [0x7E]
    for line in open(os.path.join(GOLD, "e4m3_rne_ties.txt")):
        line = line.split("#", 1)[0].split()
        if line and abs(float(line[0])) <= 448.0:
            vals.append(float(line[0]))
            want.append(int(line[1], 16))
    w = np.array([vals], np.float32)
    codes, scales = _check_quantize(w)
    assert float(gu.host(scales)[0]) == 1.0
    assert list(gu.host(codes)[0]) == want


def test_quantize_full_smollm3_gate_matrix():
    c = synth.GATE_UP
    d = synth.gate_up_inputs(c.wid, 0, c.n, c.k)
    _check_quantize(d["wg"])


def _fp8_case(n, k, m, wid=122, swiglu=True, x=None):
    import torch
    d = synth.gate_up_inputs(wid, 0, n, k, m=m)
    gc, gs, _ = _quantize(d["wg"])
    x = d["x"] if x is None else x
    if swiglu:
        uc, us, _ = _quantize(d["wu"])
        h = torch.empty((m, n), dtype=torch.int16, device="cuda")
        thinmx.tt_fp8_swiglu_matvec(gc, gs, uc, us, n, k, gu.dev(x), m, h)
        torch.cuda.synchronize()
        ref = oracle.fp8_swiglu_matvec((gu.host(gc), gu.host(gs)), (gu.host(uc), gu.host(us)), x)
    else:
        h = torch.empty((m, n), dtype=torch.int16, device="cuda")
        thinmx.tt_fp8_matvec(gc, gs, n, k, gu.dev(x), m, h)
        torch.cuda.synchronize()
        ref = oracle.fp8_matvec(gu.host(gc), gu.host(gs), x)
    return gu.host(h, np.uint16), ref


@pytest.mark.parametrize("n,k,m", [(1, 16, 1), (7, 48, 1), (129, 512, 1), (300, 2880, 1),
                                   (33, 5120, 1), (40, 2048, 2), (21, 1008, 3), (64, 1040, 5),
                                   (17, 4096, 8), (9, 16384, 1), (5, 8192, 4)])
@pytest.mark.parametrize("swiglu", [True, False])
def test_fp8_matvec_shapes(n, k, m, swiglu):
    h, ref = _fp8_case(n, k, m, swiglu=swiglu)
    assert h.shape == (m, n)
    for i in range(m):
        assert_float_parity(h[i], ref[i], f"fp8 n={n} k={k} m={m} row {i}")
    assert gu.device_error() == 0


def test_fp8_swiglu_full_smollm3_gate_up_layer():
    c = synth.GATE_UP
    h, ref = _fp8_case(c.n, c.k, 1, wid=c.wid)
    assert_float_parity(h, ref, "fp8 gate/up 11008x2048")


def test_fp8_down_projection_full_smollm3_shape():
    """The down projection of the same MLP: 11008 -> 2048."""
    h, ref = _fp8_case(2048, 11008, 1, wid=123, swiglu=False)
    assert_float_parity(h, ref, "fp8 down 2048x11008")


@pytest.mark.parametrize("n", [1, 5, 303, 3001])
def test_fp8_down_projection_k11008_row_counts(n):
    """K = 11008 at m = 1 (one row per CTA step): fewer rows than CTAs, about
    one per CTA, and rows beyond the rows in flight of every CTA."""
    h, ref = _fp8_case(n, 11008, 1, wid=125, swiglu=False)
    assert_float_parity(h, ref, f"fp8 down {n}x11008")
    assert gu.device_error() == 0


def test_fp8_large_and_outlier_activations():
    n, k, m = 64, 2048, 3
    d = synth.gate_up_inputs(124, 0, n, k, m=m)
    xf = synth.bf16_bits_to_f32(d["x"]).copy()
    xf[0] *= np.float32(2.0 ** 40)                       # beyond f16 altogether
    xf[1] *= np.float32(2.0 ** -40)                      # far below it
    xf[2, k - 3] = np.float32(1.0e4 * np.median(np.abs(xf[2])))  # one outlier
    x = synth.f32_to_bf16_bits(xf)
    for swiglu in (True, False):
        h, ref = _fp8_case(n, k, m, wid=124, swiglu=swiglu, x=x)
        for i in range(m):
            assert_float_parity(h[i], ref[i], f"fp8 row {i} swiglu={swiglu}")
        # the same rows one at a time (m = 1 has its own kernels at k = 2048)
        for i in range(m):
            h1, ref1 = _fp8_case(n, k, 1, wid=124, swiglu=swiglu, x=x[i:i + 1])
            assert_float_parity(h1[0], ref1[0], f"fp8 m=1 row {i} swiglu={swiglu}")
    assert gu.device_error() == 0


@pytest.mark.parametrize("n", [1, 7, 2433, 5000])
def test_fp8_gate_up_k2048_row_counts(n):
    """K = 2048 at m = 1 (a warp per row pair, two pairs in flight): a single
    row, a few, one more than one pass of the grid's warps, several passes."""
    h, ref = _fp8_case(n, 2048, 1, wid=126, swiglu=True)
    assert_float_parity(h, ref, f"fp8 gate/up {n}x2048")
    assert gu.device_error() == 0
