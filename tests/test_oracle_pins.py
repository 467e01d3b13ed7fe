"""Pins for the CPU oracle: each check ties the oracle to something other
than itself — hand-derived fixtures under tests/golden/, closed forms,
exhaustive tables, brute force over a whole 16-bit format, invariants of the
quantiser, and library routines (numpy matmul, scipy expit, numpy float16).

A plausible slip in the oracle (a dropped term, a wrong sign, a transposed
operand, a wrong rounding tie, a swapped gate/up) fails at least one test.
"""
import bisect
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle
from bit_weight_only_mxfp4_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


# ---------------------------------------------------------------- E2M1/E8M0
def test_e2m1_table_exhaustive():
    for code, val in _rows("e2m1_values.txt"):
        got = oracle.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e2m1_encode_roundtrip_all_codes():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_e2m1_rne_ties_and_saturation():
    for t, code in _rows("e2m1_rne_ties.txt"):
        assert oracle.e2m1_encode(float(t)) == int(code), t
    # just off every midpoint the nearest value wins
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    lo_code = [0, 1, 2, 3, 4, 5, 6]
    for mid, lo in zip(mids, lo_code):
        assert oracle.e2m1_encode(np.nextafter(mid, 0.0)) == lo
        assert oracle.e2m1_encode(np.nextafter(mid, 10.0)) == lo + 1
    for t in [6.0, 6.5, 7.0, 7.999999, 8.0, 100.0, 1e300]:
        assert oracle.e2m1_encode(t) == 7
        assert oracle.e2m1_encode(-t) == 15


def test_e8m0_closed_form():
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)


def test_floor_log2_at_powers_of_two_and_neighbours():
    # exponent read off the bits, not a rounded log2
    for e in range(-149, 128):
        a = np.float32(2.0 ** e)
        assert oracle.floor_log2(a) == e
        up = np.nextafter(a, np.float32(np.inf))
        if np.isfinite(up) and e > -149:  # 2^-149 + ulp is 2^-148
            assert oracle.floor_log2(up) == e
        if e > -149:
            dn = np.nextafter(a, np.float32(0))
            assert oracle.floor_log2(dn) == e - 1


# ------------------------------------------------------ 16-bit float formats
def _all_finite(fmt):
    """Every finite value of a 16-bit format as (Fraction, bits)."""
    bits = np.arange(65536, dtype=np.uint32)
    if fmt == "bf16":
        vals = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    else:
        vals = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    pairs = [(Fraction(float(v)), int(b)) for v, b in zip(vals, bits)
             if np.isfinite(v) and not (v == 0 and b & 0x8000)]
    pairs.sort()
    return pairs


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_16bit_round_brute_force(fmt):
    pairs = _all_finite(fmt)
    keys = [p[0] for p in pairs]
    top = pairs[-1][0]
    nxt_pow = Fraction(2) ** (128 if fmt == "bf16" else 16)
    overflow_at = (top + nxt_pow) / 2  # midpoint between max and 2^emax+1
    g = np.random.default_rng(7)
    probes = list(g.standard_normal(400) * 10.0 ** g.integers(-8, 8, 400))
    # exact midpoints between neighbours, and their float neighbours
    for i in g.integers(0, len(pairs) - 1, 300):
        mid = (keys[i] + keys[i + 1]) / 2
        m = float(mid)
        probes += [m, np.nextafter(m, -np.inf), np.nextafter(m, np.inf)]
    probes += [float(overflow_at), float(overflow_at) * (1 - 1e-12)]
    rnd = oracle.bf16_round if fmt == "bf16" else oracle.f16_round
    for v in probes:
        fv = Fraction(float(v))
        a = abs(fv)
        if a >= overflow_at:
            want = 0x7F80 if fmt == "bf16" else 0x7C00
        else:
            j = bisect.bisect_left(keys, a)
            cands = [pairs[c] for c in (j - 1, j) if 0 <= c < len(pairs)]
            cands.sort(key=lambda p: (abs(p[0] - a), p[1] & 1))
            want = cands[0][1]
        if v < 0 or (v == 0 and math.copysign(1, v) < 0):
            want |= 0x8000
        assert rnd(float(v)) == want, (fmt, v)


def test_f16_value_all_patterns_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_value(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.all(np.signbit(ref[~both_nan]) == np.signbit(got[~both_nan]))


def test_f16_round_vs_numpy_library():
    g = np.random.default_rng(3)
    v = g.standard_normal(5000) * 10.0 ** g.integers(-9, 6, 5000)
    want = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_round(float(t)) for t in v], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_value_closed_form():
    for b in [0x0000, 0x3F80, 0xBF80, 0x4000, 0x0001, 0x7F7F, 0x3E80]:
        want = np.array([b << 16], np.uint32).view(np.float32)[0]
        assert oracle.bf16_value(b) == float(want)


# -------------------------------------------------------------------- MXFP4
def test_mxfp4_worked_block():
    rows = _rows("mxfp4_worked_block.txt")
    scale = int(rows[0][1])
    vals = [r for r in rows[1:]]
    assert len(vals) == 32
    w = np.array([[float(r[0]) for r in vals]], np.float32)
    # t column is 16 w by construction
    for r in vals:
        assert float(r[1]) == 16.0 * float(r[0])
    codes, scales, st = oracle.mxfp4_quantize(w)
    assert st == oracle.OK
    assert scales[0, 0] == scale
    got = [(codes[0, i // 2] >> (4 * (i % 2))) & 15 for i in range(32)]
    assert got == [int(r[2]) for r in vals]


def _rand_w(g, n, k, std=0.02):
    return (g.standard_normal((n, k)) * std).astype(np.float32)


def test_mxfp4_power_of_two_invariance():
    g = np.random.default_rng(11)
    w = _rand_w(g, 23, 96)
    c0, s0, _ = oracle.mxfp4_quantize(w)
    for j in [-20, -7, -1, 1, 3, 20]:
        c1, s1, st = oracle.mxfp4_quantize((w * np.float32(2.0 ** j)).astype(np.float32))
        assert st == oracle.OK
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1.astype(int), s0.astype(int) + j)


def test_mxfp4_quantize_is_idempotent_on_its_grid():
    g = np.random.default_rng(12)
    n, k = 17, 128
    codes = synth.random_bytes(g, (n, k // 2))
    # every block holds at least one code of magnitude >= 4, so its amax
    # sits in the top binade and the scale is recovered exactly
    for r in range(n):
        for b in range(k // 32):
            codes[r, b * 16] = (codes[r, b * 16] & 0xF0) | 0x06 | (g.integers(0, 2) << 3)
    scales = g.integers(1, 250, size=(n, k // 32), dtype=np.uint8)
    deq = oracle.mxfp4_dequantize(codes, scales).astype(np.float32)
    c2, s2, st = oracle.mxfp4_quantize(deq)
    assert st == oracle.OK
    assert np.array_equal(s2, scales)
    # -0 and +0 dequantise to signed zeros, which requantise to 8 and 0
    assert np.array_equal(c2, codes)


def test_mxfp4_error_bound():
    g = np.random.default_rng(13)
    w = _rand_w(g, 31, 160)
    codes, scales, _ = oracle.mxfp4_quantize(w)
    deq = oracle.mxfp4_dequantize(codes, scales)
    X = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    t = np.abs(w.astype(np.float64)) / np.ldexp(1.0, X)
    half_gap = np.where(t <= 2, 0.25, np.where(t <= 4, 0.5, np.where(t <= 6, 1.0, 2.0)))
    assert np.all(np.abs(deq - w) <= half_gap * np.ldexp(1.0, X))
    # the block maximum always lands in [4, 8) before rounding
    amax = np.abs(w).reshape(31, 5, 32).max(axis=2)
    ratio = amax / np.ldexp(1.0, scales.astype(np.int64) - 127)
    assert np.all((ratio >= 4) & (ratio < 8))


def test_mxfp4_zero_and_nonfinite_blocks():
    w = np.zeros((2, 64), np.float32)
    w[0, 1] = -0.0
    w[1, 40] = np.nan
    w[1, 5] = 0.5
    codes, scales, st = oracle.mxfp4_quantize(w)
    assert st == oracle.ERR_NONFINITE
    assert scales[0, 0] == 0 and scales[0, 1] == 0
    assert codes[0, 0] == 0x80  # +0 (even k), -0 (odd k)
    assert scales[1, 1] == 0xFF and np.all(codes[1, 16:] == 0)
    assert scales[1, 0] == 124  # amax 0.5 -> X = -3
    assert (codes[1, 2] >> 4) == 6  # 0.5 / 2^-3 = 4 -> code 6


def test_mxfp4_identity_matrix():
    k = 64
    w = np.eye(k, dtype=np.float32)
    codes, scales, _ = oracle.mxfp4_quantize(w)
    assert np.array_equal(oracle.mxfp4_dequantize(codes, scales), np.eye(k))
    g = np.random.default_rng(5)
    x = synth.normal_bf16(g, (2, k))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    y = oracle.mxfp4_matvec(codes, scales, None, x)
    assert np.array_equal(y, xf)
    h = oracle.mxfp4_swiglu_matvec((codes, scales, None), (codes, scales, None), x)
    np.testing.assert_allclose(h, xf * expit(xf) * xf, rtol=1e-14, atol=0)


def test_mxfp4_matvec_equals_dense_dot_ragged():
    g = np.random.default_rng(14)
    n, k, m = 37, 96, 3
    w = _rand_w(g, n, k)
    codes, scales, _ = oracle.mxfp4_quantize(w)
    ps = synth.uniform_f32(g, (n,), 0.9, 1.1)
    x = synth.normal_bf16(g, (m, k))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    deq = oracle.mxfp4_dequantize(codes, scales)
    want = (xf @ deq.T) * ps.astype(np.float64)[None, :]
    got = oracle.mxfp4_matvec(codes, scales, ps, x)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
    # one-hot rows pick x at the right column (catches a transposed operand)
    oh = np.zeros((5, k), np.float32)
    cols = [0, 31, 32, 63, 95]
    for r, c in enumerate(cols):
        oh[r, c] = 1.0
    c1, s1, _ = oracle.mxfp4_quantize(oh)
    y1 = oracle.mxfp4_matvec(c1, s1, None, x)
    assert np.array_equal(y1, xf[:, cols])


def test_swiglu_against_expit_and_gate_up_order():
    g = np.random.default_rng(15)
    a = g.standard_normal(1000) * 4
    b = g.standard_normal(1000)
    np.testing.assert_allclose(oracle.swiglu(a, b), a * expit(a) * b, rtol=1e-14)
    # silu(g)*u is not symmetric in g and u
    assert not np.allclose(oracle.swiglu(a, b), oracle.swiglu(b, a))
    n, k = 19, 64
    wg, wu = _rand_w(g, n, k), _rand_w(g, n, k)
    cg, sg, _ = oracle.mxfp4_quantize(wg)
    cu, su, _ = oracle.mxfp4_quantize(wu)
    pg = synth.uniform_f32(g, (n,), 0.9, 1.1)
    pu = synth.uniform_f32(g, (n,), 0.9, 1.1)
    x = synth.normal_bf16(g, (1, k))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)[0]
    gv = oracle.mxfp4_dequantize(cg, sg) @ xf * pg
    uv = oracle.mxfp4_dequantize(cu, su) @ xf * pu
    h = oracle.mxfp4_swiglu_matvec((cg, sg, pg), (cu, su, pu), x)[0]
    np.testing.assert_allclose(h, gv * expit(gv) * uv, rtol=1e-12, atol=1e-18)


def test_bf16_swiglu_vs_numpy():
    g = np.random.default_rng(16)
    n, k = 13, 40
    wg = synth.normal_bf16(g, (n, k), 0.02)
    wu = synth.normal_bf16(g, (n, k), 0.02)
    x = synth.normal_bf16(g, (2, k))
    f = lambda a: synth.bf16_bits_to_f32(a).astype(np.float64)
    gv = f(x) @ f(wg).T
    uv = f(x) @ f(wu).T
    np.testing.assert_allclose(oracle.bf16_matvec(wg, x), gv, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(oracle.bf16_swiglu_matvec(wg, wu, x),
                               gv * expit(gv) * uv, rtol=1e-12, atol=1e-18)


# ---------------------------------------------------------------------- MoE
def test_topk_known_order_and_ties():
    lg = np.array([0.1, 0.5, 0.5, -1.0, 0.3, 0.5, 0.3], np.float32)
    assert list(oracle.topk(lg, 4)) == [1, 2, 5, 4]
    assert list(oracle.topk(lg, 7)) == [1, 2, 5, 4, 6, 0, 3]
    assert list(oracle.topk(np.zeros(8, np.float32), 3)) == [0, 1, 2]


def test_softmax_selected_closed_forms():
    lg = np.array([0.0, math.log(3.0), 7.0], np.float32)
    p = oracle.softmax_selected(lg, np.array([0, 1], np.int32))
    np.testing.assert_allclose(p, [1 / (1 + 3.0000001192), 3.0000001192 / (1 + 3.0000001192)], rtol=1e-7)
    p4 = oracle.softmax_selected(np.full(6, 2.5, np.float32), np.array([5, 1, 2, 0], np.int32))
    np.testing.assert_allclose(p4, [0.25] * 4, rtol=0, atol=1e-16)
    g = np.random.default_rng(17)
    lg = g.standard_normal(32).astype(np.float32)
    idx = oracle.topk(lg, 4)
    p = oracle.softmax_selected(lg, idx)
    assert abs(p.sum() - 1.0) < 1e-15
    assert np.all(np.diff(p) <= 0)


def test_moe_composite_vs_numpy():
    g = np.random.default_rng(18)
    E, H, I, K = 6, 64, 96, 3
    x = synth.normal_bf16(g, (H,))
    wr = synth.normal_bf16(g, (E, H), 0.02)
    gu = [_rand_w(g, 2 * I, H) for _ in range(E)]
    dn = [_rand_w(g, H, I) for _ in range(E)]
    q_gu = [oracle.mxfp4_quantize(a)[:2] for a in gu]
    q_dn = [oracle.mxfp4_quantize(a)[:2] for a in dn]
    gc = np.stack([q[0] for q in q_gu]); gs = np.stack([q[1] for q in q_gu])
    dc = np.stack([q[0] for q in q_dn]); ds = np.stack([q[1] for q in q_dn])
    out, idx, p, lg32, st = oracle.moe_mlp(x, wr, K, gc, gs, dc, ds)
    assert st == oracle.OK
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    logits = synth.bf16_bits_to_f32(wr).astype(np.float64) @ xf
    np.testing.assert_allclose(oracle.router_logits(x, wr), logits, rtol=1e-13)
    assert np.array_equal(lg32, logits.astype(np.float32))
    order = sorted(range(E), key=lambda e: (-float(lg32[e]), e))[:K]
    assert list(idx) == order
    sel = lg32[order].astype(np.float64)
    pw = np.exp(sel - sel.max()); pw /= pw.sum()
    np.testing.assert_allclose(p, pw, rtol=1e-14)
    want = np.zeros(H)
    for j, e in enumerate(order):
        dgu = oracle.mxfp4_dequantize(gc[e], gs[e])
        gv, uv = dgu[:I] @ xf, dgu[I:] @ xf
        hv = gv * expit(gv) * uv
        want += pw[j] * (oracle.mxfp4_dequantize(dc[e], ds[e]) @ hv)
    np.testing.assert_allclose(out, want, rtol=1e-11, atol=1e-15)


# --------------------------------------------------------------------- INT4
def test_int4_worked_groups():
    rows = _rows("int4_worked_groups.txt")
    meta = [r for r in rows if r[0].startswith("group_")]
    vals = [r for r in rows if not r[0].startswith("group_")]
    w = np.array([[float(r[0]) for r in vals]], np.float32)
    codes, scales, zp, st = oracle.int4_quantize(w, 8)
    assert st == oracle.OK
    for key, grp, val in meta:
        if key == "group_scale_bits":
            assert scales[0, int(grp)] == int(val)
        else:
            assert (zp[0, int(grp) // 2] >> (4 * (int(grp) % 2))) & 15 == int(val)
    q = [(codes[0, i // 2] >> (4 * (i % 2))) & 15 for i in range(12)]
    assert q == [int(r[1]) for r in vals]
    assert oracle.f16_value(10854) == 1.599609375 * 2.0 ** -5


def test_int4_error_bound_and_partial_group_stats():
    g = np.random.default_rng(19)
    n, k, G = 9, 2880, 128
    w = _rand_w(g, n, k)
    w[3, 2816:] *= 25.0  # the 64-wide last group has its own range
    codes, scales, zp, st = oracle.int4_quantize(w, G)
    assert st == oracle.OK and scales.shape == (n, 23) and zp.shape == (n, 12)
    assert np.all(zp[:, 11] >> 4 == 0)  # the unused high nibble stays 0
    deq = oracle.int4_dequantize(codes, scales, zp, G)
    s = np.repeat(np.array([[oracle.f16_value(int(b)) for b in row] for row in scales]), G, axis=1)[:, :k]
    assert np.all(np.abs(deq - w) <= s / 2 * (1 + 1e-12))
    last = w[3, 2816:]
    assert oracle.f16_value(int(scales[3, 22])) == pytest.approx((last.max() - last.min()) / 15, rel=1e-3)
    assert oracle.f16_value(int(scales[3, 21])) < oracle.f16_value(int(scales[3, 22])) / 5


def test_int4_degenerate_and_nonfinite_groups():
    w = np.zeros((1, 256), np.float32)
    w[0, :128] = 0.75          # constant group: s = 0, q = zp = 0
    w[0, 200] = np.inf
    codes, scales, zp, st = oracle.int4_quantize(w, 128)
    assert st == oracle.ERR_NONFINITE
    assert scales[0, 0] == 0 and (zp[0, 0] & 15) == 0 and np.all(codes[0, :64] == 0)
    assert scales[0, 1] == 0x7E00 and np.all(codes[0, 64:] == 0)


def test_int4_matvec_equals_dense_dot():
    g = np.random.default_rng(20)
    n, k, G = 21, 320, 128  # last group 64
    w = _rand_w(g, n, k)
    codes, scales, zp, _ = oracle.int4_quantize(w, G)
    x = synth.normal_bf16(g, (2, k))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    want = xf @ oracle.int4_dequantize(codes, scales, zp, G).T
    np.testing.assert_allclose(oracle.int4_matvec(codes, scales, zp, G, x), want,
                               rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- FP8 (E4M3)
# The next row of the hot path (a per-row-scaled FP8 matvec and SwiGLU).  The
# element format is pinned against torch's float8_e4m3fn (a library routine),
# the ties against hand-derived values, the quantiser by its invariants.

def _torch_e4m3():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    return torch


def test_e4m3_table_vs_torch_float8():
    torch = _torch_e4m3()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[c])
            continue
        assert v == ref[c] and math.copysign(1.0, v) == math.copysign(1.0, ref[c]), hex(c)
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_roundtrip_all_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_rne_ties_and_saturation():
    for t, code in _rows("e4m3_rne_ties.txt"):
        assert oracle.e4m3_encode(float(t)) == int(code, 16), t
    # just off every midpoint between neighbouring finite codes, the nearest wins
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2
        assert oracle.e4m3_encode(np.nextafter(mid, 0.0)) == c
        assert oracle.e4m3_encode(np.nextafter(mid, 1e9)) == c + 1
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even


def test_e4m3_encode_vs_torch_float8():
    torch = _torch_e4m3()
    g = np.random.default_rng(7)
    mag = np.exp2(g.uniform(-12.0, math.log2(448.0), 20000))
    v = (mag * g.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    mids = np.array([(vals[c] + vals[c + 1]) / 2 for c in range(0x7E)], np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(t)) for t in v], np.uint8)
    assert np.array_equal(got, ref)


def _fp8_rows(seed, n, k):
    return synth.normal_f32(synth.rng(seed), (n, k), 0.02)


def test_fp8_quantize_power_of_two_invariance():
    w = _fp8_rows(110, 24, 160)
    c0, s0, st = oracle.fp8_quantize(w)
    assert st == oracle.OK
    for j in (-20, -3, 5, 20):
        c1, s1, _ = oracle.fp8_quantize(w * np.float32(2.0 ** j))
        assert np.array_equal(c1, c0)
        assert np.array_equal(s1, s0 * np.float32(2.0 ** j))


def test_fp8_quantize_is_idempotent_on_its_grid():
    # rows of E4M3 values times 2^j, each holding a +-448: the scale is 2^j,
    # every weight is exact in fp32, and quantising gives the codes back
    g = np.random.default_rng(11)
    n, k = 16, 96
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    codes = g.choice(finite, (n, k)).astype(np.uint8)
    codes[np.arange(n), g.integers(0, k, n)] = g.choice([0x7E, 0xFE], n)
    j = g.integers(-30, 30, n)
    vals = np.vectorize(oracle.e4m3_value)(codes)
    w = (vals * np.exp2(j)[:, None]).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), vals * np.exp2(j)[:, None])
    c1, s1, st = oracle.fp8_quantize(w)
    assert st == oracle.OK
    assert np.array_equal(s1, np.exp2(j).astype(np.float32))
    assert np.array_equal(c1, codes)


def test_fp8_quantize_error_bound():
    w = _fp8_rows(111, 32, 200)
    w[3, :100] *= np.float32(1e-4)  # small values in a row with a normal max
    codes, scales, _ = oracle.fp8_quantize(w)
    deq = oracle.fp8_dequantize(codes, scales)
    s = scales.astype(np.float64)[:, None]
    t = np.abs(w.astype(np.float64)) / s
    # half the E4M3 spacing at |t|: 2^(floor(log2 t) - 3) / 2 in the normal
    # range, 2^-9 / 2 below 2^-6
    e = np.floor(np.log2(np.maximum(t, 2.0 ** -6)))
    half = np.exp2(e - 3) / 2
    assert np.all(np.abs(w - deq) <= half * s * (1 + 1e-12))
    # the row maximum maps to 448 exactly
    amax = np.abs(w).max(axis=1)
    assert np.allclose(np.abs(deq).max(axis=1), amax, rtol=2.0 ** -4)
    assert np.all(np.isin(codes[np.arange(32), np.abs(w).argmax(axis=1)], [0x7E, 0xFE]))


def test_fp8_zero_and_nonfinite_rows():
    w = _fp8_rows(112, 4, 64)
    w[1] = 0.0
    w[2, 5] = np.nan
    codes, scales, st = oracle.fp8_quantize(w)
    assert st == oracle.ERR_NONFINITE
    assert scales[1] == 0.0 and not codes[1].any()
    assert np.isnan(scales[2]) and not codes[2].any()
    ref, rs, _ = oracle.fp8_quantize(w[[0, 3]])
    assert np.array_equal(codes[[0, 3]], ref) and np.array_equal(scales[[0, 3]], rs)


def test_fp8_matvec_brute_force():
    # integer weights (E4M3 holds 0..16 exactly) and integer x: the sums
    # are exact, here checked with Python integers
    g = np.random.default_rng(13)
    n, k, m = 7, 40, 3
    iw = g.integers(-16, 17, (n, k))
    codes = np.array([[oracle.e4m3_encode(float(v)) for v in row] for row in iw], np.uint8)
    scales = np.exp2(g.integers(-4, 5, n)).astype(np.float32)
    ix = g.integers(-50, 51, (m, k))
    x = synth.f32_to_bf16_bits(ix.astype(np.float32))
    y = oracle.fp8_matvec(codes, scales, x)
    for i in range(m):
        for r in range(n):
            exact = Fraction(int(np.dot(iw[r], ix[i]))) * Fraction(float(scales[r]))
            assert y[i, r] == float(exact)


def test_fp8_swiglu_against_expit_and_gate_up_order():
    wg = _fp8_rows(114, 20, 96)
    wu = _fp8_rows(115, 20, 96) * np.float32(3.0)
    gc, gs, _ = oracle.fp8_quantize(wg)
    uc, us, _ = oracle.fp8_quantize(wu)
    x = synth.normal_bf16(synth.rng(116), (2, 96))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    g = xf @ oracle.fp8_dequantize(gc, gs).T
    u = xf @ oracle.fp8_dequantize(uc, us).T
    h = oracle.fp8_swiglu_matvec((gc, gs), (uc, us), x)
    np.testing.assert_allclose(h, g * expit(g) * u, rtol=1e-12, atol=1e-300)
    swapped = oracle.fp8_swiglu_matvec((uc, us), (gc, gs), x)
    assert not np.allclose(h, swapped)


# ---- single-token GQA attention ----------------------------------------------
def _gqa_inputs(seed, heads, kvh, d, cap, std=1.0):
    g = np.random.default_rng(seed)
    q = synth.normal_bf16(g, (heads, d), std)
    k = synth.normal_bf16(g, (kvh, cap, d), std)
    v = synth.normal_bf16(g, (kvh, cap, d), 1.0)
    return q, k, v


def _f(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_gqa_single_token_returns_its_value_row():
    q, k, v = _gqa_inputs(1, 8, 2, 16, 5)
    o, st = oracle.gqa_decode(q, k, v, 1, 0.25)
    assert st == oracle.OK
    want = np.repeat(_f(v[:, 0, :]), 4, axis=0)  # heads 0-3 -> kv 0, 4-7 -> kv 1
    assert np.array_equal(o, want)


def test_gqa_zero_scale_gives_the_mean_of_values():
    q, k, v = _gqa_inputs(2, 4, 4, 8, 37)
    o, _ = oracle.gqa_decode(q, k, v, 29, 0.0)
    assert np.allclose(o, _f(v[:, :29, :]).mean(axis=1), rtol=0, atol=1e-15)


def test_gqa_head_mapping_is_the_group_of_consecutive_heads():
    """kv head j serves query heads j*G .. j*G+G-1 (G = heads / kv_heads):
    with v of kv head j constant j + 1, output head h is h // G + 1."""
    heads, kvh, d, cap = 12, 3, 8, 6
    q, k, _ = _gqa_inputs(3, heads, kvh, d, cap)
    v = np.stack([np.full((cap, d), float(j + 1), np.float32) for j in range(kvh)])
    o, _ = oracle.gqa_decode(q, k, synth.f32_to_bf16_bits(v), cap, 0.5)
    # (sum_t p_t c) / (sum_t p_t) is c up to fp64 rounding; a wrong mapping is off by >= 1
    assert np.allclose(o[:, 0], np.array([h // 4 + 1 for h in range(heads)], np.float64),
                       rtol=0, atol=1e-12)


def test_gqa_equals_multi_head_attention_on_repeated_kv():
    heads, kvh, d, cap, n = 8, 2, 16, 20, 17
    q, k, v = _gqa_inputs(4, heads, kvh, d, cap)
    o, _ = oracle.gqa_decode(q, k, v, n, 0.25)
    o_mha, _ = oracle.gqa_decode(q, np.repeat(k, 4, axis=0), np.repeat(v, 4, axis=0), n, 0.25)
    assert np.array_equal(o, o_mha)


def test_gqa_matches_scipy_softmax_on_tiny_cases():
    from scipy.special import softmax
    for seed, (heads, kvh, d, cap, n) in enumerate([(4, 1, 8, 9, 9), (6, 3, 16, 12, 7),
                                                    (2, 2, 32, 40, 33)]):
        q, k, v = _gqa_inputs(10 + seed, heads, kvh, d, cap)
        scale = 1.0 / np.sqrt(d)
        o, _ = oracle.gqa_decode(q, k, v, n, scale)
        G = heads // kvh
        for h in range(heads):
            kk, vv = _f(k[h // G, :n]), _f(v[h // G, :n])
            p = softmax(kk @ _f(q[h]) * scale)
            assert np.allclose(o[h], p @ vv, rtol=1e-13, atol=1e-14)


def test_gqa_token_order_and_tokens_past_len_do_not_matter():
    heads, kvh, d, cap, n = 4, 2, 8, 16, 11
    q, k, v = _gqa_inputs(5, heads, kvh, d, cap)
    o, _ = oracle.gqa_decode(q, k, v, n, 0.3)
    perm = np.random.default_rng(5).permutation(n)
    k2, v2 = k.copy(), v.copy()
    k2[:, :n], v2[:, :n] = k[:, perm], v[:, perm]
    k2[:, n:] = v2[:, n:] = 0x7FC0  # bf16 NaN beyond len
    o2, _ = oracle.gqa_decode(q, k2, v2, n, 0.3)
    assert np.allclose(o, o2, rtol=1e-14, atol=1e-15)


def test_gqa_dominant_token_takes_all_the_weight():
    heads, kvh, d, cap = 2, 1, 4, 6
    q = synth.f32_to_bf16_bits(np.ones((heads, d), np.float32))
    k = np.zeros((kvh, cap, d), np.float32)
    k[0, 3] = 256.0  # score 1024 * scale above every other token's 0
    v = np.random.default_rng(6).standard_normal((kvh, cap, d)).astype(np.float32)
    o, _ = oracle.gqa_decode(q, synth.f32_to_bf16_bits(k), synth.f32_to_bf16_bits(v), cap, 1.0)
    assert np.array_equal(o, np.repeat(_f(synth.f32_to_bf16_bits(v))[:, 3], heads, axis=0))


def test_gqa_shape_errors():
    q, k, v = _gqa_inputs(7, 6, 4, 8, 4)  # 6 heads over 4 kv heads: not a group
    assert oracle.gqa_decode(q, k, v, 4, 1.0)[1] == oracle.ERR_SHAPE
    q, k, v = _gqa_inputs(7, 4, 2, 8, 4)
    assert oracle.gqa_decode(q, k, v, 5, 1.0)[1] == oracle.ERR_SHAPE  # len beyond the cache


# ---- Q1 / Q2 packed low-bit experts -----------------------------------------
def _lowbit_plane_bits(buf, bits, n, k, p, r):
    P = oracle.lowbit_plane_bytes(k)
    row = buf[p * n * P + r * P: p * n * P + (r + 1) * P]
    return np.unpackbits(row, bitorder="little")[:k]


def _lowbit_scale(buf, bits, n, k, r, b):
    P, S = oracle.lowbit_plane_bytes(k), oracle.lowbit_scale_bytes(k)
    return int(buf[bits * n * P + r * S + b])


def test_lowbit_worked_blocks():
    for row in (" ".join(r) for r in _rows("lowbit_worked_blocks.txt")):
        case, sb, q1b, q1v, q2b, q2v = [part.split() for part in row.split("|")]
        w = np.array([[float(v) for v in case[1:]]], np.float32)
        k = w.shape[1]
        for bits, planes, vals in ((1, q1b, q1v), (2, q2b, q2v)):
            buf, st = oracle.lowbit_quantize(bits, w)
            assert st == oracle.OK
            P = oracle.lowbit_plane_bytes(k)
            assert _lowbit_scale(buf, bits, 1, k, 0, 0) == int(sb[0]), case[0]
            for p, byte in enumerate(planes):
                assert buf[p * P] == int(byte), (case[0], bits, p)
            deq = oracle.lowbit_dequantize(bits, buf, 1, k)
            assert np.array_equal(deq[0], np.array([float(v) for v in vals])), (case[0], bits)


@pytest.mark.parametrize("bits", [1, 2])
def test_lowbit_layout_and_padding(bits):
    n, k = 3, 130  # a full block of 128 and a partial block of 2
    P, S = oracle.lowbit_plane_bytes(k), oracle.lowbit_scale_bytes(k)
    assert (P, S) == (32, 16)
    assert oracle.lowbit_matrix_bytes(bits, n, k) == n * (bits * 32 + 16)
    w = np.random.default_rng(40).standard_normal((n, k)).astype(np.float32)
    buf, st = oracle.lowbit_quantize(bits, w)
    assert st == oracle.OK
    for p in range(bits):
        for r in range(n):
            row = buf[p * n * P + r * P: p * n * P + (r + 1) * P]
            assert row[16] >> 2 == 0 and not row[17:].any()  # bits past k = 130
    sc = buf[bits * n * P:].reshape(n, S)
    assert not sc[:, 2:].any() and sc[:, :2].all()
    # codes as documented: Q1 = sign bit, Q2 = the two planes' bits
    signs = _lowbit_plane_bits(buf, bits, n, k, 0, 1)
    if bits == 1:
        assert np.array_equal(signs, (w[1] < 0).astype(np.uint8))


def test_lowbit_q1_step_is_the_l2_best_power_of_two():
    g = np.random.default_rng(41)
    n, k = 40, 128 * 3
    w = (g.standard_normal((n, k)) * np.exp(g.uniform(-6, 6, (n, 1)))).astype(np.float32)
    w[0, :128] = g.uniform(0.0, 1.0, 128).astype(np.float32)   # one-signed block
    w[1, :128] = np.float32(0.75)                              # the tie: mean on 1.5 * 2^-1
    buf, st = oracle.lowbit_quantize(1, w)
    assert st == oracle.OK
    deq = oracle.lowbit_dequantize(1, buf, n, k)
    for r in range(n):
        for b in range(3):
            blk = w[r, 128 * b:128 * (b + 1)].astype(np.float64)
            x = _lowbit_scale(buf, 1, n, k, r, b) - 127
            err = lambda e: float(np.sum((np.abs(blk) - 2.0 ** e) ** 2))
            assert np.array_equal(np.abs(deq[r, 128 * b:128 * (b + 1)]), np.full(128, 2.0 ** x))
            for d in (-2, -1, 1, 2):
                assert err(x) <= err(x + d), (r, b, d)
                if d == -1:
                    assert err(x) < err(x - 1), (r, b)  # ties go to the lower step
    assert _lowbit_scale(buf, 1, n, k, 1, 0) == 126


def test_lowbit_q2_codes_are_the_nearest_level():
    g = np.random.default_rng(42)
    n, k = 30, 256
    # values on a 2^-12 grid, so the block means need no rounding in any order
    w = (np.round(g.standard_normal((n, k)) * 4096 * np.exp(g.uniform(-2, 2, (n, 1))))
         / 4096).astype(np.float32)
    buf, st = oracle.lowbit_quantize(2, w)
    assert st == oracle.OK
    deq = oracle.lowbit_dequantize(2, buf, n, k)
    levels = np.array([-1.5, -0.5, 0.5, 1.5])
    for r in range(n):
        for b in range(2):
            blk = w[r, 128 * b:128 * (b + 1)].astype(np.float64)
            t = 2.0 ** (_lowbit_scale(buf, 2, n, k, r, b) - 127)
            m = np.abs(blk).mean()
            # the step is the power of two nearest the mean |w| (ties to the lower)
            assert abs(t - m) <= abs(2 * t - m) and abs(t - m) < abs(t / 2 - m)
            d = np.abs(blk[:, None] - levels[None, :] * t)
            best = d.min(axis=1)
            # nearest level; on a tie the upper of the two
            choice = np.array([np.flatnonzero(dd == bb).max() for dd, bb in zip(d, best)])
            assert np.array_equal(deq[r, 128 * b:128 * (b + 1)], levels[choice] * t)


@pytest.mark.parametrize("bits", [1, 2])
def test_lowbit_power_of_two_invariance_and_sign(bits):
    g = np.random.default_rng(43 + bits)
    n, k = 7, 300
    w = g.standard_normal((n, k)).astype(np.float32)
    buf, _ = oracle.lowbit_quantize(bits, w)
    P = oracle.lowbit_plane_bytes(k)
    for s in (-9, 5):
        buf2, _ = oracle.lowbit_quantize(bits, w * np.float32(2.0 ** s))
        assert np.array_equal(buf2[:bits * n * P], buf[:bits * n * P])
        sc, sc2 = buf[bits * n * P:].reshape(n, -1)[:, :3], buf2[bits * n * P:].reshape(n, -1)[:, :3]
        assert np.array_equal(sc2.astype(int), sc.astype(int) + s)
    if bits == 1:  # negating the weights flips every sign code, keeps the steps
        bufn, _ = oracle.lowbit_quantize(1, -w)
        assert np.array_equal(bufn[:n * P].reshape(n, P)[:, :k // 8],
                              (~buf[:n * P]).reshape(n, P)[:, :k // 8])
        assert np.array_equal(bufn[n * P:], buf[n * P:])


@pytest.mark.parametrize("bits", [1, 2])
def test_lowbit_nonfinite_block(bits):
    w = np.ones((2, 384), np.float32)
    w[1, 200] = np.nan
    buf, st = oracle.lowbit_quantize(bits, w)
    assert st == oracle.ERR_NONFINITE
    n, k = w.shape
    assert [_lowbit_scale(buf, bits, n, k, 1, b) for b in range(3)] == [127, 0xFF, 127]
    for p in range(bits):
        assert not _lowbit_plane_bits(buf, bits, n, k, p, 1)[128:256].any()
    assert np.isnan(oracle.lowbit_dequantize(bits, buf, n, k)[1, 128:256]).all()


@pytest.mark.parametrize("bits", [1, 2])
def test_moe_lowbit_layer_is_the_composition(bits):
    """Router -> top-k -> softmax -> SwiGLU of the selected experts -> the
    weighted down projections, checked against numpy / scipy on the
    dequantised matrices."""
    from scipy.special import expit, softmax
    g = np.random.default_rng(50 + bits)
    H, I, E, K = 64, 96, 6, 2
    x = synth.f32_to_bf16_bits(g.standard_normal(H).astype(np.float32))
    wr = synth.f32_to_bf16_bits((g.standard_normal((E, H)) * 0.3).astype(np.float32))
    gus, dns = [], []
    for e in range(E):
        gu, _ = oracle.lowbit_quantize(bits, g.standard_normal((2 * I, H)).astype(np.float32) * 0.05)
        dn, _ = oracle.lowbit_quantize(bits, g.standard_normal((H, I)).astype(np.float32) * 0.05)
        gus.append(gu)
        dns.append(dn)
    out, idx, p, lg, h, st = oracle.moe_lowbit_mlp(bits, x, wr, K, np.stack(gus), np.stack(dns), I)
    assert st == oracle.OK
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    logits = synth.bf16_bits_to_f32(wr).astype(np.float64) @ xv
    assert np.array_equal(lg, logits.astype(np.float32))
    order = np.lexsort((np.arange(E), -lg.astype(np.float64)))  # descending, lower index first
    assert np.array_equal(idx, order[:K])
    assert np.allclose(p, softmax(lg[idx].astype(np.float64)), rtol=1e-14)
    ref = np.zeros(H)
    for j, e in enumerate(idx):
        gu = oracle.lowbit_dequantize(bits, gus[e], 2 * I, H)
        dn = oracle.lowbit_dequantize(bits, dns[e], H, I)
        gg, uu = gu[:I] @ xv, gu[I:] @ xv
        hj = gg * expit(gg) * uu
        assert np.allclose(h[j], hj, rtol=1e-12, atol=1e-15)
        ref += p[j] * (dn @ hj)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
