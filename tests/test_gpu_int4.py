"""GPU parity of the grouped affine INT4 quantiser (bit-exact codes, fp16
scales and zero points) and matvec (float tolerance of tests/parity.py)
against the CPU oracle."""
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


def gpu_int4_quantize(w, group):
    import torch
    n, k = w.shape
    ng = (k + group - 1) // group
    wd = gu.dev(np.ascontiguousarray(w, np.float32))
    codes = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n, ng), dtype=torch.int16, device="cuda")
    zp = torch.zeros((n, (ng + 1) // 2), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    thinmx.tt_quantize_int4_grouped(wd, n, k, group, codes, scales, zp, status)
    torch.cuda.synchronize()
    return codes, scales, zp, int(gu.host(status)[0])


def gpu_int4_matvec(codes, scales, zp, n, k, group, x):
    import torch
    m = x.shape[0]
    y = torch.empty((m, n), dtype=torch.int16, device="cuda")
    thinmx.tt_int4_grouped_matvec(codes, scales, zp, n, k, group, gu.dev(x), m, y)
    torch.cuda.synchronize()
    return gu.host(y, np.uint16)


def _check_quantize(w, group):
    codes, scales, zp, st = gpu_int4_quantize(w, group)
    rc, rs, rz, rst = oracle.int4_quantize(w, group)
    assert np.array_equal(gu.host(scales, np.uint16), rs)
    assert np.array_equal(gu.host(zp), rz)
    assert np.array_equal(gu.host(codes), rc)
    assert st == rst
    return codes, scales, zp


def test_int4_quantize_worked_groups():
    rows = []
    for line in open(os.path.join(GOLD, "int4_worked_groups.txt")):
        line = line.split("#", 1)[0].split()
        if line and not line[0].startswith("group_"):
            rows.append(line)
    w = np.array([[float(r[0]) for r in rows]], np.float32)
    codes, scales, zp = _check_quantize(w, 8)
    c = gu.host(codes)[0]
    assert [(c[i // 2] >> (4 * (i % 2))) & 15 for i in range(12)] == [int(r[1]) for r in rows]
    assert list(gu.host(scales, np.uint16)[0]) == [10854, 10854]


def test_int4_quantize_random_partial_groups():
    g = synth.rng(96)
    w = synth.normal_f32(g, (37, 2880), 0.02)
    w[5, 2816:] *= 30.0
    _check_quantize(w, 128)
    _check_quantize(synth.normal_f32(g, (9, 200), 1.0), 64)  # 200 = 3*64 + 8


def test_int4_quantize_special_groups():
    w = np.zeros((4, 256), np.float32)
    w[0, :128] = 0.75            # constant group -> s = 0
    w[0, 128:] = 1e-9            # range below fp16 resolution -> s = 0
    w[1, 3] = np.nan
    w[2, 130] = np.inf
    w[3, :128] = np.linspace(-1e6, 1e6, 128)  # (max-min)/15 overflows fp16
    w[3, 128:] = np.linspace(-3, 5, 128)
    _check_quantize(w, 128)


def test_int4_quantize_full_qkv():
    c = synth.QKV
    d = synth.int4_inputs(c.wid, 0, c.n, c.k)
    _check_quantize(d["w"], c.group)


@pytest.mark.parametrize("n,k,group,m", [
    (37, 2880, 128, 1), (64, 256, 64, 2), (100, 1024, 32, 3), (17, 8192, 128, 8),
    (50, 2880, 96, 4), (300, 4096, 256, 1), (5, 32, 32, 1),
    # more rows than one pass of the grid covers (three rows per warp at m = 1)
    (9001, 256, 64, 1), (9001, 256, 64, 3),
    # m = 1, group 128: the tensor-core row-pair kernel (k in 1..4 steps of 1024,
    # partial last group, odd row counts, several pairs per warp)
    (1, 128, 128, 1), (2, 1024, 128, 1), (33, 1056, 128, 1), (40, 2048, 128, 1),
    (31, 3008, 128, 1), (64, 4096, 128, 1), (9001, 2880, 128, 1), (12, 4128, 128, 1),
])
def test_int4_matvec_shapes(n, k, group, m):
    d = synth.int4_inputs(97, 0, n, k, m)
    codes, scales, zp = _check_quantize(d["w"], group)
    y = gpu_int4_matvec(codes, scales, zp, n, k, group, d["x"])
    ref = oracle.int4_matvec(gu.host(codes), gu.host(scales, np.uint16), gu.host(zp), group,
                             d["x"])
    assert_float_parity(y, ref, f"int4 n={n} k={k} G={group} m={m}")
    assert gu.device_error() == 0


def test_int4_matvec_full_qkv():
    c = synth.QKV
    d = synth.int4_inputs(c.wid, 0, c.n, c.k, c.m)
    codes, scales, zp = _check_quantize(d["w"], c.group)
    y = gpu_int4_matvec(codes, scales, zp, c.n, c.k, c.group, d["x"])
    y2 = gpu_int4_matvec(codes, scales, zp, c.n, c.k, c.group, d["x"])
    assert np.array_equal(y, y2)
    ref = oracle.int4_matvec(gu.host(codes), gu.host(scales, np.uint16), gu.host(zp), c.group,
                             d["x"])
    assert_float_parity(y, ref, "int4 qkv 5120x2880")
    assert np.mean(y.ravel() == oracle.bf16_round_array(ref.ravel())) > 0.99


def test_int4_matvec_chunks_of_very_different_magnitude():
    """x is prescaled per 32-chunk by its own power of two: chunks spread over
    2^-60 .. 2^60 (and an all-zero chunk).  The weights of each chunk are
    scaled the other way as far as fp16 group scales allow (2^-10 .. 2^6), so
    that many chunks contribute to the result."""
    n, k, group = 64, 1024, 32
    d = synth.int4_inputs(98, 0, n, k, 1)
    g = synth.rng(98, 1)
    e = g.integers(-60, 61, k // 32)
    fx = np.repeat(np.ldexp(1.0, e), 32)
    fw = np.repeat(np.ldexp(1.0, -np.clip(e, -6, 10)), 32)
    xf = (synth.bf16_bits_to_f32(d["x"]).astype(np.float64) * fx).astype(np.float32)
    xf[:, 64:96] = 0.0
    x = synth.f32_to_bf16_bits(xf)
    w = (d["w"].astype(np.float64) * fw).astype(np.float32)
    codes, scales, zp = _check_quantize(w, group)
    y = gpu_int4_matvec(codes, scales, zp, n, k, group, x)
    ref = oracle.int4_matvec(gu.host(codes), gu.host(scales, np.uint16), gu.host(zp), group, x)
    assert_float_parity(y, ref, "int4 chunk magnitudes 2^-60..2^60")
    assert gu.device_error() == 0


def test_int4_matvec_groups_of_very_different_magnitude():
    """The m = 1, group-128 tensor-core kernel prescales x per 128-group:
    groups spread over 2^-60 .. 2^60 (and an all-zero group), weights scaled
    the other way as far as fp16 group scales allow."""
    n, k, group = 64, 2880, 128
    d = synth.int4_inputs(99, 0, n, k, 1)
    g = synth.rng(99, 1)
    ng = (k + group - 1) // group
    e = g.integers(-60, 61, ng)
    fx = np.repeat(np.ldexp(1.0, e), group)[:k]
    fw = np.repeat(np.ldexp(1.0, -np.clip(e, -6, 10)), group)[:k]
    xf = (synth.bf16_bits_to_f32(d["x"]).astype(np.float64) * fx).astype(np.float32)
    xf[:, 256:384] = 0.0
    x = synth.f32_to_bf16_bits(xf)
    w = (d["w"].astype(np.float64) * fw).astype(np.float32)
    codes, scales, zp = _check_quantize(w, group)
    y = gpu_int4_matvec(codes, scales, zp, n, k, group, x)
    ref = oracle.int4_matvec(gu.host(codes), gu.host(scales, np.uint16), gu.host(zp), group, x)
    assert_float_parity(y, ref, "int4 group magnitudes 2^-60..2^60")
    assert gu.device_error() == 0

