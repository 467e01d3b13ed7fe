"""Single-token GQA decode attention on the GPU (tt_gqa_decode_attention)
against the fp64 oracle, element by element, on seeded synthetic caches:
the SmolLM3-3B and gpt-oss-20b head layouts, MHA / MQA / 16-wide groups,
contexts from one token to 32768 (tile and split edges, ragged tails), a
cache whose rows past len hold NaN, workspace reuse, graph capture with
programmatic dependent launch, and determinism."""
import math

import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity, bf16_to_f64

pytestmark = pytest.mark.gpu

WID = 140


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _workspace(heads, kvh, d):
    """Scratch with garbage in it: the call needs no initial contents."""
    import torch
    nb = thinmx.tt_gqa_decode_workspace_bytes(heads, kvh, d)
    assert nb > 0
    return torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda"), nb


def _run(q, k, v, length, scale, ws=None):
    import torch
    heads, d = q.shape
    kvh, cap, _ = k.shape
    if ws is None:
        ws = _workspace(heads, kvh, d)
    out = torch.empty((heads, d), dtype=torch.int16, device="cuda")
    thinmx.tt_gqa_decode_attention(gu.dev(q), gu.dev(k), gu.dev(v), heads, kvh, d, cap, length,
                                   scale, out, ws[0], ws[1])
    torch.cuda.synchronize()
    return gu.host(out, np.uint16)


def _check(q, k, v, length, scale, what, ws=None):
    got = _run(q, k, v, length, scale, ws)
    ref, st = oracle.gqa_decode(q, k, v, length, float(np.float32(scale)))
    assert st == 0
    assert_float_parity(got, ref, what)
    for h in range(q.shape[0]):  # every head on its own scale too
        assert_float_parity(got[h], ref[h], f"{what} head {h}")
    assert gu.device_error() == 0
    return got, ref


@pytest.mark.parametrize("heads,kvh,d,cap,length", [
    (16, 4, 128, 4096, 4096),   # SmolLM3-3B heads
    (64, 8, 64, 4096, 4096),    # gpt-oss-20b heads
    (16, 4, 128, 3000, 2999),
    (64, 8, 64, 1000, 777),
    (8, 8, 64, 100, 77),        # MHA (one query head per kv head)
    (12, 1, 64, 257, 257),      # MQA, 12-wide group (two head tiles)
    (32, 2, 128, 600, 517),     # 16-wide groups
    (40, 10, 128, 300, 300),    # Phi-4 heads
    (28, 4, 128, 500, 333),     # 7-wide groups
    (4, 4, 128, 64, 64),
    (64, 64, 128, 400, 399),    # the most kv heads (64), one query head each
    (1024, 64, 64, 130, 130),   # 64 kv heads with 16-wide groups
])
def test_gqa_shapes(heads, kvh, d, cap, length):
    c = synth.gqa_inputs(WID, heads * 1000 + length, heads, kvh, d, cap)
    _check(c["q"], c["k"], c["v"], length, 1.0 / math.sqrt(d), f"gqa {heads}/{kvh}/{d} len {length}")


@pytest.mark.parametrize("length", [1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 4095, 4097])
@pytest.mark.parametrize("heads,kvh,d", [(16, 4, 128), (64, 8, 64)])
def test_gqa_tile_edges(heads, kvh, d, length):
    """Tiles are 32 tokens (head_dim 128) or 64 (head_dim 64): lengths around
    their multiples, and around the split boundaries of a short context."""
    c = synth.gqa_inputs(WID, 50000 + length + d, heads, kvh, d, length + 3)
    _check(c["q"], c["k"], c["v"], length, 1.0 / math.sqrt(d), f"gqa d {d} len {length}")


@pytest.mark.parametrize("heads,kvh,d", [(16, 4, 128), (64, 8, 64)])
def test_gqa_long_context(heads, kvh, d):
    """32768 cached tokens: every split of the grid is busy and each CTA's
    warps run many tiles."""
    length = 32768
    c = synth.gqa_inputs(WID, 60000 + heads, heads, kvh, d, length)
    _check(c["q"], c["k"], c["v"], length, 1.0 / math.sqrt(d), f"gqa {heads}/{kvh}/{d} 32k")


def test_gqa_rows_past_len_are_never_read():
    heads, kvh, d, cap, length = 16, 4, 128, 200, 150
    c = synth.gqa_inputs(WID, 7, heads, kvh, d, cap)
    k, v = c["k"].copy(), c["v"].copy()
    k[:, length:] = 0x7FC0  # bf16 NaN
    v[:, length:] = 0x7FC0
    got, _ = _check(c["q"], k, v, length, 1.0 / math.sqrt(d), "gqa with NaN past len")
    assert np.array_equal(got, _run(c["q"], c["k"], c["v"], length, 1.0 / math.sqrt(d)))


def test_gqa_peaked_and_flat_attention():
    heads, kvh, d, cap = 64, 8, 64, 1500
    c = synth.gqa_inputs(WID, 8, heads, kvh, d, cap, k_std=4.0)
    # keys with a large spread and a big scale: weights span many decades
    _check(c["q"], c["k"], c["v"], cap, 0.5, "gqa peaked")
    # scale 0: every head returns the mean of its kv head's values
    got, ref = _check(c["q"], c["k"], c["v"], cap, 0.0, "gqa flat")
    mean = bf16_to_f64(c["v"]).mean(axis=1)  # [kv_heads][d]
    assert np.allclose(ref, np.repeat(mean, heads // kvh, axis=0), rtol=1e-12, atol=1e-14)


def test_gqa_dominant_token():
    heads, kvh, d, cap = 16, 4, 128, 700
    c = synth.gqa_inputs(WID, 9, heads, kvh, d, cap)
    k = synth.bf16_bits_to_f32(c["k"])
    q = synth.bf16_bits_to_f32(c["q"])
    t = 411
    for j in range(kvh):  # key t of every kv head aligned with its heads' queries, scaled up
        k[j, t] = 8.0 * q[j * 4:(j + 1) * 4].sum(axis=0)
    kb = synth.f32_to_bf16_bits(k)
    got, ref = _check(c["q"], kb, c["v"], cap, 1.0 / math.sqrt(d), "gqa dominant token")
    vt = bf16_to_f64(c["v"][:, t])
    assert np.allclose(ref, np.repeat(vt, 4, axis=0), atol=1e-6)


def test_gqa_workspace_is_reused_across_calls_and_shapes():
    import torch
    ws = _workspace(64, 8, 128)  # large enough for every call below
    cases = [(16, 4, 128, 900), (64, 8, 64, 3000), (16, 4, 128, 33), (8, 8, 64, 1)]
    for i, (heads, kvh, d, length) in enumerate(cases * 2):
        assert thinmx.tt_gqa_decode_workspace_bytes(heads, kvh, d) <= ws[1]
        c = synth.gqa_inputs(WID, 70000 + i, heads, kvh, d, length)
        _check(c["q"], c["k"], c["v"], length, 1.0 / math.sqrt(d), f"reuse {i}", ws=ws)
    torch.cuda.synchronize()


def test_gqa_is_deterministic():
    heads, kvh, d, length = 64, 8, 64, 20000
    c = synth.gqa_inputs(WID, 11, heads, kvh, d, length)
    a = _run(c["q"], c["k"], c["v"], length, 0.125)
    b = _run(c["q"], c["k"], c["v"], length, 0.125)
    assert np.array_equal(a, b)


def test_gqa_layers_in_one_graph():
    """Three layers' attention PDL-chained in one CUDA graph on one workspace,
    each reading the previous call's output as its query, replayed twice."""
    import torch
    heads, kvh, d, length = 16, 4, 128, 2500
    caches = [synth.gqa_inputs(WID, 80 + l, heads, kvh, d, length) for l in range(3)]
    q0 = gu.dev(caches[0]["q"])
    ks = [gu.dev(c["k"]) for c in caches]
    vs = [gu.dev(c["v"]) for c in caches]
    outs = [torch.empty((heads, d), dtype=torch.int16, device="cuda") for _ in range(3)]
    ws = _workspace(heads, kvh, d)
    scale = 1.0 / math.sqrt(d)

    def step():
        q = q0
        for l in range(3):
            thinmx.tt_gqa_decode_attention(q, ks[l], vs[l], heads, kvh, d, length, length, scale,
                                           outs[l], ws[0], ws[1])
            q = outs[l]

    step()
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert gu.device_error() == 0
    q = caches[0]["q"]
    for l in range(3):
        got = gu.host(outs[l], np.uint16)
        ref, _ = oracle.gqa_decode(q, caches[l]["k"], caches[l]["v"], length,
                                   float(np.float32(scale)))
        assert_float_parity(got, ref, f"graph layer {l}")
        q = got  # the next layer's query is this layer's output, as the GPU saw it


def test_gqa_rejects_bad_arguments_before_launch():
    import torch
    heads, kvh, d = 16, 4, 128
    ws = _workspace(heads, kvh, d)
    t = torch.zeros(64 * 1024, dtype=torch.int16, device="cuda")
    call = lambda **kw: thinmx.load().tt_gqa_decode_attention(
        kw.get("q", t.data_ptr()), t.data_ptr(), t.data_ptr(), kw.get("heads", heads),
        kw.get("kvh", kvh), kw.get("d", d), kw.get("cap", 64), kw.get("len", 64),
        kw.get("scale", 0.1), t.data_ptr(), ws[0].data_ptr(), kw.get("wsb", ws[1]), None)
    assert call(len=0) == 2
    assert call(len=65) == 2                      # beyond the cache
    assert call(heads=15) == 2                    # not a multiple of kv_heads
    assert call(d=96) == 5
    assert call(heads=68, kvh=4) == 5             # 17-wide groups
    assert call(scale=float("nan")) == 4
    assert call(wsb=ws[1] - 1) == 8
    assert call(q=t.data_ptr() + 2) == 3
    torch.cuda.synchronize()
    assert gu.device_error() == 0
