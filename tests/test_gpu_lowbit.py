"""Q1 / Q2 packed low-bit experts on the GPU against the fp64 oracle: the
quantiser bit for bit (partial blocks, ties, zero and non-finite blocks),
and the MoE layer with low-bit experts (router, selected-expert SwiGLU,
weighted down projection) element by element, on buffers the oracle
quantised, each expert in an allocation of its own; the gpt-oss-20b
shape (hidden = inter = 2880, 32 experts, top-4), a PDL-chained graph of
layers, determinism and a bad expert pointer."""
import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import loader, synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity

pytestmark = pytest.mark.gpu

WID = 150


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _gpu_quantize(bits, w):
    import torch
    n, k = w.shape
    nb = thinmx.tt_lowbit_matrix_bytes(bits, n, k)
    assert nb == oracle.lowbit_matrix_bytes(bits, n, k)
    buf = torch.full((nb,), 0xA5, dtype=torch.uint8, device="cuda")  # garbage to overwrite
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    thinmx.tt_quantize_lowbit(bits, gu.dev(w.astype(np.float32)), n, k, buf, nb, status)
    torch.cuda.synchronize()
    return gu.host(buf), int(status.item())


@pytest.mark.parametrize("bits", [1, 2])
@pytest.mark.parametrize("n,k", [(1, 1), (3, 127), (5, 128), (4, 129), (7, 300), (64, 2880),
                                 (33, 8192), (5760, 2880)])
def test_quantize_lowbit_bit_exact(bits, n, k):
    g = synth.rng(WID, n, k)
    w = (g.standard_normal((n, k)) * np.exp(g.uniform(-8, 8, (n, 1)))).astype(np.float32)
    got, st = _gpu_quantize(bits, w)
    ref, st_ref = oracle.lowbit_quantize(bits, w)
    assert st == st_ref == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("bits", [1, 2])
def test_quantize_lowbit_special_blocks(bits):
    g = synth.rng(WID, 1)
    n, k = 8, 2880
    w = (g.standard_normal((n, k)) * 0.02).astype(np.float32)
    w[0, :128] = 0.0                                   # zero block
    w[1, 128:256] = np.float32(0.75)                   # mean on a tie (1.5 * 2^-1)
    w[1, 256:384] = np.float32(-0.75)
    w[2, 2816:] = np.float32(3.0) * np.sign(w[2, 2816:])  # the 64-wide last block
    w[3, 5] = np.nan                                   # non-finite blocks
    w[4, 2900 - 30] = np.inf
    w[5, :] = np.float32(2.0 ** -140)                  # subnormal weights: X clamps at -127
    w[6, :] = np.float32(2.0 ** 120) * np.sign(w[6, :])
    w[7, 1::2] = -0.0
    got, st = _gpu_quantize(bits, w)
    ref, st_ref = oracle.lowbit_quantize(bits, w)
    assert st == st_ref == oracle.ERR_NONFINITE
    assert np.array_equal(got, ref)


def _experts(bits, hidden, inter, E, wid=WID, layer=0):
    """Oracle-quantised expert buffers (host), and device copies of each in an
    allocation of its own with the two address tables."""
    import torch
    gus, dns = [], []
    for e in range(E):
        wgu, wdn = synth.moe_expert_weights(wid, layer, e, hidden, inter)
        gb, st = oracle.lowbit_quantize(bits, wgu)
        db, st2 = oracle.lowbit_quantize(bits, wdn)
        assert st == st2 == 0
        gus.append(gb)
        dns.append(db)
    gdev = [torch.from_numpy(b).cuda() for b in gus]
    ddev = [torch.from_numpy(b).cuda() for b in dns]
    return (np.stack(gus), np.stack(dns), loader.expert_table(gdev), loader.expert_table(ddev),
            (gdev, ddev))


def _run(bits, x, wr, top_k, gtab, dtab, hidden, inter, ws=None):
    import torch
    E = wr.shape[0]
    out = torch.empty(hidden, dtype=torch.int16, device="cuda")
    idx = torch.empty(top_k, dtype=torch.int32, device="cuda")
    prob = torch.empty(top_k, dtype=torch.float32, device="cuda")
    wsb = thinmx.tt_moe_lowbit_workspace_bytes(inter, E, top_k)
    if ws is None:
        ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device="cuda")
    thinmx.tt_moe_lowbit_topk_mlp(bits, gu.dev(x), hidden, inter, gu.dev(wr), E, top_k, gtab,
                                  dtab, out, idx, prob, ws, wsb)
    torch.cuda.synchronize()
    h = gu.host(ws[:top_k * inter * 4]).view(np.float32).reshape(top_k, inter)
    return gu.host(out, np.uint16), gu.host(idx), gu.host(prob), h


def _check_layer(bits, hidden, inter, E, top_k, wid):
    r = synth.moe_router_inputs(wid, 0, hidden, E)
    gus, dns, gtab, dtab, keep = _experts(bits, hidden, inter, E, wid)
    out, idx, prob, h = _run(bits, r["x"], r["wr"], top_k, gtab, dtab, hidden, inter)
    ref, ridx, rp, _, rh, st = oracle.moe_lowbit_mlp(bits, r["x"], r["wr"], top_k, gus, dns, inter)
    assert st == 0
    assert np.array_equal(idx, ridx)
    assert np.allclose(prob, rp, rtol=2e-6, atol=0)
    # h is fp32: within 1e-5 of its largest magnitude, cosine as for the bf16 outputs
    for j in range(top_k):
        err = np.max(np.abs(h[j] - rh[j])) / np.max(np.abs(rh[j]))
        cos = np.dot(h[j], rh[j]) / (np.linalg.norm(h[j]) * np.linalg.norm(rh[j]))
        assert err <= 1e-5 and cos >= 0.99999, (j, err, cos)
    assert_float_parity(out, ref, f"Q{bits} MoE {hidden}/{inter} E{E} top{top_k}")
    assert gu.device_error() == 0
    return keep


@pytest.mark.parametrize("bits", [1, 2])
@pytest.mark.parametrize("hidden,inter,E,top_k", [(64, 32, 4, 1), (256, 96, 8, 2),
                                                  (2880, 2880, 32, 4), (1024, 4096, 64, 8),
                                                  (4096, 512, 40, 3),
                                                  # the largest hidden and inter (8192)
                                                  (8192, 1024, 4, 2), (1024, 8192, 4, 2),
                                                  (96, 64, 256, 8)])
def test_moe_lowbit_layer(bits, hidden, inter, E, top_k):
    _check_layer(bits, hidden, inter, E, top_k, WID + hidden + E)


@pytest.mark.parametrize("bits", [1, 2])
def test_moe_lowbit_layers_in_one_graph(bits):
    """Three layers PDL-chained in one CUDA graph, each reading the previous
    layer's output, replayed twice; each layer against the oracle on the
    input the GPU gave it."""
    import torch
    hidden, inter, E, top_k = 512, 256, 16, 4
    layers = []
    for l in range(3):
        r = synth.moe_router_inputs(WID + 7, l, hidden, E)
        gus, dns, gtab, dtab, keep = _experts(bits, hidden, inter, E, WID + 7, l)
        layers.append((r["wr"], gu.dev(r["wr"]), gus, dns, gtab, dtab, keep))
    x0 = gu.dev(synth.moe_router_inputs(WID + 7, 9, hidden, E)["x"])
    wsb = thinmx.tt_moe_lowbit_workspace_bytes(inter, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    outs = [torch.empty(hidden, dtype=torch.int16, device="cuda") for _ in range(3)]
    idxs = [torch.empty(top_k, dtype=torch.int32, device="cuda") for _ in range(3)]
    probs = [torch.empty(top_k, dtype=torch.float32, device="cuda") for _ in range(3)]

    def step():
        x = x0
        for l, (_, wr, _, _, gtab, dtab, _) in enumerate(layers):
            thinmx.tt_moe_lowbit_topk_mlp(bits, x, hidden, inter, wr, E, top_k, gtab, dtab,
                                          outs[l], idxs[l], probs[l], ws, wsb)
            x = outs[l]

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
    x = gu.host(x0, np.uint16)
    for l, (wr_h, _, gus, dns, _, _, _) in enumerate(layers):
        ref, ridx, _, _, _, _ = oracle.moe_lowbit_mlp(bits, x, wr_h, top_k, gus, dns, inter)
        got = gu.host(outs[l], np.uint16)
        assert np.array_equal(gu.host(idxs[l]), ridx)
        assert_float_parity(got, ref, f"Q{bits} graph layer {l}")
        x = got


def test_moe_lowbit_is_deterministic():
    hidden, inter, E, top_k = 2880, 2880, 32, 4
    r = synth.moe_router_inputs(WID + 3, 0, hidden, E)
    _, _, gtab, dtab, keep = _experts(1, hidden, inter, E, WID + 3)
    a = _run(1, r["x"], r["wr"], top_k, gtab, dtab, hidden, inter)
    b = _run(1, r["x"], r["wr"], top_k, gtab, dtab, hidden, inter)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


def test_moe_lowbit_bad_expert_pointer_is_reported_not_used():
    import torch
    hidden, inter, E, top_k = 256, 128, 8, 2
    r = synth.moe_router_inputs(WID + 4, 0, hidden, E)
    _, _, gtab, dtab, keep = _experts(2, hidden, inter, E, WID + 4)
    null_tab = torch.zeros(E, dtype=torch.int64, device="cuda")  # every entry NULL
    out, _, _, h = _run(2, r["x"], r["wr"], top_k, null_tab, dtab, hidden, inter)
    assert gu.device_error() == 1  # TT_ERR_NULL, read and cleared
    assert not h.any() and not out.any()  # nothing was read through the NULL entries
    mis = gtab.clone() + 8  # misaligned addresses (never dereferenced)
    _run(2, r["x"], r["wr"], top_k, mis, dtab, hidden, inter)
    assert gu.device_error() == 3  # TT_ERR_ALIGN
