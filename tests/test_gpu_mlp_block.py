"""The dense decode MLP block: the down-projection matvecs (MXFP4 on canonical
buffers, bf16; the FP8 one is in test_gpu_fp8.py) against the oracle, and
gate/up SwiGLU -> down chained layer after layer in one captured CUDA graph
(programmatic dependent launch between the calls), each layer checked
against the oracle's composition on that layer's own input."""
import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _mxfp4_rows(n, k, m, post=True, wid=130, x=None):
    import torch
    d = synth.gate_up_inputs(wid, 0, n, k, m=m, postscale=post)
    codes, scales, _ = gu.quantize(d["wg"])
    ps = None if d["pg"] is None else gu.dev(d["pg"])
    x = d["x"] if x is None else x
    y = torch.empty((m, n), dtype=torch.int16, device="cuda")
    thinmx.tt_mxfp4_matvec(codes, scales, ps, n, k, gu.dev(x), m, y)
    torch.cuda.synchronize()
    ref = oracle.mxfp4_matvec(gu.host(codes), gu.host(scales), d["pg"], x)
    return gu.host(y, np.uint16), ref


@pytest.mark.parametrize("n,k,m,post", [(1, 32, 1, True), (7, 96, 2, False), (129, 1024, 1, True),
                                        (300, 2880, 3, True), (33, 5120, 8, False),
                                        (21, 16384, 1, True), (64, 8192, 4, True),
                                        (2048, 11008, 1, False),
                                        # K = 11008 at m = 1: the one-wave kernel, with one row
                                        # per warp, two rows for some warps, and few rows
                                        (2048, 11008, 1, True), (3001, 11008, 1, True),
                                        (5, 11008, 1, False), (2048, 11008, 2, True)])
def test_mxfp4_matvec_shapes(n, k, m, post):
    y, ref = _mxfp4_rows(n, k, m, post)
    for i in range(m):
        assert_float_parity(y[i], ref[i], f"mxfp4 down n={n} k={k} m={m} row {i}")
    assert gu.device_error() == 0


def test_mxfp4_matvec_blocks_of_very_different_magnitude():
    n, k = 48, 2048
    d = synth.gate_up_inputs(131, 0, n, k, m=1)
    e = synth.rng(131, 1).integers(-60, 61, k // 32)
    xf = synth.bf16_bits_to_f32(d["x"]).reshape(-1, 32) * np.ldexp(np.float32(1), e)[:, None]
    x = synth.f32_to_bf16_bits(xf.reshape(1, k).astype(np.float32))
    y, ref = _mxfp4_rows(n, k, 1, True, wid=131, x=x)
    assert_float_parity(y, ref, "mxfp4 down, x blocks over 2^-60..2^60")


@pytest.mark.parametrize("n,k,m", [(1, 8, 1), (37, 96, 2), (300, 2880, 5), (2048, 11008, 1),
                                   (65, 4104, 8),
                                   # K = 11008 at m = 1: one row per CTA step; rows beyond
                                   # two per CTA, and fewer rows than CTAs
                                   (3001, 11008, 1), (5, 11008, 1), (700, 11008, 2)])
def test_bf16_matvec_shapes(n, k, m):
    import torch
    d = synth.bf16_gate_up_inputs(132, 0, n, k, m=m)
    y = torch.empty((m, n), dtype=torch.int16, device="cuda")
    thinmx.tt_bf16_matvec(gu.dev(d["wg"]), n, k, gu.dev(d["x"]), m, y)
    torch.cuda.synchronize()
    ref = oracle.bf16_matvec(d["wg"], d["x"])
    got = gu.host(y, np.uint16)
    for i in range(m):
        assert_float_parity(got[i], ref[i], f"bf16 down n={n} k={k} m={m} row {i}")


class _Layer:
    """One MLP layer's weights on the device (and what the oracle needs)."""

    def __init__(self, profile, hidden, inter, wid, layer):
        import torch
        d = synth.gate_up_inputs(wid, layer, inter, hidden)
        wd = synth.normal_f32(synth.rng(wid, layer, 7), (hidden, inter), synth.WEIGHT_STD)
        self.profile, self.hidden, self.inter = profile, hidden, inter
        if profile in ("mxfp4+bf16", "mxfp4"):
            gc, gs, _ = gu.quantize(d["wg"])
            uc, us, _ = gu.quantize(d["wu"])
            self.pg, self.pu = gu.dev(d["pg"]), gu.dev(d["pu"])
            self.packed = gu.pack_swiglu(gc, gs, self.pg, uc, us, self.pu, inter, hidden)
            self.gate = (gu.host(gc), gu.host(gs), d["pg"])
            self.up = (gu.host(uc), gu.host(us), d["pu"])
        else:  # fp8
            self.g8 = self._fp8(d["wg"])
            self.u8 = self._fp8(d["wu"])
        if profile == "mxfp4+bf16":
            self.wd_bf16 = synth.f32_to_bf16_bits(wd)
            self.wd = gu.dev(self.wd_bf16)
        elif profile == "mxfp4":
            self.dc, self.ds, _ = gu.quantize(wd)
        else:
            self.d8 = self._fp8(wd)
        self.h = torch.empty((1, inter), dtype=torch.int16, device="cuda")
        self.y = torch.empty((1, hidden), dtype=torch.int16, device="cuda")

    @staticmethod
    def _fp8(w):
        import torch
        n, k = w.shape
        codes = torch.empty((n, k), dtype=torch.uint8, device="cuda")
        scales = torch.empty(n, dtype=torch.float32, device="cuda")
        thinmx.tt_quantize_fp8(gu.dev(w), n, k, codes, scales)
        return codes, scales

    def run(self, x):
        H, I = self.hidden, self.inter
        if self.profile == "fp8":
            thinmx.tt_fp8_swiglu_matvec(self.g8[0], self.g8[1], self.u8[0], self.u8[1], I, H, x,
                                        1, self.h)
            thinmx.tt_fp8_matvec(self.d8[0], self.d8[1], H, I, self.h, 1, self.y)
            return
        thinmx.tt_mxfp4_swiglu_matvec(self.packed, I, H, x, 1, self.h)
        if self.profile == "mxfp4+bf16":
            thinmx.tt_bf16_matvec(self.wd, H, I, self.h, 1, self.y)
        else:
            thinmx.tt_mxfp4_matvec(self.dc, self.ds, None, H, I, self.h, 1, self.y)

    def reference(self, x_bits):
        """The oracle's gate/up SwiGLU on this layer's input, rounded to bf16
        as the block hands it on, then the oracle's down projection."""
        if self.profile == "fp8":
            h = oracle.fp8_swiglu_matvec((gu.host(self.g8[0]), gu.host(self.g8[1])),
                                         (gu.host(self.u8[0]), gu.host(self.u8[1])), x_bits)
        else:
            h = oracle.mxfp4_swiglu_matvec(self.gate, self.up, x_bits)
        hb = oracle.bf16_round_array(h.ravel()).reshape(h.shape)
        if self.profile == "mxfp4+bf16":
            y = oracle.bf16_matvec(self.wd_bf16, hb)
        elif self.profile == "mxfp4":
            y = oracle.mxfp4_matvec(gu.host(self.dc), gu.host(self.ds), None, hb)
        else:
            y = oracle.fp8_matvec(gu.host(self.d8[0]), gu.host(self.d8[1]), hb)
        return h, y


@pytest.mark.parametrize("profile", ["mxfp4+bf16", "mxfp4", "fp8"])
def test_mlp_block_stack_in_one_graph(profile):
    """Three layers, each gate/up SwiGLU -> down, layer l + 1 reading layer
    l's output: six PDL-chained kernels in one CUDA graph, replayed twice."""
    import torch
    H, I = 512, 1408
    layers = [_Layer(profile, H, I, 133, l) for l in range(3)]
    x0 = gu.dev(synth.normal_bf16(synth.rng(133, 9), (1, H)))

    def step():
        x = x0
        for L in layers:
            L.run(x)
            x = L.y

    step()  # eager once (kernel attributes are set outside the capture)
    torch.cuda.synchronize()
    for L in layers:
        L.h.zero_()
        L.y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert gu.device_error() == 0
    x_bits = gu.host(x0, np.uint16)
    for l, L in enumerate(layers):
        h_ref, y_ref = L.reference(x_bits)
        h = gu.host(L.h, np.uint16)
        y = gu.host(L.y, np.uint16)
        assert_float_parity(h, h_ref, f"{profile} layer {l} h")
        # the down projection against the oracle's composition
        assert_float_parity(y, y_ref, f"{profile} layer {l} y")
        # and exactly on the h the GPU handed on
        if profile == "mxfp4+bf16":
            y_own = oracle.bf16_matvec(L.wd_bf16, h)
        elif profile == "mxfp4":
            y_own = oracle.mxfp4_matvec(gu.host(L.dc), gu.host(L.ds), None, h)
        else:
            y_own = oracle.fp8_matvec(gu.host(L.d8[0]), gu.host(L.d8[1]), h)
        assert_float_parity(y, y_own, f"{profile} layer {l} y on its own h")
        x_bits = y  # the next layer's input is this layer's output, as the GPU saw it
    assert np.any(bf16_to_f64(y) != 0)
