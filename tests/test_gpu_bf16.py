"""GPU parity of the bf16 gate/up SwiGLU matvec (the layers kept in bf16)."""
import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()


def _run(wg, wu, x):
    import torch
    n, k = wg.shape
    m = x.shape[0]
    h = torch.empty((m, n), dtype=torch.int16, device="cuda")
    thinmx.tt_bf16_swiglu_matvec(gu.dev(wg), gu.dev(wu), n, k, gu.dev(x), m, h)
    torch.cuda.synchronize()
    return gu.host(h, np.uint16)


@pytest.mark.parametrize("n,k,m", [(37, 64, 1), (300, 2048, 1), (129, 2056, 1), (50, 5120, 2),
                                   (70, 1000, 3), (33, 2880, 4), (20, 4096, 8)])
def test_bf16_swiglu_shapes(n, k, m):
    d = synth.bf16_gate_up_inputs(95, 0, n, k, m)
    h = _run(d["wg"], d["wu"], d["x"])
    ref = oracle.bf16_swiglu_matvec(d["wg"], d["wu"], d["x"])
    assert_float_parity(h, ref, f"bf16 n={n} k={k} m={m}")


def test_bf16_swiglu_full_layer():
    c = synth.STACK
    d = synth.bf16_gate_up_inputs(c.wid, c.mxfp4_layers, c.n, c.k, 1)
    h = _run(d["wg"], d["wu"], d["x"])
    ref = oracle.bf16_swiglu_matvec(d["wg"], d["wu"], d["x"])
    assert_float_parity(h, ref, "bf16 11008x2048")
    assert np.mean(h.ravel() == oracle.bf16_round_array(ref.ravel())) > 0.99
