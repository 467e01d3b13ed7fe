"""The workspace-free MoE entry point (for callers that cannot allocate
device memory) against the regular one that takes a caller workspace.

Kept in a file of its own that pytest collects last: a failure here stops a
-x run only after every other test has run.  It passes in a fresh process
and after the other tests (it builds its own inputs)."""
import numpy as np
import pytest

from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _static_call(x, wr, top_k, gup, dnp, hidden, inter):
    import torch
    E = wr.shape[0]
    out = torch.empty(hidden, dtype=torch.int16, device="cuda")
    idx = torch.empty(top_k, dtype=torch.int32, device="cuda")
    prob = torch.empty(top_k, dtype=torch.float32, device="cuda")
    thinmx.tt_moe_mxfp4_topk_mlp_static(gu.dev(x), hidden, inter, gu.dev(wr), E, top_k, gup,
                                        dnp, out, idx, prob)
    torch.cuda.synchronize()
    return gu.host(out, np.uint16), gu.host(idx), gu.host(prob)


def test_static_scratch_moe_matches_workspace_moe_twice():
    E, H, I, K = 8, 320, 640, 4
    r = synth.moe_router_inputs(77, 0, H, E)
    gus, dns = zip(*[synth.moe_expert_weights(77, 0, e, H, I) for e in range(E)])
    gup, dnp, _ = gu.build_moe_experts(list(gus), list(dns), H, I)
    ref_out, ref_idx, ref_prob = gu.run_moe(r["x"], r["wr"], K, gup, dnp, H, I)
    for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
        out, idx, prob = _static_call(r["x"], r["wr"], K, gup, dnp, H, I)
        assert list(idx) == list(ref_idx)
        np.testing.assert_allclose(prob, ref_prob, rtol=2e-6, atol=1e-7)
        assert_float_parity(out, bf16_to_f64(ref_out), "static-scratch MoE")
    assert gu.device_error() == 0


def test_static_scratch_moe_rejects_oversize_before_launch():
    A = 1 << 20  # never dereferenced: the size check comes first
    E, top_k, inter = 8, 4, 256
    hidden = 8192  # a valid shape, but beyond what the fixed scratch holds
    assert hidden > thinmx.TT_MOE_STATIC_MAX_HIDDEN
    st = thinmx.load().tt_moe_mxfp4_topk_mlp_static(A, hidden, inter, A, E, top_k, A, A, A, A, A,
                                                    None)
    assert st == 8  # TT_ERR_SIZE
