"""The workspace-free MoE entry point (for callers that cannot allocate
device memory) against the regular one that takes a caller workspace.

Kept in a file of its own that pytest collects last: a failure here stops a
-x run only after every other test has run.  It passes in a fresh process
and after the other tests (it builds its own inputs)."""
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
    assert gu.device_error() == 0


def _static_call(x, wr, top_k, gu_table, dn_table, hidden, inter):
    import torch
    E = wr.shape[0]
    out = torch.empty(hidden, dtype=torch.int16, device="cuda")
    idx = torch.empty(top_k, dtype=torch.int32, device="cuda")
    prob = torch.empty(top_k, dtype=torch.float32, device="cuda")
    thinmx.tt_moe_mxfp4_topk_mlp_static(gu.dev(x), hidden, inter, gu.dev(wr), E, top_k,
                                        gu_table, dn_table, out, idx, prob)
    torch.cuda.synchronize()
    return gu.host(out, np.uint16), gu.host(idx), gu.host(prob)


def _same(a, b):
    """Both entry points run the same kernel with fixed-order sums: the
    results agree bit for bit."""
    assert np.array_equal(a[0], b[0])
    assert list(a[1]) == list(b[1])
    assert np.array_equal(np.asarray(a[2]).view(np.uint32), np.asarray(b[2]).view(np.uint32))


@pytest.mark.parametrize("E,H,I,K", [(8, 320, 640, 4),
                                     # the gpt-oss-20b layer the 4096 cap is sized for
                                     (32, 2880, 2880, 4)])
def test_static_scratch_moe_matches_workspace_moe_twice(E, H, I, K):
    r = synth.moe_router_inputs(77, 0, H, E)
    gus, dns = zip(*[synth.moe_expert_weights(77, 0, e, H, I) for e in range(E)])
    gup, dnp, (gc, gs, dc, ds), _bufs = gu.build_moe_experts(list(gus), list(dns), H, I)
    ref = gu.run_moe(r["x"], r["wr"], K, gup, dnp, H, I)
    oref, oidx, _, _, st = oracle.moe_mlp(r["x"], r["wr"], K, gc, gs, dc, ds)
    assert list(ref[1]) == list(oidx)
    assert_float_parity(ref[0], oref, "workspace MoE")
    for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
        _same(_static_call(r["x"], r["wr"], K, gup, dnp, H, I), ref)
    assert gu.device_error() == 0


def test_static_scratch_survives_a_workspace_call_in_between():
    """static -> workspace -> static on other inputs: the counter the fixed
    scratch keeps across calls stays consistent when other calls run on
    their own workspaces in between."""
    E, H, I, K = 8, 320, 640, 4
    gus, dns = zip(*[synth.moe_expert_weights(78, 0, e, H, I) for e in range(E)])
    gup, dnp, _, _bufs = gu.build_moe_experts(list(gus), list(dns), H, I)
    ins = [synth.moe_router_inputs(78, layer, H, E) for layer in range(3)]
    refs = [gu.run_moe(d["x"], d["wr"], K, gup, dnp, H, I) for d in ins]
    _same(_static_call(ins[0]["x"], ins[0]["wr"], K, gup, dnp, H, I), refs[0])
    _same(gu.run_moe(ins[1]["x"], ins[1]["wr"], K, gup, dnp, H, I), refs[1])
    _same(_static_call(ins[2]["x"], ins[2]["wr"], K, gup, dnp, H, I), refs[2])
    assert gu.device_error() == 0


def test_static_scratch_moe_rejects_oversize_before_launch():
    A = 1 << 20  # never dereferenced: the size check comes first
    E, top_k, inter = 8, 4, 256
    hidden = 8192  # a valid shape, but beyond what the fixed scratch holds
    assert hidden > thinmx.TT_MOE_STATIC_MAX_HIDDEN
    st = thinmx.load().tt_moe_mxfp4_topk_mlp_static(A, hidden, inter, A, E, top_k, A, A, A, A, A,
                                                    None)
    assert st == 8  # TT_ERR_SIZE
