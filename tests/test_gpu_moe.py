"""GPU parity of the MoE layer: router logits -> top-k (bit-exact indices,
ties to the lower index) -> softmax -> selected experts' MXFP4 gate/up
SwiGLU and down, weighted sum (float tolerance of tests/parity.py)."""
import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth

from . import gpu_util as gu
from .parity import assert_float_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ensure_lib()
    assert gu.device_error() == 0


def _case(E, H, I, K, wid, tie_rows=None):
    r = synth.moe_router_inputs(wid, 0, H, E)
    x, wr = r["x"], r["wr"]
    if tie_rows:
        for a, b in tie_rows:
            wr[b] = wr[a]
    gus, dns = [], []
    for e in range(E):
        g, d = synth.moe_expert_weights(wid, 0, e, H, I)
        gus.append(g)
        dns.append(d)
    gup, dnp, (gc, gs, dc, ds), _bufs = gu.build_moe_experts(gus, dns, H, I)
    out, idx, prob = gu.run_moe(x, wr, K, gup, dnp, H, I)
    ref, ridx, rp, rlg, st = oracle.moe_mlp(x, wr, K, gc, gs, dc, ds)
    assert st == oracle.OK
    return out, idx, prob, ref, ridx, rp, rlg


@pytest.mark.parametrize("E,H,I,K", [(6, 64, 96, 3), (8, 320, 640, 4), (32, 1024, 512, 4),
                                     (5, 2880, 2880, 1), (16, 256, 2048, 8),
                                     # the gpt-oss expert shape (its own kernel instance) at
                                     # top-8: about ten 16-wide h slices per CTA
                                     (8, 2880, 2880, 8),
                                     (8, 4096, 1024, 8),
                                     # the down columns come in two row chunks of 3584 and
                                     # 1024 rows (shared memory too small for whole columns)
                                     (4, 4608, 1024, 4),
                                     # more experts than lanes: the general top-k path
                                     (64, 256, 128, 4),
                                     # the largest hidden (one gate/up slot per warp, two row
                                     # chunks), every expert selected, a single expert
                                     (2, 8192, 256, 2), (4, 1024, 512, 4), (1, 320, 640, 1)])
def test_moe_small_shapes(E, H, I, K):
    out, idx, prob, ref, ridx, rp, rlg = _case(E, H, I, K, 98)
    assert list(idx) == list(ridx)
    np.testing.assert_allclose(prob, rp, rtol=2e-6, atol=1e-7)
    assert_float_parity(out, ref, f"moe E={E} H={H} I={I} k={K}")
    assert gu.device_error() == 0


def test_moe_router_exact_ties_go_to_lower_index():
    # duplicated router rows give bit-identical logits on both sides
    E, H, I, K = 8, 256, 128, 4
    r = synth.moe_router_inputs(99, 0, H, E)
    lg = oracle.router_logits(r["x"], r["wr"])
    top = int(np.argmax(lg))
    ties = [(top, e) for e in range(E) if e != top][:3]
    out, idx, prob, ref, ridx, rp, rlg = _case(E, H, I, K, 99, tie_rows=ties)
    assert list(idx) == list(ridx)
    assert sorted(idx) == sorted([top] + [b for _, b in ties])
    assert list(idx) == sorted(idx)  # equal logits -> ascending index
    np.testing.assert_allclose(prob, 0.25, rtol=1e-6)
    assert_float_parity(out, ref, "moe ties")


def test_moe_full_gptoss_layer():
    c = synth.MOE
    out, idx, prob, ref, ridx, rp, rlg = _case(c.experts, c.hidden, c.inter, c.top_k, c.wid)
    srt = np.sort(rlg.astype(np.float64))[::-1]
    margin = srt[c.top_k - 1] - srt[c.top_k]
    assert margin > 0, "4th/5th logits tie in fp32: the case would not pin the order"
    assert list(idx) == list(ridx)
    np.testing.assert_allclose(prob, rp, rtol=2e-6, atol=1e-7)
    assert_float_parity(out, ref, "moe gpt-oss-20b layer")


def test_moe_workspace_reused_across_calls():
    """Consecutive calls on one workspace give the same bits as fresh
    workspaces; the 64-bit grid-wide counter advances by the grid size (one
    CTA per SM) per call and is never reset, and the router partial replicas
    are left cleared."""
    import torch
    from bit_weight_only_mxfp4_gb300 import thinmx
    E, H, I, K = 8, 320, 640, 4
    gus, dns = zip(*[synth.moe_expert_weights(41, 0, e, H, I) for e in range(E)])
    gup, dnp, _, _bufs = gu.build_moe_experts(list(gus), list(dns), H, I)
    wsb = thinmx.tt_moe_workspace_bytes(H, I, E, K)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    for layer in range(3):
        r = synth.moe_router_inputs(41, layer, H, E)
        ref_out, ref_idx, ref_prob = gu.run_moe(r["x"], r["wr"], K, gup, dnp, H, I)
        out = torch.empty(H, dtype=torch.int16, device="cuda")
        idx = torch.empty(K, dtype=torch.int32, device="cuda")
        prob = torch.empty(K, dtype=torch.float32, device="cuda")
        thinmx.tt_moe_mxfp4_topk_mlp(gu.dev(r["x"]), H, I, gu.dev(r["wr"]), E, K, gup, dnp, out,
                                     idx, prob, ws, wsb)
        torch.cuda.synchronize()
        assert np.array_equal(gu.host(out, np.uint16), ref_out)
        assert list(gu.host(idx)) == list(ref_idx)
        assert np.array_equal(gu.host(prob), ref_prob)
        cnt = gu.host(ws[:16]).view(np.uint64)
        assert list(cnt) == [0, (layer + 1) * sms]
        # the rest of the counter bytes and the router replicas (64 + 256 x 256 x 8 B)
        assert not gu.host(ws[16:524352]).any()
    assert gu.device_error() == 0


def test_moe_experts_in_scattered_allocations():
    """Experts are separate buffers at unrelated addresses: allocated in a
    shuffled order with unused allocations between them, and the tables list
    them in expert order."""
    import torch
    from bit_weight_only_mxfp4_gb300 import loader
    E, H, I, K = 8, 320, 640, 4
    r = synth.moe_router_inputs(43, 0, H, E)
    gus, dns = zip(*[synth.moe_expert_weights(43, 0, e, H, I) for e in range(E)])
    _, _, (gc, gs, dc, ds), (gb, db) = gu.build_moe_experts(list(gus), list(dns), H, I)
    order = [5, 2, 7, 0, 3, 6, 1, 4]
    moved_g, moved_d, gaps = [None] * E, [None] * E, []
    for e in order:
        gaps.append(torch.empty(4096 * (e + 1), dtype=torch.uint8, device="cuda"))
        moved_g[e] = gb[e].clone()
        gaps.append(torch.empty(256, dtype=torch.uint8, device="cuda"))
        moved_d[e] = db[e].clone()
    out, idx, prob = gu.run_moe(r["x"], r["wr"], K, loader.expert_table(moved_g),
                                loader.expert_table(moved_d), H, I)
    ref, ridx, rp, rlg, st = oracle.moe_mlp(r["x"], r["wr"], K, gc, gs, dc, ds)
    assert list(idx) == list(ridx)
    assert_float_parity(out, ref, "moe scattered experts")
    assert gu.device_error() == 0


def test_moe_bad_expert_pointer_is_reported_not_used():
    """A NULL or misaligned table entry of a SELECTED expert is reported
    through the device error word before any copy from it (the output is left
    alone); a bad entry of an expert that is not selected is never read."""
    import torch
    from bit_weight_only_mxfp4_gb300 import loader, thinmx
    E, H, I, K = 8, 256, 128, 2
    r = synth.moe_router_inputs(44, 0, H, E)
    gus, dns = zip(*[synth.moe_expert_weights(44, 0, e, H, I) for e in range(E)])
    _, _, (gc, gs, dc, ds), (gb, db) = gu.build_moe_experts(list(gus), list(dns), H, I)
    ref, ridx, rp, rlg, st = oracle.moe_mlp(r["x"], r["wr"], K, gc, gs, dc, ds)
    unused = [e for e in range(E) if e not in set(int(i) for i in ridx)][0]
    base_g = [b.data_ptr() for b in gb]
    base_d = [b.data_ptr() for b in db]

    def call(tg, td):
        tgt = torch.tensor(tg, dtype=torch.int64, device="cuda")
        tdt = torch.tensor(td, dtype=torch.int64, device="cuda")
        out, idx, prob = gu.run_moe(r["x"], r["wr"], K, tgt, tdt, H, I)
        return out, idx, gu.device_error()

    # an unselected expert's entry is never read
    tg = list(base_g)
    tg[unused] = 0
    out, idx, errw = call(tg, base_d)
    assert errw == 0 and list(idx) == list(ridx)
    assert_float_parity(out, ref, "moe with an unused NULL entry")
    # a selected expert with a misaligned gate/up or a NULL down entry
    sel = int(ridx[0])
    tg = list(base_g)
    tg[sel] += 8
    assert call(tg, base_d)[2] == 3  # TT_ERR_ALIGN
    td = list(base_d)
    td[sel] = 0
    assert call(base_g, td)[2] == 1  # TT_ERR_NULL
    # the library is fine afterwards
    out, idx, errw = call(base_g, base_d)
    assert errw == 0
    assert_float_parity(out, ref, "moe after the reported calls")
