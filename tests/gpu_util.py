"""Device-side helpers for the GPU parity tests: torch only allocates and
copies; every computation goes through the thinmx C ABI."""
import numpy as np
import torch

from bit_weight_only_mxfp4_gb300 import build as tt_build
from bit_weight_only_mxfp4_gb300 import thinmx


def ensure_lib():
    tt_build.build()
    return thinmx.load()


def dev(a) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return a.view(dtype) if dtype is not None else a


def quantize(w_np):
    """fp32 [n, k] -> (codes, scales) device tensors and the status word."""
    n, k = w_np.shape
    w = dev(w_np.astype(np.float32))
    codes = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((n, k // 32), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    thinmx.tt_quantize_mxfp4(w, n, k, codes, scales, status)
    return codes, scales, status


def pack_swiglu(gc, gs, gp, uc, us, up, n, k):
    nbytes = thinmx.tt_mxfp4_swiglu_packed_bytes(n, k)
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    thinmx.tt_mxfp4_pack_swiglu(gc, gs, gp, uc, us, up, n, k, packed, nbytes)
    return packed


def swiglu(packed, n, k, x_np):
    m = x_np.shape[0]
    x = dev(x_np)
    h = torch.empty((m, n), dtype=torch.int16, device="cuda")
    thinmx.tt_mxfp4_swiglu_matvec(packed, n, k, x, m, h)
    torch.cuda.synchronize()
    return host(h, np.uint16)


def device_error():
    return thinmx.tt_device_error_read()


def build_moe_experts(gu_list, dn_list, hidden, inter):
    """fp32 expert matrices (numpy) -> one packed gate/up and one packed down
    buffer per expert (separate allocations) and the two device tables of
    their addresses the MoE call takes, plus the canonical codes/scales
    (host) for the oracle.  Returns (gu_table, dn_table, canonical, buffers);
    the buffers must outlive every call that uses the tables."""
    import torch
    from bit_weight_only_mxfp4_gb300 import loader
    E = len(gu_list)
    sw = thinmx.tt_mxfp4_swiglu_packed_bytes(inter, hidden)
    rw = thinmx.tt_mxfp4_rows_packed_bytes(hidden, inter)
    gc_h = np.zeros((E, 2 * inter, hidden // 2), np.uint8)
    gs_h = np.zeros((E, 2 * inter, hidden // 32), np.uint8)
    dc_h = np.zeros((E, hidden, inter // 2), np.uint8)
    ds_h = np.zeros((E, hidden, inter // 32), np.uint8)
    gbufs, dbufs = [], []
    for e in range(E):
        gc, gs, _ = quantize(gu_list[e])
        g = torch.empty(sw, dtype=torch.uint8, device="cuda")
        thinmx.tt_mxfp4_pack_swiglu(gc[:inter], gs[:inter], None, gc[inter:], gs[inter:], None,
                                    inter, hidden, g, sw)
        dc, ds, _ = quantize(dn_list[e])
        d = torch.empty(rw, dtype=torch.uint8, device="cuda")
        thinmx.tt_mxfp4_pack_rows(dc, ds, hidden, inter, d, rw)
        gbufs.append(g)
        dbufs.append(d)
        gc_h[e], gs_h[e], dc_h[e], ds_h[e] = host(gc), host(gs), host(dc), host(ds)
    torch.cuda.synchronize()
    return (loader.expert_table(gbufs), loader.expert_table(dbufs), (gc_h, gs_h, dc_h, ds_h),
            (gbufs, dbufs))


def run_moe(x, wr, top_k, gu_table, dn_table, hidden, inter):
    import torch
    E = wr.shape[0]
    out = torch.empty(hidden, dtype=torch.int16, device="cuda")
    idx = torch.empty(top_k, dtype=torch.int32, device="cuda")
    prob = torch.empty(top_k, dtype=torch.float32, device="cuda")
    wsb = thinmx.tt_moe_workspace_bytes(hidden, inter, E, top_k)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    thinmx.tt_moe_mxfp4_topk_mlp(dev(x), hidden, inter, dev(wr), E, top_k, gu_table, dn_table,
                                 out, idx, prob, ws, wsb)
    torch.cuda.synchronize()
    return host(out, np.uint16), host(idx), host(prob)
