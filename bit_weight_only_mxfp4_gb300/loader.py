"""Weight loader: canonical fp32 / MXFP4 tensors on the device -> the packed
layouts the matvec kernels stream.  Every step runs in the library's CUDA
kernels through the C ABI; torch only allocates the buffers."""
from __future__ import annotations

import torch

from . import thinmx


def quantize_mxfp4(w: torch.Tensor, status: torch.Tensor | None = None):
    """fp32 [n, k] (k % 32 == 0) -> (codes uint8 [n, k/2], scales uint8 [n, k/32])."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous()
    n, k = w.shape
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n, k // 32), dtype=torch.uint8, device=w.device)
    thinmx.tt_quantize_mxfp4(w, n, k, codes, scales, status)
    return codes, scales


def pack_swiglu(gate, up, n: int, k: int) -> torch.Tensor:
    """gate/up = (codes, scales, postscale fp32 [n] or None) -> packed buffer."""
    nbytes = thinmx.tt_mxfp4_swiglu_packed_bytes(n, k)
    if nbytes == 0:
        raise ValueError(f"unsupported gate/up shape n={n} k={k}")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=gate[0].device)
    thinmx.tt_mxfp4_pack_swiglu(gate[0], gate[1], gate[2], up[0], up[1], up[2], n, k, packed,
                                nbytes)
    return packed


def mxfp4_gate_up_from_f32(wg: torch.Tensor, wu: torch.Tensor, pg=None, pu=None) -> torch.Tensor:
    """Quantise both fp32 matrices and pack them; the canonical codes are freed."""
    n, k = wg.shape
    gc, gs = quantize_mxfp4(wg)
    uc, us = quantize_mxfp4(wu)
    packed = pack_swiglu((gc, gs, pg), (uc, us, pu), n, k)
    del gc, gs, uc, us
    return packed


def expert_table(buffers) -> torch.Tensor:
    """The device array of expert buffer addresses the MoE entry points take
    (one int64 per expert, in expert order).  The buffers must stay alive as
    long as the table is used."""
    dev = buffers[0].device
    return torch.tensor([b.data_ptr() for b in buffers], dtype=torch.int64, device=dev)


def moe_expert_from_f32(w_gate_up: torch.Tensor, w_down: torch.Tensor):
    """One expert's fp32 gate/up [2*inter, hidden] (gate rows first) and down
    [hidden, inter] matrices -> its own packed gate/up and down buffers."""
    two_i, hidden = w_gate_up.shape
    inter = two_i // 2
    gc, gs = quantize_mxfp4(w_gate_up)
    gu = pack_swiglu((gc[:inter], gs[:inter], None), (gc[inter:], gs[inter:], None), inter,
                     hidden)
    dc, ds = quantize_mxfp4(w_down)
    nbytes = thinmx.tt_mxfp4_rows_packed_bytes(hidden, inter)
    dn = torch.empty(nbytes, dtype=torch.uint8, device=w_down.device)
    thinmx.tt_mxfp4_pack_rows(dc, ds, hidden, inter, dn, nbytes)
    return gu, dn
