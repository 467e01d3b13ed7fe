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
