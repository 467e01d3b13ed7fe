"""Comparison helpers for the GPU-vs-oracle parity tests (test infrastructure).

Float outputs are bf16; the oracle's reference r is the UNROUNDED fp64 value.
Tolerance (stated once, used by every float parity test):

  * max relative error <= 2e-3, normwise: max_i e_i / max_i |r_i| where
    e_i = max(0, |y_i - r_i| - ulp_bf16(r_i)/2) is the error beyond the
    unavoidable rounding of the output to bf16 (ulp/2 = 2^(floor(log2|r|)-8),
    up to 3.9e-3 relative by itself);
  * cosine(y, r) >= 0.99999, computed in fp64 over the bf16 outputs.

Codes, scales, zero points, expert indices and dequantised weights are
compared bit for bit instead.
"""
import numpy as np

TOL_REL = 2e-3
TOL_COS = 0.99999


def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_half_ulp(r) -> np.ndarray:
    a = np.abs(np.asarray(r, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def float_errors(y_bits, r):
    y = bf16_to_f64(y_bits).ravel()
    r = np.asarray(r, np.float64).ravel()
    scale = np.max(np.abs(r)) if r.size else 0.0
    excess = np.maximum(0.0, np.abs(y - r) - bf16_half_ulp(r))
    rel = float(np.max(excess) / scale) if scale > 0 else float(np.max(excess, initial=0.0))
    ny, nr = np.linalg.norm(y), np.linalg.norm(r)
    cos = float(np.dot(y, r) / (ny * nr)) if ny > 0 and nr > 0 else (1.0 if ny == nr else 0.0)
    return rel, cos


def assert_float_parity(y_bits, r, what=""):
    assert np.all(np.isfinite(bf16_to_f64(y_bits))), f"{what}: non-finite output"
    rel, cos = float_errors(y_bits, r)
    assert rel <= TOL_REL, f"{what}: normwise rel err {rel:.3e} > {TOL_REL}"
    assert cos >= TOL_COS, f"{what}: cosine {cos:.8f} < {TOL_COS}"
    return rel, cos
