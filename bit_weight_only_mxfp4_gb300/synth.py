"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and describes the workload shapes; it
holds none of the method's arithmetic (no quantisation, no dequantisation, no
matvec).  Both the CUDA path and the CPU oracle consume exactly the arrays
drawn here, so the two sides never depend on one another.

The workloads mirror the shapes the ThinTensor devlogs run on
(kerbin.cskartikey.dev/@satvikhardat, Dev Log #4: SmolLM3-3B with MXFP4
gate/up in layers 0:24; stardance.hackclub.com/projects/29750: gpt-oss-20b
MoE with INT4 dense Q/K/V/O, and Phi-4 in the final table).  No checkpoint
is involved: every weight is drawn from N(0, 0.02^2) and every activation
from N(0, 1), then stored as the format the path consumes.

Random streams: numpy PCG64 seeded with ``[0, workload_id, layer, part]``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

WEIGHT_STD = 0.02


def rng(workload: int, layer: int = 0, part: int = 0) -> np.random.Generator:
    """Independent PCG64 substream for (workload, layer, part); seed 0."""
    return np.random.default_rng([0, workload, layer, part])


def f32_to_bf16_bits(a) -> np.ndarray:
    """fp32 samples -> bf16 bit patterns, round to nearest even (the samples
    are finite).  Used only to store drawn activations in their format."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_f32(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def normal_bf16(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(g, shape, std))


def uniform_f32(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def random_bytes(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(0, 256, size=shape, dtype=np.uint8)


def random_scale_bytes(g: np.random.Generator, shape, lo: int = 118, hi: int = 124) -> np.ndarray:
    """E8M0 bytes in [lo, hi]; the default brackets 2^-9 .. 2^-3, the range
    N(0, 0.02^2) blocks quantise to."""
    return g.integers(lo, hi + 1, size=shape, dtype=np.uint8)


# --------------------------------------------------------------------------
# Workload descriptions (sizes only)
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class GateUpMLP:
    """One dense MLP gate/up layer at batch 1 (SmolLM3-3B sizes)."""
    wid: int = 0
    k: int = 2048
    n: int = 11008
    m: int = 1
    name: str = "mxfp4_gate_up_k2048_n11008_m1"


@dataclass(frozen=True)
class DecodeStack:
    """SmolLM3-3B-shaped 36-layer gate/up stack at batch 1: layers 0:24
    MXFP4 (+ fp32 row postscale), layers 24:36 bf16."""
    wid: int = 1
    k: int = 2048
    n: int = 11008
    layers: int = 36
    mxfp4_layers: int = 24
    name: str = "smollm3_3b_gate_up_stack_36l_mxfp4_0_24"


@dataclass(frozen=True)
class BatchSweep:
    """Phi-4-shaped gate/up sweep over the batch size."""
    wid: int = 2
    k: int = 5120
    n: int = 17920
    ms: tuple = (1, 2, 4, 8, 16, 32, 64)
    name: str = "phi4_gate_up_k5120_n17920_sweep"


@dataclass(frozen=True)
class MoELayer:
    """gpt-oss-20b-shaped MoE layer at batch 1: 32 experts, top-4."""
    wid: int = 3
    hidden: int = 2880
    inter: int = 2880
    experts: int = 32
    top_k: int = 4
    layers: int = 24
    name: str = "gptoss20b_moe_h2880_e32_top4"


@dataclass(frozen=True)
class Int4QKV:
    """Grouped affine INT4 dense QKV projection at batch 1 (gpt-oss-20b:
    64 q heads + 8 k + 8 v heads of 64; group 128, last group 64)."""
    wid: int = 4
    k: int = 2880
    n: int = 5120
    group: int = 128
    m: int = 1
    name: str = "gptoss20b_int4_qkv_k2880_n5120_g128"


@dataclass(frozen=True)
class GQADecode:
    """Single-token GQA attention over a bf16 KV cache: SmolLM3-3B heads
    (16 query heads, 4 kv heads, head_dim 128) and gpt-oss-20b heads (64,
    8, 64), at short and long contexts."""
    wid: int = 5
    shapes: tuple = (("smollm3_3b", 16, 4, 128), ("gptoss20b", 64, 8, 64))
    lens: tuple = (4096, 32768)
    name: str = "gqa_decode"


GATE_UP = GateUpMLP()
STACK = DecodeStack()
SWEEP = BatchSweep()
MOE = MoELayer()
QKV = Int4QKV()
GQA = GQADecode()


# --------------------------------------------------------------------------
# Draws for each workload
# --------------------------------------------------------------------------
def gate_up_inputs(wid: int, layer: int, n: int, k: int, m: int = 1,
                   postscale: bool = True):
    """fp32 gate/up weights, bf16 x [m, k] and fp32 postscales."""
    wg = normal_f32(rng(wid, layer, 0), (n, k), WEIGHT_STD)
    wu = normal_f32(rng(wid, layer, 1), (n, k), WEIGHT_STD)
    x = normal_bf16(rng(wid, layer, 2), (m, k), 1.0)
    if postscale:
        pg = uniform_f32(rng(wid, layer, 3), (n,), 0.9, 1.1)
        pu = uniform_f32(rng(wid, layer, 4), (n,), 0.9, 1.1)
    else:
        pg = pu = None
    return dict(wg=wg, wu=wu, x=x, pg=pg, pu=pu)


def bf16_gate_up_inputs(wid: int, layer: int, n: int, k: int, m: int = 1):
    wg = normal_bf16(rng(wid, layer, 0), (n, k), WEIGHT_STD)
    wu = normal_bf16(rng(wid, layer, 1), (n, k), WEIGHT_STD)
    x = normal_bf16(rng(wid, layer, 2), (m, k), 1.0)
    return dict(wg=wg, wu=wu, x=x)


def moe_router_inputs(wid: int, layer: int, hidden: int, experts: int):
    x = normal_bf16(rng(wid, layer, 0), (hidden,), 1.0)
    wr = normal_bf16(rng(wid, layer, 1), (experts, hidden), WEIGHT_STD)
    return dict(x=x, wr=wr)


def moe_expert_weights(wid: int, layer: int, expert: int, hidden: int, inter: int):
    """fp32 fused gate/up [2*inter, hidden] (gate rows first) and down
    [hidden, inter] for one expert."""
    gu = normal_f32(rng(wid, layer, 100 + 2 * expert), (2 * inter, hidden), WEIGHT_STD)
    dn = normal_f32(rng(wid, layer, 101 + 2 * expert), (hidden, inter), WEIGHT_STD)
    return gu, dn


def gqa_inputs(wid: int, case: int, heads: int, kv_heads: int, d: int, cap: int,
               k_std: float = 1.0):
    """q bf16 [heads][d] ~ N(0,1); k, v bf16 [kv_heads][cap][d] ~ N(0, k_std^2),
    N(0,1)."""
    q = normal_bf16(rng(wid, case, 0), (heads, d), 1.0)
    k = normal_bf16(rng(wid, case, 1), (kv_heads, cap, d), k_std)
    v = normal_bf16(rng(wid, case, 2), (kv_heads, cap, d), 1.0)
    return dict(q=q, k=k, v=v)


def int4_inputs(wid: int, layer: int, n: int, k: int, m: int = 1):
    w = normal_f32(rng(wid, layer, 0), (n, k), WEIGHT_STD)
    x = normal_bf16(rng(wid, layer, 1), (m, k), 1.0)
    return dict(w=w, x=x)



# --------------------------------------------------------------------------
# Bulk device-side draws for the benchmark (full-size stacks would take
# minutes in numpy).  torch's CUDA Philox generator, seeded per
# (workload, layer, part); same distributions as above.
# --------------------------------------------------------------------------
def torch_seed(workload: int, layer: int = 0, part: int = 0) -> int:
    return ((workload * 1000003 + layer) * 1009 + part) & 0x7FFFFFFF


def torch_normal(shape, std, workload, layer=0, part=0, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(torch_seed(workload, layer, part))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def torch_uniform(shape, lo, hi, workload, layer=0, part=0, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(torch_seed(workload, layer, part))
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo
