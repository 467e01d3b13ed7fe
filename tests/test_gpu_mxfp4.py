"""GPU parity of the MXFP4 quantiser, dequantiser, loader and gate/up SwiGLU
matvec against the CPU oracle (bit-exact for codes/scales/dequantised
weights; the float tolerance of tests/parity.py for h)."""
import os

import numpy as np
import pytest

import oracle
from bit_weight_only_mxfp4_gb300 import synth, thinmx

from . import gpu_util as gu
from .parity import assert_float_parity, bf16_to_f64

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available()
    gu.ensure_lib()
    assert gu.device_error() == 0


def _special_rows(k=128):
    g = np.random.default_rng(99)
    rows = [
        np.zeros(k),
        -np.zeros(k),
        g.standard_normal(k) * 1e-40,                       # subnormal fp32
        g.standard_normal(k) * 1e30,
        np.ldexp(1.0, g.integers(-130, 120, k)) * g.choice([-1, 1], k),
        np.nextafter(np.ldexp(1.0, g.integers(-20, 20, k)), 0) * g.choice([-1, 1], k),
        np.full(k, 3.4e38),
        g.standard_normal(k) * 0.02,
    ]
    return np.array(rows, dtype=np.float32)


def _check_quantize(w):
    codes, scales, status = gu.quantize(w)
    rc, rs, rst = oracle.mxfp4_quantize(w)
    assert np.array_equal(gu.host(scales), rs)
    assert np.array_equal(gu.host(codes), rc)
    assert int(gu.host(status)[0]) == rst
    return codes, scales


def test_quantize_worked_block_matches_hand_values():
    rows = []
    for line in open(os.path.join(GOLD, "mxfp4_worked_block.txt")):
        line = line.split("#", 1)[0].split()
        if line:
            rows.append(line)
    w = np.array([[float(r[0]) for r in rows[1:]]], np.float32)
    codes, scales, status = gu.quantize(w)
    c = gu.host(codes)[0]
    got = [(c[i // 2] >> (4 * (i % 2))) & 15 for i in range(32)]
    assert int(gu.host(scales)[0, 0]) == int(rows[0][1])
    assert got == [int(r[2]) for r in rows[1:]]


def test_quantize_random_ragged():
    g = synth.rng(90)
    _check_quantize(synth.normal_f32(g, (37, 96), 0.02))


def test_quantize_special_values():
    _check_quantize(_special_rows())


def test_quantize_nonfinite_blocks_flag_status():
    w = _special_rows(64)
    w[1, 3] = np.nan
    w[5, 40] = np.inf
    w[6, 63] = -np.inf
    codes, scales = _check_quantize(w)
    s = gu.host(scales)
    assert s[1, 0] == 255 and s[5, 1] == 255 and s[6, 1] == 255


def test_quantize_full_gate_up_layer():
    d = synth.gate_up_inputs(synth.GATE_UP.wid, 0, synth.GATE_UP.n, synth.GATE_UP.k)
    _check_quantize(d["wg"])
    _check_quantize(d["wu"])


def test_dequantize_bit_exact_all_codes_and_scales():
    g = synth.rng(91)
    n, k = 256, 64
    codes = synth.random_bytes(g, (n, k // 2))
    scales = g.integers(0, 256, size=(n, k // 32), dtype=np.uint8)
    scales[:, 0] = np.arange(n) % 256  # every scale byte, including 0 and 255
    out = gu.dev(np.zeros((n, k), np.float32))
    from bit_weight_only_mxfp4_gb300 import thinmx
    thinmx.tt_mxfp4_dequantize(gu.dev(codes), gu.dev(scales), n, k, out)
    got = gu.host(out)
    ref = oracle.mxfp4_dequantize(codes, scales)
    with np.errstate(over="ignore", invalid="ignore"):
        ref32 = ref.astype(np.float32)
    nan = np.isnan(ref32)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref32[~nan].view(np.uint32))


def _swiglu_case(n, k, m, postscale=True, wid=92, layer=0):
    d = synth.gate_up_inputs(wid, layer, n, k, m=m, postscale=postscale)
    gc, gs, st1 = gu.quantize(d["wg"])
    uc, us, st2 = gu.quantize(d["wu"])
    gp = None if d["pg"] is None else gu.dev(d["pg"])
    up = None if d["pu"] is None else gu.dev(d["pu"])
    packed = gu.pack_swiglu(gc, gs, gp, uc, us, up, n, k)
    h = gu.swiglu(packed, n, k, d["x"])
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), d["x"])
    return h, ref, packed, d


@pytest.mark.parametrize("n,k,m,post", [
    (37, 96, 1, True), (64, 32, 1, False), (129, 1024, 1, True), (300, 2880, 1, True),
    (50, 5120, 1, False), (33, 8192, 1, True), (21, 16384, 1, True),
    # m = 1 kernels with K fixed at compile time (2048, 5120), with K a
    # multiple of 1024 (no bounds tests: 3072, 4096) and the runtime-K kernel
    # at 6 chunks; rows spread over every CTA with ragged per-CTA counts
    (3001, 2048, 1, True), (517, 5120, 1, True), (200, 3072, 1, True), (150, 4096, 1, False),
    (61, 6144, 1, True),
    (77, 2048, 2, True), (77, 2048, 3, False),
    # m <= 8, k <= 5120: the mma.sync streaming kernel; 8-row tiles with
    # ragged ends, n below one tile, fewer 32-blocks than consumer warps
    (31, 1056, 5, True), (37, 2080, 4, True), (29, 1120, 8, False),
    (1, 2048, 1, True), (7, 64, 3, True), (9, 4096, 7, False), (17, 160, 1, True),
    (45, 5120, 4, True), (40, 2880, 8, True), (8, 5120, 6, True),
    # m = 4..8 with k > 5120: tcgen05 (k % 64 == 0) or CUDA-core FMA kernels
    (19, 6144, 6, False), (23, 5152, 5, True), (13, 6176, 2, True),
    # tcgen05 tensor-core path (m >= 9, k % 64 == 0); ragged row tiles
    (128, 128, 16, True), (130, 2048, 16, True), (300, 2880, 32, False), (256, 5120, 64, True),
    (77, 1024, 9, True), (129, 4096, 40, True), (1000, 768, 63, True),
    # wide K on tcgen05: the block-scale area takes most of shared memory,
    # so fewer raw k-tiles are in flight (three at m = 64, k = 16384)
    (70, 16384, 16, True), (130, 12288, 40, False), (33, 16384, 64, True),
])
def test_swiglu_matvec_shapes(n, k, m, post):
    h, ref, _, _ = _swiglu_case(n, k, m, post)
    assert h.shape == (m, n)
    assert_float_parity(h, ref, f"n={n} k={k} m={m}")
    assert gu.device_error() == 0


def test_swiglu_matvec_full_gate_up_layer_is_deterministic():
    c = synth.GATE_UP
    h, ref, packed, d = _swiglu_case(c.n, c.k, 1, True, wid=c.wid)
    rel, cos = assert_float_parity(h, ref, "gate/up 11008x2048")
    h2 = gu.swiglu(packed, c.n, c.k, d["x"])
    assert np.array_equal(h, h2)
    # most outputs equal the oracle's own bf16 rounding
    match = np.mean(h.ravel() == oracle.bf16_round_array(ref.ravel()))
    assert match > 0.99, match


def test_swiglu_identity_weights_give_silu_x_times_x():
    k = 64
    eye = np.eye(k, dtype=np.float32)
    gc, gs, _ = gu.quantize(eye)
    x = synth.normal_bf16(synth.rng(93), (2, k))
    packed = gu.pack_swiglu(gc, gs, None, gc, gs, None, k, k)
    h = gu.swiglu(packed, k, k, x)
    xf = bf16_to_f64(x)
    from scipy.special import expit
    assert_float_parity(h, xf * expit(xf) * xf, "identity")


def test_swiglu_large_activations_use_exact_prescale():
    # activations far outside the f16 range still give exact products
    n, k = 64, 256
    d = synth.gate_up_inputs(94, 0, n, k, m=1)
    x = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(d["x"]) * np.float32(2.0 ** 40))
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    assert_float_parity(h, ref, "x * 2^40")


def test_swiglu_full_batch_sweep_sampled_rows():
    """Phi-4-sized gate/up (k=5120, n=17920) at m = 1..8 in the launch
    configuration the benchmark times, checked on sampled rows."""
    import torch
    c = synth.SWEEP
    g = synth.rng(c.wid, 0, 50)
    wg = synth.normal_f32(synth.rng(c.wid, 0, 0), (c.n, c.k), synth.WEIGHT_STD)
    wu = synth.normal_f32(synth.rng(c.wid, 0, 1), (c.n, c.k), synth.WEIGHT_STD)
    pg = synth.uniform_f32(synth.rng(c.wid, 0, 3), (c.n,), 0.9, 1.1)
    pu = synth.uniform_f32(synth.rng(c.wid, 0, 4), (c.n,), 0.9, 1.1)
    gc, gs, _ = gu.quantize(wg)
    uc, us, _ = gu.quantize(wu)
    del wg, wu
    packed = gu.pack_swiglu(gc, gs, gu.dev(pg), uc, us, gu.dev(pu), c.n, c.k)
    rows = np.sort(g.choice(c.n, 192, replace=False))
    rows = np.unique(np.concatenate([rows, [0, c.n - 1]]))
    hgc, hgs, huc, hus = gu.host(gc), gu.host(gs), gu.host(uc), gu.host(us)
    for m in [1, 2, 4, 8, 16, 32, 64]:
        x = synth.normal_bf16(synth.rng(c.wid, 0, 2), (m, c.k))
        h = gu.swiglu(packed, c.n, c.k, x)
        ref = oracle.mxfp4_swiglu_matvec((hgc[rows], hgs[rows], pg[rows]),
                                         (huc[rows], hus[rows], pu[rows]), x)
        assert_float_parity(h[:, rows], ref, f"sweep m={m}")
    torch.cuda.empty_cache()


def test_tensor_path_rejects_k_not_multiple_of_64():
    import torch
    from bit_weight_only_mxfp4_gb300 import thinmx
    n, k = 64, 96
    packed = torch.zeros(thinmx.tt_mxfp4_swiglu_packed_bytes(n, k), dtype=torch.uint8, device="cuda")
    x = torch.zeros((16, k), dtype=torch.int16, device="cuda")
    h = torch.zeros((16, n), dtype=torch.int16, device="cuda")
    with pytest.raises(thinmx.ThinmxError) as e:
        thinmx.tt_mxfp4_swiglu_matvec(packed, n, k, x, 16, h)
    assert e.value.status == 5  # TT_ERR_UNSUPPORTED, nothing launched


@pytest.mark.parametrize("m", [9, 16, 64])
def test_tensor_path_serves_activations_beyond_f16_range(m):
    """The tensor path (m >= 9 with k % 64 == 0) converts x to f16 for the MMA
    after an exact power-of-two prescale taken from each x row's largest
    value over all of K: an activation beyond f16's range, in a late k-tile,
    is served exactly (no flag), row by row."""
    n, k = 128, 1024
    d = synth.gate_up_inputs(98, 0, n, k, m=m)
    x = d["x"].copy()
    x[min(3, m - 1), 900] = synth.f32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
    x[0, 17] = synth.f32_to_bf16_bits(np.array([-3.0e9], np.float32))[0]
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    assert gu.device_error() == 0
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    for i in range(m):
        assert_float_parity(h[i], ref[i], f"row {i}")


@pytest.mark.parametrize("m", [4, 16])
def test_outlier_activation_row(m):
    """A realistic hidden-state outlier: one activation 10^4 times its row's
    median magnitude, in the last k-tile of an otherwise quiet row, on the
    path m takes at the Phi-4 K (m = 4: mma.sync streaming kernel; m = 16:
    tcgen05)."""
    n, k = 96, 5120
    d = synth.gate_up_inputs(99, 0, n, k, m=m)
    xf = synth.bf16_bits_to_f32(d["x"]).copy()
    med = np.median(np.abs(xf[1]))
    xf[1, k - 5] = np.float32(1.0e4 * med)
    x = synth.f32_to_bf16_bits(xf)
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    assert gu.device_error() == 0
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    for i in range(m):
        assert_float_parity(h[i], ref[i], f"row {i}")


def test_tensor_path_small_activations_keep_precision():
    """The tensor path scales each x row by an exact power of two before the
    f16 conversion, so rows of tiny activations (which f16 alone would flush)
    match the oracle row by row, also where the first k-tile is far below
    the rest of the row."""
    n, k, m = 160, 1024, 16
    d = synth.gate_up_inputs(95, 0, n, k, m=m)
    xf = synth.bf16_bits_to_f32(d["x"]).copy()
    for i in range(m):
        xf[i] *= np.float32(2.0 ** (-3 * i))          # rows down to 2^-45
    xf[5, :64] *= np.float32(2.0 ** -12)               # first tile far below the rest
    xf[7] = 0.0                                         # an all-zero row
    x = synth.f32_to_bf16_bits(xf)
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    assert gu.device_error() == 0
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    for i in range(m):
        if i == 7:
            assert not np.any(bf16_to_f64(h[i]))
            continue
        assert_float_parity(h[i], ref[i], f"row {i} scaled by 2^-{3 * i}")


@pytest.mark.parametrize("k", [2048, 2880, 8192])
def test_swiglu_m1_blocks_of_very_different_magnitude(k):
    """The m = 1 kernel prescales each 32-block of x by its own power of two:
    blocks spread over 2^-60 .. 2^60 (and an all-zero block) still match the
    oracle, here with the output dominated by no single block."""
    n = 96
    d = synth.gate_up_inputs(96, 0, n, k, m=1)
    g = synth.rng(96, 1)
    nblk = k // 32
    e = g.integers(-60, 61, nblk)
    xf = synth.bf16_bits_to_f32(d["x"]).reshape(nblk, 32).copy()
    xf *= np.ldexp(np.float32(1.0), e).astype(np.float32)[:, None]
    xf[nblk // 2] = 0.0
    # weights scaled by the inverse so that every block contributes alike
    wg = (d["wg"].reshape(n, nblk, 32) * np.ldexp(np.float32(1.0), -e)[None, :, None]).reshape(n, k)
    wu = (d["wu"].reshape(n, nblk, 32) * np.ldexp(np.float32(1.0), -e)[None, :, None]).reshape(n, k)
    x = synth.f32_to_bf16_bits(xf.reshape(1, k))
    gc, gs, _ = gu.quantize(wg.astype(np.float32))
    uc, us, _ = gu.quantize(wu.astype(np.float32))
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    assert gu.device_error() == 0
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    assert_float_parity(h, ref, f"block magnitudes 2^-60..2^60, k={k}")


@pytest.mark.parametrize("k", [1056, 2048])
def test_small_batches_serve_large_activations(k):
    """m = 5 runs on the streaming kernels, whose prescale is taken from the
    data itself per 32-block: an activation of 1e5 is served exactly, with no
    flag."""
    n, m = 96, 5
    d = synth.gate_up_inputs(97, 0, n, k, m=m)
    x = d["x"].copy()
    x[3, 17] = synth.f32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    packed = gu.pack_swiglu(gc, gs, gu.dev(d["pg"]), uc, us, gu.dev(d["pu"]), n, k)
    h = gu.swiglu(packed, n, k, x)
    assert gu.device_error() == 0
    ref = oracle.mxfp4_swiglu_matvec((gu.host(gc), gu.host(gs), d["pg"]),
                                     (gu.host(uc), gu.host(us), d["pu"]), x)
    for i in range(m):
        assert_float_parity(h[i], ref[i], f"row {i}")


@pytest.mark.parametrize("n,k,post", [(5, 32, True), (37, 96, False), (64, 2048, True),
                                      (7, 2880, True), (3, 5152, False)])
def test_pack_swiglu_is_a_byte_rearrangement(n, k, post):
    """The packed gate/up buffer holds exactly the canonical bytes, moved:
    per output row r, one record [gate codes k/2][up codes k/2][gate scales
    k/32][up scales k/32][pad to 8][post_g f32][post_u f32][pad to 16], the
    records back to back (the layout the kernels read).  Every byte is
    compared, so a layout slip that cancels inside a dot product still
    fails here."""
    d = synth.gate_up_inputs(140, 0, n, k, m=1, postscale=post)
    gc, gs, _ = gu.quantize(d["wg"])
    uc, us, _ = gu.quantize(d["wu"])
    gp = None if d["pg"] is None else gu.dev(d["pg"])
    up = None if d["pu"] is None else gu.dev(d["pu"])
    packed = gu.host(gu.pack_swiglu(gc, gs, gp, uc, us, up, n, k))
    nblk = k // 32
    post_off = (k + 2 * nblk + 7) & ~7
    rec = (post_off + 8 + 15) & ~15
    assert packed.size == n * rec
    recs = packed.reshape(n, rec)
    assert np.array_equal(recs[:, :k // 2], gu.host(gc))
    assert np.array_equal(recs[:, k // 2:k], gu.host(uc))
    assert np.array_equal(recs[:, k:k + nblk], gu.host(gs))
    assert np.array_equal(recs[:, k + nblk:k + 2 * nblk], gu.host(us))
    ps = np.ascontiguousarray(recs[:, post_off:post_off + 8]).view(np.float32)
    want_g = d["pg"] if post else np.ones(n, np.float32)
    want_u = d["pu"] if post else np.ones(n, np.float32)
    assert np.array_equal(ps[:, 0].view(np.uint32), want_g.view(np.uint32))
    assert np.array_equal(ps[:, 1].view(np.uint32), want_u.view(np.uint32))
    assert not recs[:, k + 2 * nblk:post_off].any() and not recs[:, post_off + 8:].any()


@pytest.mark.parametrize("n,k", [(5, 32), (37, 96), (2880, 2880), (9, 5152)])
def test_pack_rows_is_a_byte_rearrangement(n, k):
    """The column-sliced single-matrix layout (the MoE down projections):
    for each 16-wide slice s of k, the 8 code bytes 8s..8s+7 of every row in
    row order, then for each 32-block b the E8M0 byte of every row; each
    part padded to 16 bytes."""
    import torch
    w = synth.normal_f32(synth.rng(141), (n, k), synth.WEIGHT_STD)
    codes, scales, _ = gu.quantize(w)
    nbytes = thinmx.tt_mxfp4_rows_packed_bytes(n, k)
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    thinmx.tt_mxfp4_pack_rows(codes, scales, n, k, packed, nbytes)
    p = gu.host(packed)
    c, s = gu.host(codes), gu.host(scales)
    cbytes = (n * (k // 2) + 15) // 16 * 16
    assert nbytes == cbytes + (n * (k // 32) + 15) // 16 * 16
    got_codes = p[:n * (k // 2)].reshape(k // 16, n, 8)
    assert np.array_equal(got_codes, c.reshape(n, k // 16, 8).transpose(1, 0, 2))
    got_scales = p[cbytes:cbytes + n * (k // 32)].reshape(k // 32, n)
    assert np.array_equal(got_scales, s.T)
