"""GPU parity: every CUDA entry point against the CPU oracle on the same seeded inputs.

Bit-exact for packing, dequantisation, q8_1 and the Q4_K quantiser; within the
tolerance of tests/helpers.py for GEMV / FFN / MMQ outputs.  Small cases span several
tiles and ragged tails; the full-size workloads run in the launch configuration the
bench times.
"""
import numpy as np
import pytest

import oracle as O
from bit_quantized_linear_q8_gb300 import synth
from helpers import (bf16_dev_to_u16, check_bf16_vs_f64, tile_quadrant_rows, to_dev_u16_as_bf16, to_dev_u8, u8_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from bit_quantized_linear_q8_gb300 import build
    build.build()
    import bit_quantized_linear_q8_gb300 as B
    return B


def dev_q2(B, codes, scales, group=128):
    return B.q2_pack(to_dev_u8(codes), to_dev_u16_as_bf16(scales), group)


# ------------------------------------------------------------------------------ packing
@pytest.mark.parametrize("n,k,group", [(1, 128, 128), (37, 640, 128), (5, 1024, 256), (300, 5120, 128)])
def test_q2_pack_bitexact(B, n, k, group):
    d = synth.small_q2(100 + n, n, k, 1, group=group)
    w = dev_q2(B, d["codes"], d["scales"], group)
    assert np.array_equal(u8_dev(w.data), O.q2_pack(d["codes"], d["scales"], group))


def test_q2_pack_full_qkvz(B):
    d = synth.qkvz_gemv()
    w = dev_q2(B, d["codes"], d["scales"])
    assert np.array_equal(u8_dev(w.data), O.q2_pack(d["codes"], d["scales"]))


# ------------------------------------------------------------------------------ dequant
@pytest.mark.parametrize("n,k,group", [(3, 128, 128), (37, 640, 128), (9, 1024, 256), (1000, 5120, 128)])
def test_dequant_bitexact(B, n, k, group):
    d = synth.small_q2(200 + n, n, k, 1, group=group)
    p = O.q2_pack(d["codes"], d["scales"], group)
    w = dev_q2(B, d["codes"], d["scales"], group)
    out = bf16_dev_to_u16(B.dequant_q2_to_bf16(w))
    assert np.array_equal(out, O.q2_dequant_bf16(p, n, k, group))


def test_dequant_full_prefill_weight(B):
    d = synth.q2_prefill_weight()
    w = dev_q2(B, d["codes"], d["scales"])
    out = bf16_dev_to_u16(B.dequant_q2_to_bf16(w))
    ref = O.q2_dequant_bf16(O.q2_pack(d["codes"], d["scales"]), d["n"], d["k"])
    assert np.array_equal(out, ref)


# ------------------------------------------------------------------------------ q8_1
@pytest.mark.parametrize("m,k", [(1, 256), (3, 300), (5, 1000), (7, 5120), (2, 17408), (4, 8), (1030, 300),
                                 (1100, 1000)])
def test_q8_1_bitexact(B, m, k):
    x = synth.activations(synth._gen(300 + m + k), m, k, outlier_frac=0.3)
    out = u8_dev(B.quantize_act_q8_1(to_dev_u16_as_bf16(x)))
    assert np.array_equal(out, O.quantize_q8_1(x))


@pytest.mark.parametrize("m", [512, 2048, 4096])
def test_q8_1_full_prefill(B, m):
    x = synth.q2_prefill_x(m)
    out = u8_dev(B.quantize_act_q8_1(to_dev_u16_as_bf16(x)))
    assert np.array_equal(out, O.quantize_q8_1(x))


def test_q8_1_edge_values(B):
    x = np.zeros((2, 256), np.float32)
    x[0, 0] = 127.0
    x[0, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -3.25]
    x[1, 32:64] = 1e-30                    # tiny values, one block
    import torch
    xb = torch.tensor(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    out = u8_dev(B.quantize_act_q8_1(xb.cuda()))
    assert np.array_equal(out, O.quantize_q8_1(bits))


def test_q8_1_half_integer_boundaries(B):
    """Blocks whose values sit on, and one or two BF16 steps beside, the points where
    x / d is a half-integer (d = amax / 127): there the rounding of RN(x / d) decides the code,
    so the kernel's reciprocal path must hand these values to the exact division."""
    import torch
    rng = np.random.default_rng(77)
    m, k = 1024, 256
    amax = (rng.uniform(0.5, 2.0, m) * np.exp2(rng.integers(-60, 60, m))).astype(np.float32)
    amax_b = torch.tensor(amax).to(torch.bfloat16).to(torch.float32).numpy()
    x = np.zeros((m, k), np.float32)
    h = rng.integers(0, 127, size=(m, k)) + 0.5
    x[:] = (h * amax_b[:, None] / 127.0) * rng.choice([-1.0, 1.0], size=(m, k))
    xb = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    # one and two BF16 steps beside the half-integer points, in either direction
    step = rng.integers(-2, 3, size=(m, k)).astype(np.int32)
    xb = np.where(xb & 0x7FFF, (xb.astype(np.int32) + step) & 0xFFFF, xb).astype(np.uint16)
    amax_bits = torch.tensor(amax_b).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb[:, ::32] = amax_bits[:, None]  # every 32-value block holds its row's amax
    out = u8_dev(B.quantize_act_q8_1(to_dev_u16_as_bf16(xb)))
    assert np.array_equal(out, O.quantize_q8_1(xb))


def test_q8_1_block_scale_range(B):
    """Blocks whose maxima span the whole BF16 range, subnormals included (the quantiser takes
    d = RN(amax / 127) without a division for amax >= 2^-94 and by IEEE division below), with
    values on and beside the half-integer points of x / d, and a row of maxima only."""
    import torch
    rng = np.random.default_rng(94)
    m, k = 192, 512
    e = rng.integers(-133, 127, size=(m, k // 32))
    e[:8] = np.arange(-98, -90).reshape(8, 1)   # around the switch between the two forms
    amax = np.ldexp(rng.uniform(1.0, 2.0, size=(m, k // 32)), e).astype(np.float32)
    amax_b = torch.tensor(amax).to(torch.bfloat16).to(torch.float32).numpy()
    h = rng.integers(0, 127, size=(m, k)) + rng.choice([0.0, 0.5], size=(m, k))
    x = (h * np.repeat(amax_b, 32, axis=1) / 127.0) * rng.choice([-1.0, 1.0], size=(m, k))
    xb = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    step = rng.integers(-1, 2, size=(m, k)).astype(np.int32)
    xb = np.where(xb & 0x7FFF, (xb.astype(np.int32) + step) & 0xFFFF, xb).astype(np.uint16)
    ab = torch.tensor(amax_b).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb[:, ::32] = ab                            # each block holds its maximum
    xb[-1] = np.repeat(ab[-1], 32)              # a row of maxima only
    out = u8_dev(B.quantize_act_q8_1(to_dev_u16_as_bf16(xb)))
    assert np.array_equal(out, O.quantize_q8_1(xb))


def test_q8_1_after_gemv_on_one_stream(B):
    """The q8_1 launch may start while the kernel before it on the stream drains (programmatic
    dependent launch), and the decode GEMV lets its dependents start early; q8_1 must still read
    the GEMV's finished output.  Five GEMV -> q8_1 pairs back to back on one stream, with no
    synchronisation between them; each q8_1 result against the oracle's q8_1 of that GEMV
    output, bit for bit."""
    import torch
    n, k, m = 4096, 5120, 4     # the GEMV's output rows [m, 4096] are q8_1's input (4096 % 256 == 0)
    d = synth.small_q2(970, n, k, m)
    w = dev_q2(B, d["codes"], d["scales"])
    x = to_dev_u16_as_bf16(d["x"])
    ys, acts = [], []
    for i in range(5):
        xi = x if i == 0 else (x * (1.0 + 0.25 * i)).contiguous()
        y = B.q2_gemv_batchm(xi, w)
        ys.append(y)
        acts.append(B.quantize_act_q8_1(y))
    torch.cuda.synchronize()
    for y, a in zip(ys, acts):
        assert np.array_equal(u8_dev(a), O.quantize_q8_1(bf16_dev_to_u16(y)))


# ------------------------------------------------------------------------------ NVFP4 -> BF16
def _nvfp4(B, d, scale2=None):
    import torch
    s2 = d["scale2"] if scale2 is None else scale2
    out = B.dequant_nvfp4_to_bf16(torch.from_numpy(d["packed"]).cuda(), torch.from_numpy(d["scales"]).cuda(), s2,
                                  d["n"], d["k"])
    return bf16_dev_to_u16(out), O.dequant_nvfp4(d["packed"], d["scales"], s2, d["n"], d["k"])


@pytest.mark.parametrize("n,k", [(1, 16), (3, 32), (37, 320), (300, 5120)])
def test_nvfp4_dequant_bitexact(B, n, k):
    out, ref = _nvfp4(B, synth.nvfp4_weight(800 + n, n, k))
    assert np.array_equal(out, ref)


def test_nvfp4_dequant_edges(B):
    d = synth.nvfp4_weight(850, 6, 64)
    sc = d["scales"]
    sc[0] = [0x01, 0x02, 0x03, 0x07]            # E4M3 subnormal scales
    sc[1] = [0x00, 0x80, 0x08, 0x7E]            # +-0, the smallest normal, the largest value (448)
    sc[2] = [0xB8, 0xC0, 0xF0, 0xFE]            # negative scales
    d["packed"][3] = 0x88                        # every code -0
    for s2 in (d["scale2"], 3e-39, 1e-30, 1.0, 1e36):  # BF16 subnormal products (exact fp64 path) ... overflow to inf
        out, ref = _nvfp4(B, d, s2)
        assert np.array_equal(out, ref), s2


def test_nvfp4_dequant_every_code_and_scale(B):
    """Every (scale byte, code byte) pair, under scale2 values from the BF16 subnormal range
    to overflow: the kernel's per-group table (exponent adds of BF16(Q) and BF16(1.5 Q)) and
    its per-value fallback must both give the oracle's bits."""
    n, k = 256, 512  # row r: scale byte r for all 32 groups; every code byte once per row
    packed = np.tile(np.arange(256, dtype=np.uint8), (n, 1))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], k // 16, axis=1)
    d = dict(n=n, k=k, packed=packed, scales=scales, scale2=1.0)
    nan_rows = np.array([0x7F, 0xFF])  # E4M3 NaN scales: NaN outputs, bit pattern unspecified
    ok_rows = np.setdiff1d(np.arange(n), nan_rows)
    for s2 in (0.0021, -0.37, 1.0, 2.0 ** -120, 3e-39, 2.0 ** 118, 1e36):
        out, ref = _nvfp4(B, d, s2)
        bad = np.argwhere(out[ok_rows] != ref[ok_rows])
        assert bad.size == 0, "scale2 %g: %d differ, first (scale byte, value) %s: got %04x want %04x" % (
            s2, len(bad), (ok_rows[bad[0][0]], bad[0][1]), out[ok_rows][tuple(bad[0])], ref[ok_rows][tuple(bad[0])])
        assert np.all((out[nan_rows] & 0x7FFF) > 0x7F80)


def test_nvfp4_dequant_full(B):
    out, ref = _nvfp4(B, synth.nvfp4_ffn_weight())
    assert np.array_equal(out, ref)


# ------------------------------------------------------------------------------ SiLU * mul
def test_silu_mul_within_one_ulp(B):
    rng = np.random.default_rng(7)
    import torch
    g = torch.tensor(rng.standard_normal(100003) * 3, dtype=torch.float32).to(torch.bfloat16)
    u = torch.tensor(rng.standard_normal(100003), dtype=torch.float32).to(torch.bfloat16)
    gb, ub = g.view(torch.int16).numpy().view(np.uint16), u.view(torch.int16).numpy().view(np.uint16)
    ref = O.silu_mul_bf16(gb, ub)
    for n in (100003, 100000):  # scalar tail path and vector path
        out = bf16_dev_to_u16(B.silu_mul_bf16(g[:n].cuda(), u[:n].cuda()))
        diff = np.abs(out.astype(np.int32).view(np.int32) - ref[:n].astype(np.int32))
        # same sign: bit patterns of neighbouring BF16 values differ by 1
        assert diff.max() <= 1
        assert np.mean(diff == 0) > 0.99


# ------------------------------------------------------------------------------ GEMV
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("n,k,group", [(37, 640, 128), (16, 128, 128), (300, 1024, 256), (1100, 2048, 128),
                                       (48, 512, 128), (200, 1536, 256)])
def test_gemv_small(B, m, n, k, group):
    d = synth.small_q2(400 + n + m, n, k, m, group=group)
    w = dev_q2(B, d["codes"], d["scales"], group)
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(d["x"]), w))
    ref = O.q2_gemv(d["x"], O.q2_pack(d["codes"], d["scales"], group), n, k, group)
    check_bf16_vs_f64(y, ref, "gemv m=%d n=%d k=%d" % (m, n, k))


# Shapes with few row tiles and long rows: the FP16 kernel's 2048-column chunks where its
# activation table fits (one 3-D request per chunk; 2-D boxes and a ragged last chunk of 13
# blocks for k = 9856), else (k = 24576 at m = 8) the BF16 kernel with its cluster K split;
# the down projection [5120, 17408] is the full-size case.
@pytest.mark.parametrize("m", [1, 3, 8])
@pytest.mark.parametrize("n,k,group", [(300, 8192, 128), (37, 6144, 256), (40, 9856, 128), (100, 24576, 128),
                                       (5120, 17408, 128)])
def test_gemv_ksplit(B, m, n, k, group):
    d = synth.small_q2(900 + n + m, n, k, m, group=group)
    w = dev_q2(B, d["codes"], d["scales"], group)
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(d["x"]), w))
    ref = O.q2_gemv(d["x"], O.q2_pack(d["codes"], d["scales"], group), n, k, group)
    check_bf16_vs_f64(y, ref, "gemv ksplit m=%d n=%d k=%d" % (m, n, k))


def test_gemv_closed_forms(B):
    n, k = 40, 384
    d = synth.small_q2(450, n, k, 2)
    import torch
    # all codes 2 -> every weight is 0: the output is 0 within the bar (the kernel's
    # offset correction cancels to a residue of a few fp32 ulps of the partial sums)
    w = dev_q2(B, np.full((n, k), 2, np.uint8), d["scales"])
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(d["x"]), w))
    check_bf16_vs_f64(y, np.zeros((2, n)), "all-zero weight")
    # one-hot x -> a column of the dequantised weight, exactly
    w = dev_q2(B, d["codes"], d["scales"])
    x = np.zeros((1, k), np.uint16)
    x[0, 201] = 0x3F80
    y = bf16_dev_to_u16(B.q2_gemv(to_dev_u16_as_bf16(x), w))[0]
    deq = O.q2_dequant_bf16(O.q2_pack(d["codes"], d["scales"]), n, k)
    assert np.array_equal(y, deq[:, 201])


@pytest.mark.parametrize("m", [1, 4])
def test_gemv_exact_differential(B, m):
    # integer activations (|x| <= 127, exact in BF16) and power-of-two group scales: every
    # product and partial sum is an exact binary value, so the stored BF16 must be the
    # round-to-nearest-even of the exact product, bit for bit
    import torch
    rng = np.random.default_rng(20 + m)
    n, k = 300, 1024
    xi = rng.integers(-127, 128, size=(m, k))
    codes = rng.integers(0, 4, size=(n, k)).astype(np.uint8)
    sexp = rng.integers(-6, -1, size=(n, k // 128))
    scales = torch.tensor(np.exp2(sexp).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = torch.tensor(xi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w = dev_q2(B, codes, scales)
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(xb), w))
    exact = O.q2_gemv(xb, O.q2_pack(codes, scales), n, k)
    assert np.array_equal(y, O.f64_to_bf16(exact))


def test_gemv_m1_activation_range(B):
    """The one-row GEMV holds activations as 16-bit fixed point per row: rows with a wide
    dynamic range, a single tiny nonzero value, all zeros, and a negative maximum."""
    import torch
    n, k = 200, 1024
    d = synth.small_q2(470, n, k, 1)
    w = dev_q2(B, d["codes"], d["scales"])
    packed = O.q2_pack(d["codes"], d["scales"])
    rng = np.random.default_rng(3)
    cases = {
        "wide range": rng.standard_normal(k) * np.exp2(rng.integers(-30, 12, size=k)),
        "one tiny value": np.where(np.arange(k) == 77, 3e-30, 0.0),
        "zeros": np.zeros(k),
        "negative max": np.where(np.arange(k) == 5, -6.0e4, rng.standard_normal(k)),
        "large": rng.standard_normal(k) * 1e30,
    }
    for what, xv in cases.items():
        xb = torch.tensor(xv[None, :].astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        y = bf16_dev_to_u16(B.q2_gemv(to_dev_u16_as_bf16(xb), w))
        ref = O.q2_gemv(xb, packed, n, k)
        if what == "zeros":
            assert not np.any(y & 0x7FFF), what
        else:
            check_bf16_vs_f64(y, ref, "gemv m=1 " + what)


def test_gemv_q2_gemv_1024(B):
    d = synth.q2_gemv_1024()
    w = dev_q2(B, d["codes"], d["scales"])
    y = bf16_dev_to_u16(B.q2_gemv(to_dev_u16_as_bf16(d["x"]), w))
    ref = O.q2_gemv(d["x"], O.q2_pack(d["codes"], d["scales"]), d["n"], d["k"])
    check_bf16_vs_f64(y, ref, "q2_gemv_1024")


@pytest.mark.parametrize("m", [1, 4])
def test_gemv_qkvz_full(B, m):
    d = synth.qkvz_gemv()
    w = dev_q2(B, d["codes"], d["scales"])
    x = d["x"][:m]
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(x), w))
    ref = O.q2_gemv(x, O.q2_pack(d["codes"], d["scales"]), d["n"], d["k"])
    check_bf16_vs_f64(y, ref, "qkvz m=%d" % m)
    # the sequential [QKV | Z] output layout is plain row order
    assert y.shape == (m, d["n_qkv"] + d["n_z"])


def test_gemv_weight_descriptor_follows_the_tensor(B):
    """The binding keeps each weight's checked C descriptor between calls; replacing the
    weight's tensor or its shape fields must rebuild (and re-check) it."""
    import torch
    n, k, m = 64, 512, 2
    d1 = synth.small_q2(480, n, k, m)
    d2 = synth.small_q2(481, n, k, m)
    w = dev_q2(B, d1["codes"], d1["scales"])
    x = to_dev_u16_as_bf16(d1["x"])
    y1 = bf16_dev_to_u16(B.q2_gemv_batchm(x, w))
    check_bf16_vs_f64(y1, O.q2_gemv(d1["x"], O.q2_pack(d1["codes"], d1["scales"]), n, k), "first weight")
    w.data = dev_q2(B, d2["codes"], d2["scales"]).data          # another tensor, same shape
    y2 = bf16_dev_to_u16(B.q2_gemv_batchm(x, w))
    check_bf16_vs_f64(y2, O.q2_gemv(d1["x"], O.q2_pack(d2["codes"], d2["scales"]), n, k), "replaced weight")
    w.n = 2 * n                                                  # too few bytes for the new shape
    with pytest.raises(ValueError):
        B.q2_gemv_batchm(x, w)


def test_gemv_edge_shapes(B):
    import torch
    from bit_quantized_linear_q8_gb300 import Q2Weight
    # k = 0: the sum is empty, output zeros
    w = Q2Weight(torch.zeros(16, dtype=torch.uint8, device="cuda"), 8, 0)
    x = torch.zeros((2, 0), dtype=torch.bfloat16, device="cuda")
    y = torch.full((2, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    B.q2_gemv_batchm(x, w, out=y)
    assert torch.count_nonzero(y).item() == 0
    # n = 1 (one partial tile)
    d = synth.small_q2(460, 1, 256, 3)
    w = dev_q2(B, d["codes"], d["scales"])
    y = bf16_dev_to_u16(B.q2_gemv_batchm(to_dev_u16_as_bf16(d["x"]), w))
    check_bf16_vs_f64(y, O.q2_gemv(d["x"], O.q2_pack(d["codes"], d["scales"]), 1, 256), "n=1")


# ------------------------------------------------------------------------------ FFN chain
def _bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ffn_check(B, x, gate, up, down, hidden, inter):
    from helpers import ABS_TOL, REL_TOL, bf16_half_ulp
    wg, wu, wd = (dev_q2(B, c, s) for c, s in (gate, up, down))
    out, hdev, udev = B.ffn_q2_km(to_dev_u16_as_bf16(x), wg, wu, wd)
    pg, pu, pd = (O.q2_pack(c, s) for c, s in (gate, up, down))
    g_ref, u_ref, h_ref, y_ref = O.ffn_q2(x, pg, pu, pd, hidden, inter)
    g64 = O.q2_gemv(x, pg, inter, hidden)
    u64 = O.q2_gemv(x, pu, inter, hidden)
    # stage u (left in up_scratch) against the fp64 GEMV
    check_bf16_vs_f64(bf16_dev_to_u16(udev), u64, "ffn up")
    # stage h (left in gate_scratch) against SiLU(g)*u of the fp64 GEMVs, with the GEMV bar
    # on g and u carried through SiLU's derivative, plus h's own BF16 rounding
    h = _bits_to_f64(bf16_dev_to_u16(hdev))
    tol = lambda v: np.maximum(REL_TOL * np.abs(v), ABS_TOL) + bf16_half_ulp(v)
    sig = 1.0 / (1.0 + np.exp(-g64))
    silu = g64 * sig
    dsilu = sig * (1.0 + g64 * (1.0 - sig))
    h_exact = silu * u64
    bound = 1.25 * (np.abs(dsilu * u64) * tol(g64) + np.abs(silu) * tol(u64) + tol(g64) * tol(u64)) + \
        bf16_half_ulp(np.maximum(np.abs(h), np.abs(h_exact))) + 1e-12
    assert np.all(np.abs(h - h_exact) <= bound), "ffn h: %d outside" % int((np.abs(h - h_exact) > bound).sum())
    assert np.mean(bf16_dev_to_u16(hdev) == h_ref) > 0.95
    # output against the oracle chain's y; the bar is widened by the effect of the (rare)
    # one-step differences between the kernel's h and the oracle chain's h
    hr = _bits_to_f64(h_ref)
    wdq = np.abs(_bits_to_f64(O.q2_dequant_bf16(pd, hidden, inter)))
    y = _bits_to_f64(bf16_dev_to_u16(out))
    extra = np.abs(h - hr) @ wdq.T
    bound_y = np.maximum(REL_TOL * np.abs(y_ref), ABS_TOL) + extra + bf16_half_ulp(np.maximum(np.abs(y), np.abs(y_ref)))
    assert np.all(np.abs(y - y_ref) <= bound_y), "ffn out: %d outside" % int((np.abs(y - y_ref) > bound_y).sum())


@pytest.mark.parametrize("m", [1, 3])
def test_ffn_small(B, m):
    hidden, inter = 256, 640
    g0 = synth._gen(500)
    gate = synth.q2_codes_scales(g0, inter, hidden)
    up = synth.q2_codes_scales(g0, inter, hidden)
    down = synth.q2_codes_scales(g0, hidden, inter)
    x = synth.activations(g0, m, hidden)
    _ffn_check(B, x, gate, up, down, hidden, inter)


@pytest.mark.parametrize("m", [1, 2, 3, 8])
def test_ffn_decode_full(B, m):
    d = synth.ffn_q2_decode()
    _ffn_check(B, d["x"][:m], d["gate"], d["up"], d["down"], d["hidden"], d["inter"])


# ------------------------------------------------------------------------------ Q4_K quantiser
@pytest.mark.parametrize("n,k", [(1, 256), (13, 512), (64, 5120)])
def test_q4k_quantiser_bitexact(B, n, k):
    d = synth.small_dense(600 + n, n, k, 1)
    out = u8_dev(B.quantize_weight_q4k(to_dev_u16_as_bf16(d["w"])))
    assert np.array_equal(out, O.quantize_q4k(d["w"]))


def test_q4k_quantiser_full_down_proj(B):
    d = synth.q4k_ffn_prefill()
    w = d["w_down"]
    out = u8_dev(B.quantize_weight_q4k(to_dev_u16_as_bf16(w)))
    assert np.array_equal(out, O.quantize_q4k(w))


# ------------------------------------------------------------------------------ Q2 MMQ
def _mmq_q2(B, x_bits, codes, scales):
    w = dev_q2(B, codes, scales)
    act = B.quantize_act_q8_1(to_dev_u16_as_bf16(x_bits))
    return bf16_dev_to_u16(B.q2_mmq_gemm(act, w, x_bits.shape[0]))


@pytest.mark.parametrize("m,n,k", [(1, 8, 128), (5, 37, 640), (130, 300, 1024), (257, 129, 384), (64, 1000, 2048)])
def test_q2_mmq_small(B, m, n, k):
    d = synth.small_q2(700 + m + n, n, k, m, outlier_frac=0.05)
    y = _mmq_q2(B, d["x"], d["codes"], d["scales"])
    ref = O.q2_mmq(O.quantize_q8_1(d["x"]), O.q2_pack(d["codes"], d["scales"]), m, n, k)
    check_bf16_vs_f64(y, ref, "q2 mmq m=%d n=%d k=%d" % (m, n, k))


def test_q2_mmq_exact_differential(B):
    # integer activations with a +-127 in every 32-block (q8_1 is then lossless, d = 1) and
    # power-of-two scales: every partial sum is exact in fp32, so the stored BF16 must be
    # exactly the round-to-nearest of the exact product
    rng = np.random.default_rng(11)
    m, n, k = 70, 200, 512
    xi = rng.integers(-127, 128, size=(m, k))
    xi[:, ::32] = 127
    codes = rng.integers(0, 4, size=(n, k)).astype(np.uint8)
    sexp = rng.integers(-4, -1, size=(n, k // 128))
    import torch
    scales = torch.tensor(np.exp2(sexp).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb = torch.tensor(xi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = _mmq_q2(B, xb, codes, scales)
    exact = O.q2_mmq(O.quantize_q8_1(xb), O.q2_pack(codes, scales), m, n, k)
    assert np.array_equal(y, O.f64_to_bf16(exact))


@pytest.mark.parametrize("m", [512, 2048, 4096])
def test_q2_mmq_prefill_full(B, m):
    d = synth.q2_prefill_weight()
    x = synth.q2_prefill_x(m)
    w = dev_q2(B, d["codes"], d["scales"])
    act = B.quantize_act_q8_1(to_dev_u16_as_bf16(x))
    y = bf16_dev_to_u16(B.q2_mmq_gemm(act, w, m))
    act_ref = O.quantize_q8_1(x)
    assert np.array_equal(u8_dev(act), act_ref)
    packed = O.q2_pack(d["codes"], d["scales"])
    # every 128-row tile and every 32-row lane quadrant of it, plus the outlier rows
    amax = np.abs(O.bf16_to_f32(x)).max(axis=1)
    rows = tile_quadrant_rows(m, m, extra=np.argsort(-amax)[: max(1, m // 100)])
    ref = O.q2_mmq(act_ref, packed, m, d["n"], d["k"], rows=rows)
    check_bf16_vs_f64(y[rows], ref, "q2 mmq prefill m=%d" % m)


@pytest.mark.parametrize("m", [512, 2048])
def test_dequant_gemm_prefill_full(B, m):
    """The fallback route (dequantise to BF16, then the dense BF16 GEMM) against the fp64
    product of the BF16 activations and the dequantised weight, element by element on rows
    that hit every 128-row tile and lane quadrant."""
    d = synth.q2_prefill_weight()
    x = synth.q2_prefill_x(m)
    w = dev_q2(B, d["codes"], d["scales"])
    out, mode = B.q2_prefill_proj(to_dev_u16_as_bf16(x), w, mode="dequant")
    assert mode == "dequant"
    y = bf16_dev_to_u16(out)
    amax = np.abs(O.bf16_to_f32(x)).max(axis=1)
    rows = tile_quadrant_rows(m, 7 * m, extra=np.argsort(-amax)[: max(1, m // 100)])
    ref = O.q2_gemv(x[rows], O.q2_pack(d["codes"], d["scales"]), d["n"], d["k"])
    check_bf16_vs_f64(y[rows], ref, "dequant + gemm m=%d" % m)


# ------------------------------------------------------------------------------ dense BF16 GEMM
@pytest.mark.parametrize("m,n,k", [(1, 8, 64), (37, 300, 128), (128, 256, 64), (129, 257, 192), (300, 520, 1024),
                                   (256, 512, 5120)])
def test_dense_gemm_bf16_small(B, m, n, k):
    """Every output element against the oracle: ragged m and n tails, one and several K
    steps, several m and n tiles."""
    g = synth._gen(1300 + m + n + k)
    a = synth.activations(g, m, k)
    w = synth.dense_weight(g, n, k)
    y = bf16_dev_to_u16(B.dense_gemm_bf16(to_dev_u16_as_bf16(a), to_dev_u16_as_bf16(w)))
    check_bf16_vs_f64(y, O.gemm_bf16(a, w), "dense gemm m=%d n=%d k=%d" % (m, n, k))


@pytest.mark.parametrize("m,n,k", [(300, 20000, 128), (129, 39000, 64), (300, 19000, 128), (520, 36000, 64)])
def test_dense_gemm_bf16_persistent(B, m, n, k):
    """More output tiles than SMs, so every CTA (pair) walks several tiles through its
    tensor-memory accumulators, with ragged last m and n tiles; every element against the
    oracle.  (300, 20000) and (129, 39000) take the 256 x 256 pair tiles (three rounds, two
    accumulator buffers), (300, 19000) and (520, 36000) the 256 x 512 pair tiles (one and three
    rounds through the one 512-column accumulator; in the last tile of n = 19000 the second
    MMA's weight rows lie wholly past n)."""
    g = synth._gen(1400 + m + n + k)
    a = synth.activations(g, m, k)
    w = synth.dense_weight(g, n, k)
    y = bf16_dev_to_u16(B.dense_gemm_bf16(to_dev_u16_as_bf16(a), to_dev_u16_as_bf16(w)))
    check_bf16_vs_f64(y, O.gemm_bf16(a, w), "dense gemm m=%d n=%d k=%d" % (m, n, k))
    assert B.lib().bq_device_status() == 0


def test_dense_gemm_bf16_edges(B):
    import torch
    a = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    # k not a multiple of 64 is refused before any launch
    with pytest.raises(B.BQ8Error):
        B.dense_gemm_bf16(a[:, :48].contiguous(), w[:, :48].contiguous())
    # k = 0 writes zeros
    out = torch.full((4, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    B.dense_gemm_bf16(a[:, :0].contiguous(), w[:, :0].contiguous(), out=out)
    assert torch.count_nonzero(out).item() == 0
    assert B.lib().bq_device_status() == 0


# ------------------------------------------------------------------------------ Q4_K MMQ
@pytest.mark.parametrize("m,n,k", [(1, 8, 256), (5, 37, 512), (130, 300, 1024), (257, 129, 768), (64, 1000, 2048)])
def test_q4k_mmq_small(B, m, n, k):
    d = synth.small_dense(800 + m + n, n, k, m)
    wq = B.quantize_weight_q4k(to_dev_u16_as_bf16(d["w"]))
    act = B.quantize_act_q8_1(to_dev_u16_as_bf16(d["x"]))
    y = bf16_dev_to_u16(B.q4k_mmq_gemm(act, wq, m, n, k))
    ref = O.q4k_mmq(O.quantize_q8_1(d["x"]), O.quantize_q4k(d["w"]), m, n, k)
    check_bf16_vs_f64(y, ref, "q4k mmq m=%d n=%d k=%d" % (m, n, k))


def test_q4k_ffn_prefill_full(B):
    """The FFN prefill at m = 2048 (gate and up MMQ, SiLU*mul, q8_1 of h, down MMQ), stage
    by stage and element by element on rows that hit every 128-row tile and lane quadrant:
    gate and up against the oracle on the same q8_1 input; h against the oracle's SiLU*mul
    of the kernels' own g and u (within one BF16 step); the q8_1 of h bit for bit; and the
    chain's output against the oracle's down GEMM of the kernels' own h."""
    d = synth.q4k_ffn_prefill()
    m, hidden, inter = d["m"], d["hidden"], d["inter"]
    wq = {kk: B.quantize_weight_q4k(to_dev_u16_as_bf16(d[kk])) for kk in ("w_gate", "w_up", "w_down")}
    wq_ref = {kk: O.quantize_q4k(d[kk]) for kk in ("w_gate", "w_up", "w_down")}
    for kk in wq:
        assert np.array_equal(u8_dev(wq[kk]), wq_ref[kk]), kk
    a1 = B.quantize_act_q8_1(to_dev_u16_as_bf16(d["x"]))
    a1_ref = O.quantize_q8_1(d["x"])
    assert np.array_equal(u8_dev(a1), a1_ref)
    gt = B.q4k_mmq_gemm(a1, wq["w_gate"], m, inter, hidden)
    ut = B.q4k_mmq_gemm(a1, wq["w_up"], m, inter, hidden)
    h = B.silu_mul_bf16(gt, ut)
    a2 = B.quantize_act_q8_1(h)
    out = B.q4k_mmq_gemm(a2, wq["w_down"], m, hidden, inter)
    rows = tile_quadrant_rows(m, 5)
    g_ref = O.q4k_mmq(a1_ref, wq_ref["w_gate"], m, inter, hidden, rows=rows)
    u_ref = O.q4k_mmq(a1_ref, wq_ref["w_up"], m, inter, hidden, rows=rows)
    g_bits, u_bits = bf16_dev_to_u16(gt)[rows], bf16_dev_to_u16(ut)[rows]
    check_bf16_vs_f64(g_bits, g_ref, "q4k gate")
    check_bf16_vs_f64(u_bits, u_ref, "q4k up")
    h_bits = bf16_dev_to_u16(h)[rows]
    h_or = O.silu_mul_bf16(g_bits, u_bits)
    step = np.abs(h_bits.astype(np.int32) - h_or.astype(np.int32))
    assert step.max() <= 1 and np.mean(step == 0) > 0.99
    # q8_1 of the kernels' h, the rows picked out of the planar buffer
    a2_ref = O.quantize_q8_1(h_bits)
    c_dev, ds_dev = O.q8_1_views(u8_dev(a2), m, inter)
    c_ref, ds_ref = O.q8_1_views(a2_ref, len(rows), inter)
    assert np.array_equal(c_dev[rows], c_ref) and np.array_equal(ds_dev[rows], ds_ref)
    y_ref = O.q4k_mmq(a2_ref, wq_ref["w_down"], len(rows), hidden, inter)
    check_bf16_vs_f64(bf16_dev_to_u16(out)[rows], y_ref, "q4k chain out (down, k=17408)")
