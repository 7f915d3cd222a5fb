"""Pins the CPU oracle to things other than itself (CPU only, no GPU).

Each test checks the oracle against a closed form, an invariant, a hand-derived value
from the documented layout, a special case that reduces to a library routine (numpy /
torch), or a value printed on the reference pages (tests/golden/page_sizes.json).  The
cases are chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from bit_quantized_linear_q8_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits_to_bf16_torch(vals):
    return torch.tensor(np.asarray(vals, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16(vals):
    return f32_bits_to_bf16_torch(vals)


# --------------------------------------------------------------------------- formats
def test_bf16_round_to_nearest_even_hand_values():
    assert O.f64_to_bf16(1.0) == 0x3F80
    assert O.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80           # tie -> even (down)
    assert O.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even (up)
    assert O.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # just above the tie
    assert O.f64_to_bf16(-2.5) == 0xC020
    assert O.f64_to_bf16(0.0) == 0x0000 and O.f64_to_bf16(-0.0) == 0x8000
    assert O.f64_to_bf16(3.5e38) == 0x7F80                    # overflow -> inf
    assert O.f64_to_bf16(2.0 ** -133) == 0x0001               # smallest subnormal


def test_bf16_rounding_matches_torch_conversion():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(3000) * np.exp2(rng.integers(-130, 120, 3000))).astype(np.float32)
    ours = O.f64_to_bf16(v.astype(np.float64))
    assert np.array_equal(ours, f32_bits_to_bf16_torch(v))


def test_f16_conversions_match_numpy():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(3000) * np.exp2(rng.integers(-28, 17, 3000))).astype(np.float32)
    ours = O.f64_to_f16(v.astype(np.float64))
    with np.errstate(over="ignore"):
        assert np.array_equal(ours, v.astype(np.float16).view(np.uint16))
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7C00) != 0x7C00
    back = O.f16_to_f32(bits[finite])
    assert np.array_equal(back.view(np.uint32), bits[finite].view(np.float16).astype(np.float32).view(np.uint32))


def test_page_printed_sizes():
    d = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    assert O.QK_K == d["QK_K"]["value"]
    assert O.Q4K_BLOCK_BYTES == d["Q4K_BLOCK_BYTES"]["value"]
    for n, k, b in d["q4k_weight_bytes"]["cases"]:
        assert O.q4k_bytes(n, k) == b
    for k, kp in d["quantize_act_q8_1_launch"]["kpad_cases"]:
        assert O.kpad(k) == kp
    # our q8_1 buffer (1 code byte + 8/32 bytes of (d, s) per padded value) fits the
    # scratch the page budgets for it
    for m, k, b in d["q8_1_scratch_bytes"]["cases"]:
        assert O.q8_1_bytes(m, k) <= b
        assert O.q8_1_bytes(m, k) == m * O.kpad(k) * 5 // 4


# --------------------------------------------------------------------------- Q2_0 layout
def test_q2_pack_hand_derived_bytes():
    k = 128
    scales = np.array([[0x3F80]], np.uint16)
    # codes[32i + l] = i  ->  every byte holds 0,1,2,3 in bit pairs 0,2,4,6 = 0b11100100
    codes = np.repeat(np.arange(4, dtype=np.uint8), 32)[None, :]
    p = O.q2_pack(codes, scales)
    assert np.all(p[:32] == 0xE4)
    assert p[32:].view(np.uint16)[0] == 0x3F80
    # codes[32i + l] = l % 4  ->  byte l = (l % 4) * 0b01010101
    codes = np.tile(np.arange(32, dtype=np.uint8) % 4, 4)[None, :]
    p = O.q2_pack(codes, scales)
    assert list(p[:8]) == [0x00, 0x55, 0xAA, 0xFF] * 2
    # a single 3 at column 77 = 32*2 + 13  ->  byte 13, bits 4..5
    codes = np.zeros((1, k), np.uint8)
    codes[0, 77] = 3
    p = O.q2_pack(codes, scales)
    expect = np.zeros(32, np.uint8)
    expect[13] = 0x30
    assert np.array_equal(p[:32], expect)
    # second pack block starts at byte 32
    codes = np.zeros((1, 256), np.uint8)
    codes[0, 128 + 32 * 3 + 0] = 1
    p = O.q2_pack(codes, np.array([[0x3F80, 0x4000]], np.uint16))
    assert p[32] == 0x40 and p[:32].sum() == 0 and p[33:64].sum() == 0
    assert list(p[64:].view(np.uint16)) == [0x3F80, 0x4000]


def test_q2_pack_unpack_round_trip():
    d = synth.small_q2(5, 7, 384, 1)
    p = O.q2_pack(d["codes"], d["scales"])
    assert p.size == O.q2_bytes(7, 384) == 7 * 384 // 4 + 7 * 3 * 2
    codes, sc = O.q2_unpack(p, 7, 384)
    assert np.array_equal(codes, d["codes"]) and np.array_equal(sc, d["scales"])
    # every byte value decodes and re-encodes to itself
    raw = np.arange(256, dtype=np.uint8)
    plane = raw.reshape(2, 128).copy()  # 2 rows x 512 codes = 2 x 128 bytes
    buf = np.concatenate([plane.ravel(), np.zeros(2 * 4 * 2, np.uint8)])
    codes, sc = O.q2_unpack(buf, 2, 512)
    again = O.q2_pack(codes, sc)
    assert np.array_equal(again[: 2 * 128], plane.ravel())


def test_q2_dequant_exact_values():
    d = synth.small_q2(6, 5, 256, 1)
    p = O.q2_pack(d["codes"], d["scales"])
    deq = O.q2_dequant_bf16(p, 5, 256)
    dsc = O.bf16_to_f32(d["scales"]).astype(np.float64)
    expect = np.repeat(dsc, 128, axis=1) * (d["codes"].astype(np.float64) - 2.0)
    assert np.array_equal(deq, f32_bits_to_bf16_torch(expect.astype(np.float32)))
    # code 2 gives +0 exactly, code 3 gives d, code 0 gives -2d
    zero = deq[d["codes"] == 2]
    assert np.all(zero == 0x0000)
    c3 = d["codes"] == 3
    assert np.array_equal(deq[c3], np.repeat(d["scales"], 128, axis=1)[c3])


def test_q2_dequant_group_256():
    d = synth.small_q2(7, 3, 512, 1, group=256)
    p = O.q2_pack(d["codes"], d["scales"], group=256)
    deq = O.bf16_to_f32(O.q2_dequant_bf16(p, 3, 512, 256)).astype(np.float64)
    dsc = O.bf16_to_f32(d["scales"]).astype(np.float64)
    assert np.array_equal(deq, np.repeat(dsc, 256, axis=1) * (d["codes"] - 2.0))


# --------------------------------------------------------------------------- GEMV
def _dq(d):
    dsc = O.bf16_to_f32(d["scales"]).astype(np.float64)
    return np.repeat(dsc, d["group"], axis=1) * (d["codes"].astype(np.float64) - 2.0)


@pytest.mark.parametrize("m", [1, 3, 8])
def test_q2_gemv_matches_numpy_matmul(m):
    d = synth.small_q2(10 + m, 37, 640, m)
    p = O.q2_pack(d["codes"], d["scales"])
    y = O.q2_gemv(d["x"], p, 37, 640)
    x = O.bf16_to_f32(d["x"]).astype(np.float64)
    ref = x @ _dq(d).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_q2_gemv_closed_forms():
    n, k = 9, 384
    d = synth.small_q2(20, n, k, 2)
    # all codes 2 -> every weight is 0 -> y == 0 exactly
    p = O.q2_pack(np.full((n, k), 2, np.uint8), d["scales"])
    assert np.all(O.q2_gemv(d["x"], p, n, k) == 0.0)
    # one-hot x picks one column of the dequantised weight, exactly
    p = O.q2_pack(d["codes"], d["scales"])
    x = np.zeros((1, k), np.uint16)
    x[0, 201] = 0x3F80
    y = O.q2_gemv(x, p, n, k)[0]
    assert np.array_equal(y, _dq(d)[:, 201])
    # codes all 3 and x = 1 -> y[r] = 128 * sum of the row's group scales
    p = O.q2_pack(np.full((n, k), 3, np.uint8), d["scales"])
    y = O.q2_gemv(np.full((1, k), 0x3F80, np.uint16), p, n, k)[0]
    assert np.array_equal(y, 128.0 * O.bf16_to_f32(d["scales"]).astype(np.float64).sum(axis=1))
    # x = -1 flips the sign
    y2 = O.q2_gemv(np.full((1, k), 0xBF80, np.uint16), p, n, k)[0]
    assert np.array_equal(y2, -y)


# --------------------------------------------------------------------------- dense BF16 GEMM
def test_gemm_bf16_hand_product():
    # a = [[1, 2, 3], [-1, 0.5, 4]], w = [[1, 0, -1], [2, 2, 2]] (all exact in BF16):
    # out = a @ w^T = [[1 - 3, 2 + 4 + 6], [-1 - 4, -2 + 1 + 8]] = [[-2, 12], [-5, 7]]
    a = bf16([[1, 2, 3], [-1, 0.5, 4]])
    w = bf16([[1, 0, -1], [2, 2, 2]])
    assert np.array_equal(O.gemm_bf16(a, w), np.array([[-2.0, 12.0], [-5.0, 7.0]]))


def test_gemm_bf16_identity_and_shape():
    g = np.random.default_rng(31)
    m, k = 5, 64
    a = bf16(g.standard_normal((m, k)))
    eye = bf16(np.eye(k))
    # w = I returns a exactly
    assert np.array_equal(O.gemm_bf16(a, eye), O.bf16_to_f32(a).astype(np.float64))
    # a non-square product against numpy's matmul of the same values: a transposed operand
    # or a swapped index would change the shape or the values
    n = 7
    w = bf16(g.standard_normal((n, k)))
    ref = O.bf16_to_f32(a).astype(np.float64) @ O.bf16_to_f32(w).astype(np.float64).T
    out = O.gemm_bf16(a, w)
    assert out.shape == (m, n)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- SiLU*mul and FFN
def test_silu_mul_matches_torch():
    rng = np.random.default_rng(3)
    g = bf16(rng.standard_normal(2000) * 4)
    u = bf16(rng.standard_normal(2000))
    h = O.silu_mul_bf16(g, u)
    gt = torch.tensor(O.bf16_to_f32(g), dtype=torch.float64)
    ut = torch.tensor(O.bf16_to_f32(u), dtype=torch.float64)
    ref = (torch.nn.functional.silu(gt) * ut).numpy()
    assert np.array_equal(h, O.f64_to_bf16(ref))
    # SiLU(0) = 0; SiLU(z) ~ z for large z; SiLU(z) ~ 0 for very negative z
    z = bf16([0.0, 30.0, -60.0])
    one = bf16([1.0, 1.0, 1.0])
    out = O.bf16_to_f32(O.silu_mul_bf16(z, one))
    assert out[0] == 0.0 and out[1] == 30.0 and abs(out[2]) < 1e-20


def test_ffn_chain_stages():
    hidden, inter, m = 256, 384, 3
    g0 = synth._gen(30)
    gate = synth.q2_codes_scales(g0, inter, hidden)
    up = synth.q2_codes_scales(g0, inter, hidden)
    down = synth.q2_codes_scales(g0, hidden, inter)
    x = synth.activations(g0, m, hidden)
    pg, pu, pd = (O.q2_pack(c, s) for c, s in (gate, up, down))
    g, u, h, y = O.ffn_q2(x, pg, pu, pd, hidden, inter)
    xf = O.bf16_to_f32(x).astype(np.float64)
    dq = lambda cs: np.repeat(O.bf16_to_f32(cs[1]).astype(np.float64), 128, axis=1) * (cs[0] - 2.0)
    assert np.array_equal(g, bf16((xf @ dq(gate).T).astype(np.float32)))
    assert np.array_equal(u, bf16((xf @ dq(up).T).astype(np.float32)))
    hf = O.bf16_to_f32(h).astype(np.float64)
    np.testing.assert_allclose(y, hf @ dq(down).T, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- q8_1
def _q8(x_bits):
    m, k = x_bits.shape
    buf = O.quantize_q8_1(x_bits)
    codes, ds = O.q8_1_views(buf, m, k)
    return buf, codes, ds


def test_q8_1_invariants():
    m, k = 3, 300
    x = synth.activations(synth._gen(40), m, k, outlier_frac=0.34)
    buf, codes, ds = _q8(x)
    kp = O.kpad(k)
    assert kp == 512 and buf.size == m * kp + m * (kp // 32) * 8
    xf = np.zeros((m, kp), np.float32)
    xf[:, :k] = O.bf16_to_f32(x)
    blocks = xf.reshape(m, kp // 32, 32)
    q = codes.reshape(m, kp // 32, 32).astype(np.int64)
    d, s = ds[..., 0], ds[..., 1]
    amax = np.abs(blocks).max(axis=2)
    # d = amax / 127 as one fp32 division
    assert np.array_equal(d, amax / np.float32(127))
    # s = d * sum(q) as one fp32 product -- the q8_1 invariant
    assert np.array_equal(s, d * q.sum(axis=2).astype(np.float32))
    assert np.abs(q).max() <= 127
    # the largest |x| of every nonzero block maps to +-127
    nz = amax > 0
    assert np.all(np.abs(q).max(axis=2)[nz] == 127)
    # reconstruction error at most half a step, plus the rounding of the fp32 quotient
    # x/d (|x/d| <= 127, so that rounding is below 127 * 2^-24 of a step)
    err = np.abs(blocks.astype(np.float64) - d[..., None].astype(np.float64) * q)
    assert np.all(err <= d[..., None].astype(np.float64) * (0.5 + 127 * 2.0 ** -24))
    # padding beyond k: zero codes, zero d and s
    assert np.all(codes[:, k:] == 0)
    assert np.all(ds[:, (k + 31) // 32:] == 0)


def test_q8_1_integer_rows_are_lossless():
    # integers in [-127, 127] with a +-127 in every block: d = 1, q = x, s = sum x
    rng = np.random.default_rng(4)
    m, k = 2, 512
    xi = rng.integers(-127, 128, size=(m, k))
    xi[:, ::32] = 127 * np.where(rng.random((m, k // 32)) < 0.5, 1, -1)
    buf, codes, ds = _q8(bf16(xi.astype(np.float32)))
    assert np.all(ds[..., 0] == 1.0)
    assert np.array_equal(codes.astype(np.int64), xi)
    assert np.array_equal(ds[..., 1], xi.reshape(m, -1, 32).sum(axis=2).astype(np.float32))


def test_q8_1_rounding_half_away_from_zero():
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 127.0                       # amax 127 -> d = 1 exactly
    x[0, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -3.25]
    _, codes, ds = _q8(bf16(x))
    assert ds[0, 0, 0] == 1.0
    assert list(codes[0, :9]) == [127, 3, -3, 1, -1, 2, -2, 127, -3]
    # all-zero row: every block is 0
    _, codes, ds = _q8(np.zeros((1, 64), np.uint16))
    assert np.all(codes == 0) and np.all(ds == 0)


# --------------------------------------------------------------------------- Q2 MMQ
def test_q2_mmq_exact_differential():
    # integer activations (q8_1 lossless) and power-of-two scales: every product and
    # sum is exact, so the MMQ result must equal an exact integer matmul
    rng = np.random.default_rng(5)
    m, n, k = 5, 11, 384
    xi = rng.integers(-127, 128, size=(m, k))
    xi[:, ::32] = 127
    codes = rng.integers(0, 4, size=(n, k)).astype(np.uint8)
    sexp = rng.integers(-8, -3, size=(n, k // 128))
    scales = bf16(np.exp2(sexp).astype(np.float32))
    p = O.q2_pack(codes, scales)
    act = O.quantize_q8_1(bf16(xi.astype(np.float32)))
    out = O.q2_mmq(act, p, m, n, k)
    wi = codes.astype(np.int64) - 2
    exact = np.zeros((m, n))
    for g in range(k // 128):
        part = xi[:, 128 * g:128 * (g + 1)] @ wi[:, 128 * g:128 * (g + 1)].T
        exact += part * np.exp2(sexp[:, g])[None, :]
    assert np.array_equal(out, exact)


def test_q2_mmq_matches_numpy_on_dequantised_operands():
    d = synth.small_q2(50, 19, 640, 6, outlier_frac=0.2)
    p = O.q2_pack(d["codes"], d["scales"])
    act = O.quantize_q8_1(d["x"])
    codes, ds = O.q8_1_views(act, 6, 640)
    xa = (codes[:, :640].astype(np.float64).reshape(6, 20, 32) * ds[:, :20, :1].astype(np.float64)).reshape(6, 640)
    ref = xa @ _dq(d).T
    out = O.q2_mmq(act, p, 6, 19, 640)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    sub = O.q2_mmq(act, p, 6, 19, 640, rows=np.array([4, 0]))
    assert np.array_equal(sub, out[[4, 0]])


# --------------------------------------------------------------------------- Q4_K
def test_q4k_scale_bytes_hand_derived():
    s = O.q4k_pack_scales(np.arange(1, 9), np.arange(10, 18))
    assert list(s) == [1, 2, 3, 4, 10, 11, 76, 77, 229, 246, 7, 24]
    s = O.q4k_pack_scales([0, 0, 0, 0, 63, 16, 32, 48], [0, 0, 0, 0, 63, 0, 17, 33])
    assert list(s) == [192, 64, 128, 192, 192, 0, 64, 128, 255, 0, 16, 16]


def test_q4k_scale_pack_round_trip_all_pairs():
    rng = np.random.default_rng(6)
    for j in range(8):
        for a in range(64):
            sc = rng.integers(0, 64, 8)
            mn = rng.integers(0, 64, 8)
            sc[j] = a
            mn[j] = np.arange(64)[(a * 7 + j) % 64]
            for b in (0, 63, (a * 7 + j) % 64):
                mn[j] = b
                s2, m2 = O.q4k_unpack_scales(O.q4k_pack_scales(sc, mn))
                assert np.array_equal(s2, sc) and np.array_equal(m2, mn)


def _hand_block(d_bits, dmin_bits, sc, mn, q):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[2:4] = np.array([dmin_bits], np.uint16).view(np.uint8)
    blk[4:16] = O.q4k_pack_scales(sc, mn)
    for c in range(4):
        for l in range(32):
            blk[16 + 32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return blk


def test_q4k_dequant_hand_block():
    sc = np.arange(1, 9)
    mn = np.arange(10, 18)
    q = np.arange(256) % 16
    blk = _hand_block(0x3C00, 0x3800, sc, mn, q)   # d = 1.0, dmin = 0.5
    w = O.dequant_q4k(blk, 1, 256)[0]
    j = np.arange(256) // 32
    assert np.array_equal(w, 1.0 * sc[j] * q - 0.5 * mn[j])
    assert O.q4k_bytes(1, 256) == blk.size == 144


def test_q4k_quantiser_zero_and_bound():
    w = np.zeros((2, 512), np.uint16)
    assert np.all(O.quantize_q4k(w) == 0)
    d = synth.small_dense(7, 6, 1024, 1)
    blocks = O.quantize_q4k(d["w"])
    assert blocks.size == O.q4k_bytes(6, 1024)
    deq = O.dequant_q4k(blocks, 6, 1024)
    x = O.bf16_to_f32(d["w"]).astype(np.float64)
    # per sub-block error bound: half a code step, plus the error of the stored min and
    # of the stored scale across the 15 steps
    xb = x.reshape(6, 4, 8, 32)
    eb = np.abs(xb - deq.reshape(6, 4, 8, 32))
    lo = np.minimum(xb.min(axis=3), 0.0)
    step_ideal = (xb.max(axis=3) - lo) / 15.0
    bl = blocks.reshape(6, 4, 144)
    dd = O.f16_to_f32(bl[..., 0:2].copy().view(np.uint16)[..., 0]).astype(np.float64)
    dm = O.f16_to_f32(bl[..., 2:4].copy().view(np.uint16)[..., 0]).astype(np.float64)
    for r in range(6):
        for b in range(4):
            sc, mn = O.q4k_unpack_scales(bl[r, b, 4:16])
            ds = dd[r, b] * sc
            bound = 0.5 * ds + 0.5 * dm[r, b] + 15 * np.abs(step_ideal[r, b] - ds) + 1e-7
            assert np.all(eb[r, b] <= bound[:, None])
    rel = np.sqrt(((x - deq) ** 2).mean()) / np.sqrt((x ** 2).mean())
    assert rel < 0.12


def test_q4k_mmq_matches_numpy():
    d = synth.small_dense(8, 13, 512, 5)
    blocks = O.quantize_q4k(d["w"])
    act = O.quantize_q8_1(d["x"])
    codes, ds = O.q8_1_views(act, 5, 512)
    xa = (codes.astype(np.float64).reshape(5, 16, 32) * ds[..., :1].astype(np.float64)).reshape(5, 512)
    ref = xa @ O.dequant_q4k(blocks, 13, 512).T
    out = O.q4k_mmq(act, blocks, 5, 13, 512)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # q = 0 everywhere -> w = -dmin * m_j
    blk = _hand_block(0x3C00, 0x3400, np.ones(8, int), np.arange(8), np.zeros(256, int))
    w = O.dequant_q4k(blk, 1, 256)[0]
    assert np.array_equal(w, -0.25 * (np.arange(256) // 32))


# ------------------------------------------------------------------------------ NVFP4
# The page (q4k_mmq.rs, `dequant_nvfp4_to_bf16`) names packed E2M1 values, E4M3 group scales
# and a per-tensor scale2; the values of the two element formats are fixed by the OCP
# microscaling (FP4 E2M1) and OCP 8-bit floating point (E4M3) specifications.
def test_e2m1_values_are_the_published_table():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [O.e2m1_value(c) for c in range(8)] == mags
    assert [O.e2m1_value(8 + c) for c in range(8)] == [-v for v in mags]
    assert np.signbit(O.e2m1_value(8))  # code 8 is -0


def test_e4m3_endpoints_and_order():
    assert O.e4m3_value(0x38) == 1.0
    assert O.e4m3_value(0x7E) == 448.0          # largest finite value (no infinities)
    assert O.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert O.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert O.e4m3_value(0x00) == 0.0
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))
    pos = [O.e4m3_value(b) for b in range(0x7F)]  # 0x00 .. 0x7E
    assert all(a < b for a, b in zip(pos, pos[1:]))  # strictly increasing with the byte
    assert [O.e4m3_value(0x80 | b) for b in range(1, 0x7F)] == [-v for v in pos[1:]]


def test_nvfp4_dequant_worked_examples():
    import torch
    # one row of 32 values: codes 0..15 twice (low nibble first), scales 2.0 (0x40) and
    # 1.875 (0x3F); scale2 = 1 + 2^-10, so every product has <= 17 significant bits and is
    # exact in fp32: torch's own fp32 -> BF16 rounding then gives the expected bits
    codes = np.concatenate([np.arange(16), np.arange(16)]).astype(np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8).reshape(1, 16)
    scales = np.array([[0x40, 0x3F]], np.uint8)
    s2 = np.float32(1 + 2.0 ** -10)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)
    e2m1 = np.concatenate([mags, -mags])
    want = np.concatenate([e2m1 * 2.0, e2m1 * 1.875]) * float(s2)
    ref = torch.tensor(want.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = O.dequant_nvfp4(packed, scales, float(s2), 1, 32)[0]
    assert np.array_equal(out, ref)
    # exact BF16 values survive unchanged; code 8 with any scale is -0
    out = O.dequant_nvfp4(packed, np.array([[0x38, 0x38]], np.uint8), 1.0, 1, 32)[0]
    assert out[8] == 0x8000 and out[1] == 0x3F00 and out[7] == 0x40C0  # -0, 0.5, 6.0
