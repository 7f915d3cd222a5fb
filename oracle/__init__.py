"""CPU oracle for the quantized-weight linear projection.

TEST INFRASTRUCTURE ONLY: the tests, the package's ``smoke()`` check and the bench's
CPU-baseline leg may import this module; the product library never does.  It wraps the
plain C oracle in ``bq8_oracle.c`` (fp64 sums, fp32 decisions where a format fixes them)
and shares no code with the CUDA path.

All arrays are numpy; BF16 and FP16 values travel as their ``uint16`` bit patterns.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  bf16/fp16 rounding   -- pinned against numpy/torch conversions and hand values
  q2_pack / q2_unpack  -- pinned by a hand-derived byte pattern and round trips
  q2_dequant_bf16      -- pinned by the four code values and numpy products
  q2_gemv / q2_mmq     -- pinned by closed forms and numpy matmul of the operands
  gemm_bf16            -- pinned by a hand-computed product, the identity, numpy matmul
  silu_mul_bf16        -- pinned against torch's SiLU in float64
  quantize_q8_1        -- pinned by invariants (s = d*sum q), exact integer rows, ties
  quantize_q4k         -- pinned by the error bound, zero blocks, and layout round trips
  dequant_q4k / q4k_mmq-- pinned by hand-built blocks and numpy matmul
"""
import ctypes
import os

import numpy as np

from . import build as _build

QK_K = 256
Q4K_BLOCK_BYTES = 144
Q2_PACK = 128
Q8_BLOCK = 32

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        sig = {
            "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_f64_to_f16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_kpad": (I, [I]),
            "orc_q2_bytes": (I, [I, I, I]),
            "orc_q8_1_bytes": (I, [I, I]),
            "orc_q4k_bytes": (I, [I, I]),
            "orc_q2_pack": (None, [P, P, I, I, I, P]),
            "orc_q2_unpack": (None, [P, I, I, I, P, P]),
            "orc_q2_dequant_bf16": (None, [P, I, I, I, P]),
            "orc_q2_gemv": (None, [P, P, I, I, I, I, P]),
            "orc_gemm_bf16": (None, [P, P, I, I, I, P]),
            "orc_silu_mul_bf16": (None, [P, P, I, P]),
            "orc_ffn_q2": (None, [P, P, P, P, I, I, I, I, P, P, P, P]),
            "orc_quantize_q8_1": (None, [P, I, I, P]),
            "orc_q2_mmq": (None, [P, P, I, I, I, I, P, I, P]),
            "orc_q4k_pack_scales": (None, [P, P, P]),
            "orc_q4k_unpack_scales": (None, [P, P, P]),
            "orc_quantize_q4k": (None, [P, I, I, P]),
            "orc_dequant_q4k": (None, [P, I, I, P]),
            "orc_q4k_mmq": (None, [P, P, I, I, I, P, I, P]),
            "orc_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_dequant_nvfp4": (None, [P, P, ctypes.c_float, I, I, P]),
            "orc_num_threads": (ctypes.c_int, []),
            "orc_set_num_threads": (None, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_num_threads(n: int) -> None:
    """Threads used by the oracle's parallel loops from now on."""
    lib().orc_set_num_threads(int(n))


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ---------------------------------------------------------------- number formats
def bf16_to_f32(bits):
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(v):
    v = np.asarray(v, dtype=np.float64)
    f = lib().orc_f64_to_bf16
    return np.array([f(float(t)) for t in v.ravel()], dtype=np.uint16).reshape(v.shape)


def f64_to_f16(v):
    v = np.asarray(v, dtype=np.float64)
    f = lib().orc_f64_to_f16
    return np.array([f(float(t)) for t in v.ravel()], dtype=np.uint16).reshape(v.shape)


def f16_to_f32(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    f = lib().orc_f16_to_f32
    return np.array([f(int(t)) for t in bits.ravel()], dtype=np.float32).reshape(bits.shape)


# ---------------------------------------------------------------- sizes
def kpad(k: int) -> int:
    return int(lib().orc_kpad(k))


def q2_bytes(n: int, k: int, group: int = 128) -> int:
    return int(lib().orc_q2_bytes(n, k, group))


def q8_1_bytes(m: int, k: int) -> int:
    return int(lib().orc_q8_1_bytes(m, k))


def q4k_bytes(n: int, k: int) -> int:
    return int(lib().orc_q4k_bytes(n, k))


# ---------------------------------------------------------------- Q2_0
def q2_pack(codes, scales_bits, group: int = 128):
    codes = _c(codes, np.uint8)
    n, k = codes.shape
    sc = _c(scales_bits, np.uint16)
    assert sc.shape == (n, k // group)
    out = np.zeros(q2_bytes(n, k, group), dtype=np.uint8)
    lib().orc_q2_pack(_p(codes), _p(sc), n, k, group, _p(out))
    return out


def q2_unpack(packed, n: int, k: int, group: int = 128):
    packed = _c(packed, np.uint8)
    codes = np.zeros((n, k), dtype=np.uint8)
    sc = np.zeros((n, k // group), dtype=np.uint16)
    lib().orc_q2_unpack(_p(packed), n, k, group, _p(codes), _p(sc))
    return codes, sc


def q2_dequant_bf16(packed, n: int, k: int, group: int = 128):
    packed = _c(packed, np.uint8)
    out = np.zeros((n, k), dtype=np.uint16)
    lib().orc_q2_dequant_bf16(_p(packed), n, k, group, _p(out))
    return out


def q2_gemv(x_bits, packed, n: int, k: int, group: int = 128):
    x = _c(x_bits, np.uint16)
    m = x.shape[0]
    assert x.shape == (m, k)
    packed = _c(packed, np.uint8)
    y = np.zeros((m, n), dtype=np.float64)
    lib().orc_q2_gemv(_p(x), _p(packed), m, n, k, group, _p(y))
    return y


def gemm_bf16(a_bits, w_bits):
    """Dense BF16 GEMM of the fallback prefill route (init_q2.rs `qkvz_q2_prefill_gemm`,
    `dense_gemm_bf16_pipelined`): out [m, n] = a [m, k] @ w [n, k]^T of the BF16 values,
    summed in fp64 (the store's BF16 rounding is left to the caller)."""
    a = _c(a_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    m, k = a.shape
    n = w.shape[0]
    assert w.shape == (n, k)
    out = np.zeros((m, n), dtype=np.float64)
    lib().orc_gemm_bf16(_p(a), _p(w), m, n, k, _p(out))
    return out


def silu_mul_bf16(gate_bits, up_bits):
    g = _c(gate_bits, np.uint16)
    u = _c(up_bits, np.uint16)
    assert g.shape == u.shape
    out = np.zeros(g.shape, dtype=np.uint16)
    lib().orc_silu_mul_bf16(_p(g), _p(u), g.size, _p(out))
    return out


def ffn_q2(x_bits, gate, up, down, hidden: int, inter: int, group: int = 128):
    """Returns (g, u, h) as BF16 bits [m, inter] and y as fp64 [m, hidden]."""
    x = _c(x_bits, np.uint16)
    m = x.shape[0]
    g = np.zeros((m, inter), dtype=np.uint16)
    u = np.zeros((m, inter), dtype=np.uint16)
    h = np.zeros((m, inter), dtype=np.uint16)
    y = np.zeros((m, hidden), dtype=np.float64)
    lib().orc_ffn_q2(_p(x), _p(_c(gate, np.uint8)), _p(_c(up, np.uint8)), _p(_c(down, np.uint8)),
                     m, hidden, inter, group, _p(g), _p(u), _p(h), _p(y))
    return g, u, h, y


# ---------------------------------------------------------------- q8_1
def quantize_q8_1(x_bits):
    """Returns the q8_1 buffer (uint8) plus views (codes int8 [m, kp], ds float32 [m, kp/32, 2])."""
    x = _c(x_bits, np.uint16)
    m, k = x.shape
    out = np.zeros(q8_1_bytes(m, k), dtype=np.uint8)
    lib().orc_quantize_q8_1(_p(x), m, k, _p(out))
    return out


def q8_1_views(buf, m: int, k: int):
    kp = kpad(k)
    codes = buf[: m * kp].view(np.int8).reshape(m, kp)
    ds = buf[m * kp: m * kp + m * (kp // 32) * 8].view(np.float32).reshape(m, kp // 32, 2)
    return codes, ds


def q2_mmq(act, packed, m: int, n: int, k: int, group: int = 128, rows=None):
    act = _c(act, np.uint8)
    packed = _c(packed, np.uint8)
    rows = np.arange(m, dtype=np.int64) if rows is None else _c(rows, np.int64)
    out = np.zeros((rows.size, n), dtype=np.float64)
    lib().orc_q2_mmq(_p(act), _p(packed), m, n, k, group, _p(rows), rows.size, _p(out))
    return out


# ---------------------------------------------------------------- Q4_K
def q4k_pack_scales(sc, mn):
    sc = _c(sc, np.int32)
    mn = _c(mn, np.int32)
    out = np.zeros(12, dtype=np.uint8)
    lib().orc_q4k_pack_scales(_p(sc), _p(mn), _p(out))
    return out


def q4k_unpack_scales(s12):
    s12 = _c(s12, np.uint8)
    sc = np.zeros(8, dtype=np.int32)
    mn = np.zeros(8, dtype=np.int32)
    lib().orc_q4k_unpack_scales(_p(s12), _p(sc), _p(mn))
    return sc, mn


def quantize_q4k(w_bits):
    w = _c(w_bits, np.uint16)
    n, k = w.shape
    assert k % QK_K == 0
    out = np.zeros(q4k_bytes(n, k), dtype=np.uint8)
    lib().orc_quantize_q4k(_p(w), n, k, _p(out))
    return out


def dequant_q4k(blocks, n: int, k: int):
    blocks = _c(blocks, np.uint8)
    out = np.zeros((n, k), dtype=np.float64)
    lib().orc_dequant_q4k(_p(blocks), n, k, _p(out))
    return out


def q4k_mmq(act, blocks, m: int, n: int, k: int, rows=None):
    act = _c(act, np.uint8)
    blocks = _c(blocks, np.uint8)
    rows = np.arange(m, dtype=np.int64) if rows is None else _c(rows, np.int64)
    out = np.zeros((rows.size, n), dtype=np.float64)
    lib().orc_q4k_mmq(_p(act), _p(blocks), m, n, k, _p(rows), rows.size, _p(out))
    return out


def e2m1_value(code: int) -> float:
    """FP4 E2M1 code (0..15) -> its real value (OCP microscaling formats)."""
    return lib().orc_e2m1_value(int(code))


def e4m3_value(b: int) -> float:
    """FP8 E4M3 byte -> its real value (OCP 8-bit floating point; 0x7F / 0xFF are NaN)."""
    return lib().orc_e4m3_value(int(b))


def dequant_nvfp4(packed, scales, scale2: float, n: int, k: int):
    """NVFP4 [n, k] (packed E2M1 [n][k/2], E4M3 scales [n][k/16], fp32 scale2) -> BF16 bits,
    the exact product rounded once (q4k_mmq.rs, `dequant_nvfp4_to_bf16`)."""
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    out = np.zeros((n, k), dtype=np.uint16)
    lib().orc_dequant_nvfp4(_p(packed), _p(scales), ctypes.c_float(scale2), n, k, _p(out))
    return out
