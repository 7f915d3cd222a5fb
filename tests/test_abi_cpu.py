"""The C ABI library builds, loads and exports every entry point of include/bq8.h, and its
host-side argument checks answer with the documented status codes -- all without a GPU
(none of these calls launches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bq8.h")


@pytest.fixture(scope="module")
def L():
    from bit_quantized_linear_q8_gb300 import build, _abi
    build.build()
    return _abi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ["quantize_act_q8_1", "q2_gemv", "q2_gemv_batchm", "ffn_q2_km", "q2_mmq_gemm", "q4k_mmq_gemm",
              "dequant_q2_to_bf16", "silu_mul_bf16", "bq_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from bit_quantized_linear_q8_gb300 import _abi
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in _abi.SIGNATURES, name


def test_size_helpers(L):
    assert L.bq_q2_weight_bytes(16384, 5120, 128) == 16384 * 5120 // 4 + 16384 * 40 * 2 == 22282240
    assert L.bq_q2_weight_bytes(1024, 1024, 128) == 278528
    assert L.bq_q2_weight_bytes(4, 100, 128) == 0          # k not a multiple of the group
    assert L.bq_q8_1_bytes(2048, 5120) == 2048 * 5120 * 5 // 4
    assert L.bq_q8_1_bytes(3, 300) == 3 * 512 * 5 // 4
    assert L.bq_q4k_weight_bytes(17408, 5120) == 50135040
    assert L.bq_q4k_weight_bytes(5, 300) == 0


def test_status_codes_without_launch(L):
    from bit_quantized_linear_q8_gb300 import _abi
    null = ctypes.c_void_p(0)
    W = _abi.Q2WeightDesc
    # invalid group / k
    w = W(0x1000, 64, 100, 128)
    assert L.q2_gemv_batchm(null, ctypes.byref(w), null, 1, null) == _abi.BQ_ERR_INVALID
    assert b"multiple of 128" in L.bq_last_error()
    w = W(0x1000, 64, 256, 96)
    assert L.dequant_q2_to_bf16(ctypes.byref(w), null, null) == _abi.BQ_ERR_INVALID
    # m out of range for the batched GEMV
    w = W(0x1000, 64, 256, 128)
    assert L.q2_gemv_batchm(ctypes.c_void_p(0x2000), ctypes.byref(w), ctypes.c_void_p(0x3000), 9, null) == 1
    # misaligned pointers
    assert L.q2_gemv_batchm(ctypes.c_void_p(0x2004), ctypes.byref(w), ctypes.c_void_p(0x3000), 2, null) == 1
    assert b"aligned" in L.bq_last_error()
    # NULL weight data / descriptor
    w0 = W(0, 64, 256, 128)
    assert L.q2_gemv(ctypes.c_void_p(0x2000), ctypes.byref(w0), ctypes.c_void_p(0x3000), null) == 1
    assert L.q2_gemv(ctypes.c_void_p(0x2000), None, ctypes.c_void_p(0x3000), null) == 1
    # empty work is a successful no-op
    assert L.q2_gemv_batchm(null, ctypes.byref(w), null, 0, null) == _abi.BQ_OK
    assert L.quantize_act_q8_1(null, null, 0, 128, null) == _abi.BQ_OK
    assert L.silu_mul_bf16(null, null, null, 0, null) == _abi.BQ_OK
    # Q4_K needs k % 256 == 0
    assert L.quantize_weight_q4k(ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), 4, 300, null) == 1
    # FFN shape mismatch
    g = W(0x1000, 512, 256, 128)
    u = W(0x1000, 512, 256, 128)
    d = W(0x1000, 256, 384, 128)
    p = ctypes.c_void_p(0x4000)
    assert L.ffn_q2_km(p, ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), p, p, p, 2, null) == 1
    # FFN scratch buffers that overlap: the up projection's epilogue reads the gate buffer
    # while it writes the up buffer, so they must be disjoint ([2][512] BF16 = 2048 bytes each)
    d = W(0x1000, 256, 512, 128)
    gs, us, out = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10000 + 1024), ctypes.c_void_p(0x20000)
    assert L.ffn_q2_km(p, ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), gs, us, out, 2, null) == 1
    assert b"overlap" in L.bq_last_error()
    assert L.ffn_q2_km(p, ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), gs, gs, out, 2, null) == 1
    # MMQ argument checks: Q2 needs group 128, Q4_K needs k % 256 == 0
    w256 = W(0x1000, 64, 512, 256)
    assert L.q2_mmq_gemm(ctypes.c_void_p(0x2000), ctypes.byref(w256), ctypes.c_void_p(0x3000), 4, null) == 1
    assert b"group size 128" in L.bq_last_error()
    assert L.q4k_mmq_gemm(ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000), 4, 8, 300,
                          null) == 1
    assert b"multiple of 256" in L.bq_last_error()
    # NVFP4 dequant: k % 16 == 0, 16-byte aligned codes and output; empty work is a no-op
    a, b, c = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000)
    assert L.dequant_nvfp4_to_bf16(a, b, c, ctypes.c_float(1.0), 4, 40, null) == 1
    assert b"multiple of 16" in L.bq_last_error()
    assert L.dequant_nvfp4_to_bf16(ctypes.c_void_p(0x2008), b, c, ctypes.c_float(1.0), 4, 64, null) == 1
    assert L.dequant_nvfp4_to_bf16(null, b, c, ctypes.c_float(1.0), 4, 64, null) == 1
    assert L.dequant_nvfp4_to_bf16(null, null, null, ctypes.c_float(1.0), 0, 64, null) == _abi.BQ_OK


def test_python_binding_refuses_cpu_tensors(L):
    import torch
    import bit_quantized_linear_q8_gb300 as B
    x = torch.zeros((1, 256), dtype=torch.bfloat16)
    w = B.Q2Weight(torch.zeros(64, dtype=torch.uint8), 1, 256)
    with pytest.raises(ValueError):
        B.q2_gemv(x, w)
