"""ffn_q2_km_noalloc: the FFN decode chain for callers that cannot allocate device memory.

Some callers (a plugin that only receives its inputs and outputs, a runtime whose memory
pool owns the whole device, C code linked without an allocator) cannot hand ffn_q2_km its
two scratch buffers; ffn_q2_km_noalloc keeps them in a fixed array inside the library.
This checks, through the C ABI, that two calls in a row (different m and data, so the
second one runs over what the first left in the array) give exactly what ffn_q2_km gives
on the same inputs, also when the intermediates fill the whole array, and that a size
beyond the array is refused without a launch.

The file's name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

from bit_quantized_linear_q8_gb300 import synth
from helpers import bf16_dev_to_u16, to_dev_u16_as_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from bit_quantized_linear_q8_gb300 import build
    build.build()
    import bit_quantized_linear_q8_gb300 as B
    return B


def _weights(B, g0, hidden, inter):
    ws = []
    for n, k in ((inter, hidden), (inter, hidden), (hidden, inter)):
        codes, scales = synth.q2_codes_scales(g0, n, k)
        ws.append(B.q2_pack(to_dev_u8(codes), to_dev_u16_as_bf16(scales)))
    return ws


def _noalloc_c(B, x, gate, up, down, m):
    """ffn_q2_km_noalloc through the C ABI on the current stream; returns out [m, hidden]."""
    import torch
    from bit_quantized_linear_q8_gb300 import _abi
    L = _abi.lib()
    out = torch.full((m, gate.k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dg, du, dd = gate.desc(), up.desc(), down.desc()
    st = L.ffn_q2_km_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.byref(dg), ctypes.byref(du), ctypes.byref(dd),
                             ctypes.c_void_p(out.data_ptr()), m, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _abi.BQ_OK, L.bq_last_error()
    torch.cuda.synchronize()
    assert L.bq_device_status() == _abi.BQ_OK
    return out


def test_noalloc_matches_ffn_q2_km_twice(B):
    # the same three kernels run on the same inputs, so the outputs agree bit for bit;
    # two calls in a row (different m and data: the second runs over what the first left in
    # the array)
    hidden, inter = 640, 1152          # several row tiles per CTA and ragged group counts
    g0 = synth._gen(9100)
    gate, up, down = _weights(B, g0, hidden, inter)
    for call, m in enumerate((3, 8)):
        x = to_dev_u16_as_bf16(synth.activations(g0, m, hidden))
        ref, _, _ = B.ffn_q2_km(x, gate, up, down)
        out = _noalloc_c(B, x, gate, up, down, m)
        assert np.array_equal(bf16_dev_to_u16(out), bf16_dev_to_u16(ref)), "call %d (m=%d)" % (call, m)


def test_noalloc_fills_the_array(B):
    # m * inter equal to the array's capacity: both intermediates reach its last element
    # (the up buffer starts right after the gate buffer); then the Python wrapper
    hidden, m = 256, 8
    inter = 262144 // m
    g0 = synth._gen(9200)
    gate, up, down = _weights(B, g0, hidden, inter)
    x = to_dev_u16_as_bf16(synth.activations(g0, m, hidden))
    ref, _, _ = B.ffn_q2_km(x, gate, up, down)
    out = _noalloc_c(B, x, gate, up, down, m)
    assert np.array_equal(bf16_dev_to_u16(out), bf16_dev_to_u16(ref))
    out2 = B.ffn_q2_km_noalloc(x[:1].contiguous(), gate, up, down)
    ref2, _, _ = B.ffn_q2_km(x[:1].contiguous(), gate, up, down)
    assert np.array_equal(bf16_dev_to_u16(out2), bf16_dev_to_u16(ref2))


def test_noalloc_rejects_oversize(B):
    from bit_quantized_linear_q8_gb300 import _abi
    L = _abi.lib()
    W = _abi.Q2WeightDesc
    inter, hidden = 65536, 256          # 8 * 65536 > 262144 values per intermediate
    gate, up, down = W(0x1000, inter, hidden, 128), W(0x1000, inter, hidden, 128), W(0x1000, hidden, inter, 128)
    null = ctypes.c_void_p(0)
    st = L.ffn_q2_km_noalloc(ctypes.c_void_p(0x2000), ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down),
                             ctypes.c_void_p(0x3000), 8, null)
    assert st == _abi.BQ_ERR_INVALID
    assert b"exceeds the built-in scratch" in L.bq_last_error()
