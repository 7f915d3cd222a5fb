"""GB300 (sm_103a) quantized-weight linear projection.

Python binding of libbq8's C ABI (``include/bq8.h``).  Each function here only marshals
torch tensors into device pointers, sizes and the current CUDA stream, calls the C entry
point of the same name and raises on a nonzero status; every step of the computation runs
in the library's CUDA kernels.  PyTorch is used for device memory and streams only.

The projection contract is ``out[m, n] = input[m, k] @ W^T`` (the serving stack's
init_q2.rs `qkvz_q2_prefill_gemm`, q4k_mmq.rs `q4k_mmq_gemm`).  BF16 tensors are
``torch.bfloat16``; packed weights and q8_1 buffers are ``torch.uint8``.
"""
import ctypes
import functools
from dataclasses import dataclass

from . import _abi
from ._abi import BQ8Error, LibraryNotBuilt, check, lib  # noqa: F401

__all__ = [
    "Q2Weight", "q2_pack", "quantize_weight_q4k", "quantize_act_q8_1", "q2_gemv", "q2_gemv_batchm",
    "silu_mul_bf16", "ffn_q2_km", "ffn_q2_km_noalloc", "q2_mmq_gemm", "q4k_mmq_gemm", "dequant_q2_to_bf16",
    "dense_gemm_bf16", "dequant_nvfp4_to_bf16", "q2_prefill_proj",
    "q2_weight_bytes", "q8_1_bytes", "q4k_weight_bytes", "BQ8Error", "LibraryNotBuilt",
]


def _torch():
    import torch
    return torch


def _ptr(t):
    # the C signatures declare void*, so ctypes converts the int (None is NULL)
    return t.data_ptr() if t is not None else None


_raw_stream = None


def _stream():
    """The current CUDA stream of the current device, as a handle for the C ABI."""
    global _raw_stream
    if _raw_stream is None:
        torch = _torch()
        get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        if get_raw is not None and get_dev is not None:
            _raw_stream = lambda: get_raw(get_dev())  # noqa: E731  (no Stream object per call)
        else:
            _raw_stream = lambda: torch.cuda.current_stream().cuda_stream  # noqa: E731
    return _raw_stream()


def _need(t, dtype, name, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (the library has no CPU path)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _need_bytes(t, nbytes, name):
    """A uint8 CUDA buffer of at least `nbytes` bytes."""
    _need(t, _torch().uint8, name)
    if t.numel() < nbytes:
        raise ValueError("%s holds %d bytes, needs %d" % (name, t.numel(), nbytes))
    return t


@functools.lru_cache(maxsize=256)
def q2_weight_bytes(n: int, k: int, group: int = 128) -> int:
    return int(lib().bq_q2_weight_bytes(n, k, group))


@functools.lru_cache(maxsize=256)
def q8_1_bytes(m: int, k: int) -> int:
    return int(lib().bq_q8_1_bytes(m, k))


def q4k_weight_bytes(n: int, k: int) -> int:
    return int(lib().bq_q4k_weight_bytes(n, k))


@dataclass
class Q2Weight:
    """A packed Q2_0 weight (init_q2.rs `PackedQ2Weight { weight, n, k, group }`)."""
    data: object  # torch.uint8 CUDA tensor of q2_weight_bytes(n, k, group) bytes
    n: int
    k: int
    group: int = 128

    def desc(self):
        """The C struct for this weight; checked and built again whenever the tensor or the
        shape fields change."""
        t = self.data
        key = (id(t), t.data_ptr() if hasattr(t, "data_ptr") else None, getattr(t, "dtype", None),
               getattr(t, "shape", None), self.n, self.k, self.group)
        cached = self.__dict__.get("_desc")
        if cached is not None and cached[0] == key:
            return cached[1]
        _need_bytes(t, q2_weight_bytes(self.n, self.k, self.group), "Q2Weight.data")
        d = _abi.Q2WeightDesc(t.data_ptr(), self.n, self.k, self.group)
        self.__dict__["_desc"] = (key, d)
        return d


def q2_pack(codes, scales, group: int = 128) -> Q2Weight:
    """codes [n, k] uint8 (0..3), scales [n, k/group] bf16 -> packed Q2Weight."""
    torch = _torch()
    n, k = codes.shape
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.bfloat16, "scales", (n, k // group))
    out = torch.empty(q2_weight_bytes(n, k, group), dtype=torch.uint8, device=codes.device)
    check(lib().bq_q2_pack(_ptr(codes), _ptr(scales), _ptr(out), n, k, group, _stream()))
    return Q2Weight(out, n, k, group)


def quantize_weight_q4k(w):
    """w [n, k] bf16 -> block_q4_K bytes (n * k/256 * 144)."""
    torch = _torch()
    n, k = w.shape
    _need(w, torch.bfloat16, "w")
    out = torch.empty(q4k_weight_bytes(n, k), dtype=torch.uint8, device=w.device)
    check(lib().quantize_weight_q4k(_ptr(w), _ptr(out), n, k, _stream()))
    return out


def quantize_act_q8_1(x, out=None):
    """x [m, k] bf16 -> q8_1 buffer (q8_1_bytes(m, k) uint8)."""
    torch = _torch()
    m, k = x.shape
    _need(x, torch.bfloat16, "x")
    if out is None:
        out = torch.empty(q8_1_bytes(m, k), dtype=torch.uint8, device=x.device)
    _need_bytes(out, q8_1_bytes(m, k), "out")
    check(lib().quantize_act_q8_1(_ptr(x), _ptr(out), m, k, _stream()))
    return out


def q2_gemv(x, w: Q2Weight, out=None):
    """x [1, k] bf16 -> y [1, n] bf16."""
    torch = _torch()
    _need(x, torch.bfloat16, "x", (1, w.k))
    if out is None:
        out = torch.empty((1, w.n), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", (1, w.n))
    d = w.desc()
    check(lib().q2_gemv(_ptr(x), ctypes.byref(d), _ptr(out), _stream()))
    return out


def q2_gemv_batchm(x, w: Q2Weight, out=None):
    """x [m, k] bf16 (1 <= m <= 8) -> y [m, n] bf16."""
    torch = _torch()
    m = x.shape[0]
    _need(x, torch.bfloat16, "x", (m, w.k))
    if out is None:
        out = torch.empty((m, w.n), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", (m, w.n))
    d = w.desc()
    check(lib().q2_gemv_batchm(_ptr(x), ctypes.byref(d), _ptr(out), m, _stream()))
    return out


def silu_mul_bf16(gate, up, out=None):
    torch = _torch()
    _need(gate, torch.bfloat16, "gate")
    _need(up, torch.bfloat16, "up", tuple(gate.shape))
    if out is None:
        out = torch.empty_like(gate)
    _need(out, torch.bfloat16, "out", tuple(gate.shape))
    check(lib().silu_mul_bf16(_ptr(gate), _ptr(up), _ptr(out), gate.numel(), _stream()))
    return out


def ffn_q2_km(x, gate: Q2Weight, up: Q2Weight, down: Q2Weight, gate_scratch=None, up_scratch=None, out=None):
    """Packed-Q2 FFN decode for m = x.shape[0] rows; returns (out, gate_scratch=h, up_scratch=u)."""
    torch = _torch()
    m = x.shape[0]
    _need(x, torch.bfloat16, "x", (m, gate.k))
    inter, hidden = gate.n, gate.k
    if gate_scratch is None:
        gate_scratch = torch.empty((m, inter), dtype=torch.bfloat16, device=x.device)
    if up_scratch is None:
        up_scratch = torch.empty((m, inter), dtype=torch.bfloat16, device=x.device)
    if out is None:
        out = torch.empty((m, hidden), dtype=torch.bfloat16, device=x.device)
    _need(gate_scratch, torch.bfloat16, "gate_scratch", (m, inter))
    _need(up_scratch, torch.bfloat16, "up_scratch", (m, inter))
    _need(out, torch.bfloat16, "out", (m, down.n))
    dg, du, dd = gate.desc(), up.desc(), down.desc()
    check(lib().ffn_q2_km(_ptr(x), ctypes.byref(dg), ctypes.byref(du), ctypes.byref(dd), _ptr(gate_scratch),
                          _ptr(up_scratch), _ptr(out), m, _stream()))
    return out, gate_scratch, up_scratch


def ffn_q2_km_noalloc(x, gate: Q2Weight, up: Q2Weight, down: Q2Weight, out=None):
    """ffn_q2_km with its two intermediates in the library's built-in device array (for
    callers that cannot allocate; m * inter <= 262144).  Calls that overlap on the GPU race
    on that array.  Returns out [m, hidden]."""
    torch = _torch()
    m = x.shape[0]
    _need(x, torch.bfloat16, "x", (m, gate.k))
    if out is None:
        out = torch.empty((m, gate.k), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out", (m, gate.k))
    dg, du, dd = gate.desc(), up.desc(), down.desc()
    check(lib().ffn_q2_km_noalloc(_ptr(x), ctypes.byref(dg), ctypes.byref(du), ctypes.byref(dd), _ptr(out), m,
                                  _stream()))
    return out


def q2_mmq_gemm(act_q8, w: Q2Weight, m: int, out=None):
    """q8_1 activations for [m, w.k] -> out [m, n] bf16 (group must be 128)."""
    torch = _torch()
    _need_bytes(act_q8, q8_1_bytes(m, w.k), "act_q8")
    if out is None:
        out = torch.empty((m, w.n), dtype=torch.bfloat16, device=act_q8.device)
    _need(out, torch.bfloat16, "out", (m, w.n))
    d = w.desc()
    check(lib().q2_mmq_gemm(_ptr(act_q8), ctypes.byref(d), _ptr(out), m, _stream()))
    return out


def q4k_mmq_gemm(act_q8, w_q4k, m: int, n: int, k: int, out=None):
    torch = _torch()
    _need_bytes(act_q8, q8_1_bytes(m, k), "act_q8")
    _need_bytes(w_q4k, q4k_weight_bytes(n, k), "w_q4k")
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=act_q8.device)
    _need(out, torch.bfloat16, "out", (m, n))
    check(lib().q4k_mmq_gemm(_ptr(act_q8), _ptr(w_q4k), _ptr(out), m, n, k, _stream()))
    return out


def dequant_q2_to_bf16(w: Q2Weight, out=None):
    torch = _torch()
    if out is None:
        out = torch.empty((w.n, w.k), dtype=torch.bfloat16, device=w.data.device)
    _need(out, torch.bfloat16, "out", (w.n, w.k))
    d = w.desc()
    check(lib().dequant_q2_to_bf16(ctypes.byref(d), _ptr(out), _stream()))
    return out


def dense_gemm_bf16(a, w, out=None):
    """out [m, n] = a [m, k] @ w [n, k]^T, BF16 in and out, fp32 accumulation (the fallback
    route's dense GEMM, init_q2.rs `dense_gemm_bf16_pipelined`); k a multiple of 64."""
    torch = _torch()
    m, k = a.shape
    n = w.shape[0]
    _need(a, torch.bfloat16, "a", (m, k))
    _need(w, torch.bfloat16, "w", (n, k))
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _need(out, torch.bfloat16, "out", (m, n))
    check(lib().dense_gemm_bf16(_ptr(a), _ptr(w), _ptr(out), m, n, k, _stream()))
    return out


def dequant_nvfp4_to_bf16(packed, scales, scale2: float, n: int, k: int, out=None):
    """NVFP4 [n, k] -> BF16 [n, k]: packed E2M1 codes [n, k/2] (uint8), E4M3 scale bytes
    [n, k/16] (uint8) and the per-tensor fp32 scale2 (q4k_mmq.rs, `dequant_nvfp4_to_bf16`)."""
    torch = _torch()
    _need(packed, torch.uint8, "packed")
    _need(scales, torch.uint8, "scales")
    if packed.numel() != n * (k // 2) or scales.numel() != n * (k // 16):
        raise ValueError("packed must hold n*k/2 bytes and scales n*k/16 bytes")
    if out is None:
        out = torch.empty((n, k), dtype=torch.bfloat16, device=packed.device)
    _need(out, torch.bfloat16, "out", (n, k))
    check(lib().dequant_nvfp4_to_bf16(_ptr(packed), _ptr(scales), _ptr(out), ctypes.c_float(scale2), n, k,
                                      _stream()))
    return out


def q2_prefill_proj(x, w: Q2Weight, mode: str = "mmq", act_q8=None, scratch=None, out=None):
    """The prefill projection out = x @ W^T by either route of init_q2.rs
    `qkvz_q2_prefill_gemm`: "mmq" (q8_1 quantisation + Q2 MMQ, group 128 only) or
    "dequant" (dequantise to BF16 into `scratch` [n, k], then this library's tcgen05 BF16
    GEMM).  Returns (out, mode_used)."""
    torch = _torch()
    m = x.shape[0]
    if mode == "mmq":
        if w.group != 128:
            raise ValueError("the MMQ route needs group size 128")
        act_q8 = quantize_act_q8_1(x, out=act_q8)
        return q2_mmq_gemm(act_q8, w, m, out=out), "mmq"
    if mode == "dequant":
        _need(x, torch.bfloat16, "x", (m, w.k))
        wd = dequant_q2_to_bf16(w, out=scratch)
        return dense_gemm_bf16(x, wd, out=out), "dequant"
    raise ValueError("mode must be 'mmq' or 'dequant'")
