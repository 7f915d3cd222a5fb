"""ctypes declarations of libbq8's C ABI (include/bq8.h).  Marshalling only.

The library is loaded from ``_build/libbq8.so`` next to this file.  There is no fallback:
if the library has not been built (``python -m bit_quantized_linear_q8_gb300.build`` or
``__graft_entry__.build()``), every call raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libbq8.so")

BQ_OK, BQ_ERR_INVALID, BQ_ERR_UNSUPPORTED, BQ_ERR_LAUNCH, BQ_ERR_DEVICE = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "BQ_OK", 1: "BQ_ERR_INVALID", 2: "BQ_ERR_UNSUPPORTED", 3: "BQ_ERR_LAUNCH", 4: "BQ_ERR_DEVICE"}


class Q2WeightDesc(ctypes.Structure):
    """struct bq_q2_weight { const void* data; uint32_t n, k, group; }"""
    _fields_ = [("data", ctypes.c_void_p), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32), ("group", ctypes.c_uint32)]


P = ctypes.c_void_p
U32 = ctypes.c_uint32
SZ = ctypes.c_size_t
I = ctypes.c_int
WD = ctypes.POINTER(Q2WeightDesc)

# name -> (restype, argtypes); every name here is declared in include/bq8.h
SIGNATURES = {
    "bq_q2_weight_bytes": (SZ, [U32, U32, U32]),
    "bq_q8_1_bytes": (SZ, [U32, U32]),
    "bq_q4k_weight_bytes": (SZ, [U32, U32]),
    "bq_q2_pack": (I, [P, P, P, U32, U32, U32, P]),
    "quantize_weight_q4k": (I, [P, P, U32, U32, P]),
    "quantize_act_q8_1": (I, [P, P, U32, U32, P]),
    "q2_gemv": (I, [P, WD, P, P]),
    "q2_gemv_batchm": (I, [P, WD, P, U32, P]),
    "silu_mul_bf16": (I, [P, P, P, SZ, P]),
    "ffn_q2_km": (I, [P, WD, WD, WD, P, P, P, U32, P]),
    "ffn_q2_km_noalloc": (I, [P, WD, WD, WD, P, U32, P]),
    "q2_mmq_gemm": (I, [P, WD, P, U32, P]),
    "q4k_mmq_gemm": (I, [P, P, P, U32, U32, U32, P]),
    "dequant_q2_to_bf16": (I, [WD, P, P]),
    "dense_gemm_bf16": (I, [P, P, P, U32, U32, U32, P]),
    "dequant_nvfp4_to_bf16": (I, [P, P, P, ctypes.c_float, U32, U32, P]),
    "bq_device_status": (I, []),
    "bq_last_error": (ctypes.c_char_p, []),
    "bq_build_info": (ctypes.c_char_p, []),
}

_lib = None


class LibraryNotBuilt(RuntimeError):
    pass


def lib():
    """The loaded libbq8 (raises LibraryNotBuilt if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryNotBuilt(
                "libbq8.so not found at %s; build it with `python -m bit_quantized_linear_q8_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class BQ8Error(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


def check(status: int):
    if status != BQ_OK:
        msg = lib().bq_last_error()
        raise BQ8Error(status, msg.decode() if msg else "")
    return status
