"""Seeded synthetic inputs for the quantized-weight linear projection.

This module only draws random numbers; it holds none of the method's arithmetic (no
packing, quantisation or products).  Both the CUDA path and the CPU oracle are fed from
it.  Draws use ``torch.Generator('cpu')`` seeded per workload and happen in the order
documented at each function, so every workload is reproducible bit for bit.

BF16 values are returned as their ``uint16`` bit patterns (numpy), 2-bit weight codes as
``uint8`` in {0, 1, 2, 3}.

Workloads (shapes and distributions of the serving stack's decode and prefill
projections):
  q2_gemv_1024     n = k = 1024, m = 1, seed 0
  qkvz_gemv        n = 16384 ([QKV 10240 | Z 6144]), k = 5120, m in {1, 4}, seed 1
  ffn_q2_decode    hidden 5120, intermediate 17408, m in {2, 3, 8}, seed 2
  q2_prefill       n = 16384, k = 5120, m in {512, 2048, 4096}, 1% outlier rows x20, seed 3
  q4k_ffn_prefill  hidden 5120, intermediate 17408, m = 2048, seed 4
"""
import numpy as np
import torch

SCALE_STD = 0.02      # Q2_0 group scales are |N(0, 0.02)|
WEIGHT_STD = 0.02     # dense weights quantised to Q4_K are N(0, 0.02)
OUTLIER_FRAC = 0.01   # prefill: 1% of activation rows ...
OUTLIER_SCALE = 20.0  # ... scaled by 20


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return g


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """float tensor -> BF16 bit patterns (torch's round-to-nearest-even conversion)."""
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def q2_codes_scales(g: torch.Generator, n: int, k: int, group: int = 128):
    """Draw order: codes randint(0, 4, [n, k]); scales |randn([n, k/group])| * 0.02 -> bf16."""
    codes = torch.randint(0, 4, (n, k), generator=g, dtype=torch.uint8).numpy()
    scales = bf16_bits(torch.randn((n, k // group), generator=g).abs_() * SCALE_STD)
    return codes, scales


def activations(g: torch.Generator, m: int, k: int, outlier_frac: float = 0.0,
                outlier_scale: float = OUTLIER_SCALE):
    """Draw order: x randn([m, k]); if outlier_frac > 0, rows randperm(m)[:round(frac*m)]
    are multiplied by outlier_scale before the BF16 conversion."""
    x = torch.randn((m, k), generator=g)
    if outlier_frac > 0:
        nout = int(round(outlier_frac * m))
        rows = torch.randperm(m, generator=g)[:nout]
        x[rows] *= outlier_scale
    return bf16_bits(x)


def dense_weight(g: torch.Generator, n: int, k: int, std: float = WEIGHT_STD):
    """Draw order: randn([n, k]) * std -> bf16."""
    return bf16_bits(torch.randn((n, k), generator=g) * std)


# ----------------------------------------------------------------------------- workloads
def q2_gemv_1024():
    g = _gen(0)
    codes, scales = q2_codes_scales(g, 1024, 1024)
    x = activations(g, 1, 1024)
    return dict(n=1024, k=1024, group=128, codes=codes, scales=scales, x=x)


def qkvz_gemv():
    g = _gen(1)
    codes, scales = q2_codes_scales(g, 16384, 5120)
    x = activations(g, 4, 5120)   # m = 1 uses row 0
    return dict(n=16384, k=5120, group=128, n_qkv=10240, n_z=6144, codes=codes, scales=scales, x=x)


def ffn_q2_decode():
    g = _gen(2)
    hidden, inter = 5120, 17408
    gate = q2_codes_scales(g, inter, hidden)
    up = q2_codes_scales(g, inter, hidden)
    down = q2_codes_scales(g, hidden, inter)
    x = activations(g, 8, hidden)  # m in {2, 3, 8} uses x[:m]
    return dict(hidden=hidden, inter=inter, group=128, gate=gate, up=up, down=down, x=x)


def q2_prefill_weight():
    g = _gen(3)
    codes, scales = q2_codes_scales(g, 16384, 5120)
    return dict(n=16384, k=5120, group=128, codes=codes, scales=scales)


def q2_prefill_x(m: int, k: int = 5120):
    """Reseeded per m (seed 3 * 1_000_000 + m) so each m is drawn independently."""
    return activations(_gen(3 * 1_000_000 + m), m, k, outlier_frac=OUTLIER_FRAC)


def q4k_ffn_prefill(m: int = 2048):
    g = _gen(4)
    hidden, inter = 5120, 17408
    w_gate = dense_weight(g, inter, hidden)
    w_up = dense_weight(g, inter, hidden)
    w_down = dense_weight(g, hidden, inter)
    x = activations(g, m, hidden)
    return dict(hidden=hidden, inter=inter, m=m, w_gate=w_gate, w_up=w_up, w_down=w_down, x=x)


# ----------------------------------------------------------------------------- small cases
def small_q2(seed: int, n: int, k: int, m: int, group: int = 128, outlier_frac: float = 0.0):
    g = _gen(seed)
    codes, scales = q2_codes_scales(g, n, k, group)
    x = activations(g, m, k, outlier_frac=outlier_frac)
    return dict(n=n, k=k, m=m, group=group, codes=codes, scales=scales, x=x)


def small_dense(seed: int, n: int, k: int, m: int, std: float = WEIGHT_STD):
    g = _gen(seed)
    w = dense_weight(g, n, k, std)
    x = activations(g, m, k)
    return dict(n=n, k=k, m=m, w=w, x=x)


def nvfp4_weight(seed: int, n: int, k: int):
    """A synthetic NVFP4 weight: uniform random E2M1 code bytes [n, k/2], E4M3 scale bytes
    [n, k/16] drawn from the positive normal codes with exponent fields 4..11 (scales
    2^-3 .. 2^4, as a per-16 amax / 6 of unit-scale weights), and a per-tensor scale2."""
    g = _gen(seed)
    packed = torch.randint(0, 256, (n, k // 2), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    ex = torch.randint(4, 12, (n, k // 16), generator=g, dtype=torch.int32)
    mant = torch.randint(0, 8, (n, k // 16), generator=g, dtype=torch.int32)
    scales = ((ex << 3) | mant).to(torch.uint8).numpy()
    return dict(n=n, k=k, packed=packed, scales=scales, scale2=0.0021)


def nvfp4_ffn_weight():
    """The Q4_K FFN weight source shape: gate/up projection [17408, 5120] in NVFP4."""
    return nvfp4_weight(5, 17408, 5120)
