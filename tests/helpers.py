"""Shared test helpers: tolerance checks and host<->device conversions (no method arithmetic)."""
import numpy as np

# GEMV / MMQ bar: |y - ref| <= max(2e-3 * |ref|, 1e-3) measured on the value before the BF16
# store, so the comparison of the stored BF16 y allows, in addition, half a BF16 spacing at
# max(|ref|, |y|) (the store alone can move a value by up to 2^-8 relative).
REL_TOL = 2e-3
ABS_TOL = 1e-3

# (what, fraction of outputs that are a BF16 neighbour of the fp64 reference) for every
# tolerance check of the session; tests/conftest.py prints them after the run.
FAITHFUL_REPORT = []


def bf16_half_ulp(a):
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 8)


def check_bf16_vs_f64(y_bits, ref, what=""):
    """y_bits: BF16 bit patterns (any shape); ref: fp64 of the same shape."""
    y = (np.asarray(y_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    err = np.abs(y - ref)
    bound = np.maximum(REL_TOL * np.abs(ref), ABS_TOL) + bf16_half_ulp(np.maximum(np.abs(ref), np.abs(y)))
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d outside tolerance; e.g. %s" % (
            what, int(bad.sum()), bad.size, [(tuple(i), float(y[tuple(i)]), float(ref[tuple(i)])) for i in idx]))
    frac = faithful_fraction(y, ref)
    FAITHFUL_REPORT.append((what, frac, int(y.size), float((err / np.maximum(bound, 1e-300)).max()) if y.size else 0.0))
    return frac


def tile_quadrant_rows(m, seed, extra=()):
    """Rows that hit every 128-row tile and, inside it, every 32-row quadrant (the tensor
    memory lane quadrant of an M = 128 MMA) at least once, plus the first and last row and
    `extra`; seeded, sorted and unique."""
    rng = np.random.default_rng(seed)
    rows = [0, m - 1] + list(extra)
    for base in range(0, m, 32):
        rows.append(base + int(rng.integers(0, min(32, m - base))))
    return np.unique(np.asarray(rows, np.int64))


def faithful_fraction(y, ref):
    """Fraction of outputs that are one of the two BF16 neighbours of ref (a report, not a bar)."""
    import torch
    r32 = torch.tensor(ref.astype(np.float32))
    lo = r32.to(torch.bfloat16).to(torch.float64).numpy()
    step = 2 * bf16_half_ulp(ref)
    return float(np.mean((np.abs(y - ref) <= step) & (np.abs(y - lo) <= step)))


def to_dev_u16_as_bf16(a_u16, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def to_dev_u8(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(device)


def bf16_dev_to_u16(t):
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def u8_dev(t):
    return t.detach().to("cpu").numpy()
