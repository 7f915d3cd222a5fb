"""Host check of the arithmetic the flat q8_1 kernel uses in place of IEEE divisions.

The q8_1 kernels (formats.cu) take d = RN(amax / 127) as RN(q0 + c RN(amax - 127 q0))
with q0 = RN(amax c), c = RN(1/127), and each code from y = RN(y0 + r RN(a - d y0)), y0 = RN(a r),
r = RN(1/d), as floor(RZ(y + 1/2)).  The q8_1 definition (q4k_mmq.rs, `quantize_act_q8_1`) asks
for d = RN(amax / 127) and code = round-half-away(RN(x / d)).  Here both are evaluated on the
host, float32 semantics emulated exactly, for every BF16 |x| <= amax and every BF16 significand
of amax at several binades (scaling both by a power of two scales every step exactly while d is
normal).  No GPU.
"""
from fractions import Fraction

import numpy as np

F32 = np.float32


def _rn32(x64):
    """float64 values that are exact results -> float32 rounded to nearest even."""
    return x64.astype(np.float32)


def _rz32(x64):
    r = x64.astype(np.float32)
    over = np.abs(r.astype(np.float64)) > np.abs(x64)
    return np.where(over, np.nextafter(r, F32(0)), r)


def _fma32(a, b, c):
    """RN(a*b + c) for float32 arrays whose exact result fits a float64 (checked by the caller's
    magnitudes: products of two float32 carry 48 bits, and the sums taken here cancel to far
    fewer); near float32 ties the exact value is taken with fractions."""
    ex = a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)
    r = ex.astype(np.float32)
    lo, hi = np.nextafter(r, F32(-np.inf)), np.nextafter(r, F32(np.inf))
    near = (np.abs(ex - (r.astype(np.float64) + lo) / 2) <= np.abs(ex) * 2.0 ** -50) | \
           (np.abs(ex - (r.astype(np.float64) + hi) / 2) <= np.abs(ex) * 2.0 ** -50)
    for i in np.nonzero(near)[0]:
        e = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        cands = [lo[i], r[i], hi[i]]
        r[i] = min(cands, key=lambda v: (abs(Fraction(float(v)) - e), int(np.array([v]).view(np.uint32)[0] & 1)))
    return r


def _all_bf16_magnitudes():
    v = (np.arange(1 << 15, dtype=np.uint32) << 16).view(np.float32)
    return v[np.isfinite(v)]


def _kernel_codes(a, amax):
    c = F32(1.0) / F32(127.0)
    am = np.full(a.shape, amax, np.float32)
    q0 = _rn32(am.astype(np.float64) * np.float64(c))
    d = _fma32(_fma32(-q0, np.full(a.shape, F32(127.0)), am), np.full(a.shape, c), q0)
    r = (F32(1.0) / d).astype(np.float32)
    y0 = _rn32(a.astype(np.float64) * r.astype(np.float64))
    y = _fma32(_fma32(-d, y0, a), r, y0)
    t = _rz32(y.astype(np.float64) + 0.5)
    return d, np.floor(t.astype(np.float64))


def _ieee_codes(a, amax):
    d = F32(amax) / F32(127.0)
    y = (a / d).astype(np.float32)
    return d, np.minimum(np.floor(y.astype(np.float64) + 0.5), 127)


def test_scale_matches_division_for_every_bf16_significand():
    for mnt in range(128, 256):
        amax = F32(mnt / 128.0)
        d_k, _ = _kernel_codes(np.array([amax], np.float32), amax)
        assert d_k[0] == F32(amax) / F32(127.0), mnt


def test_codes_match_ieee_division_exhaustively():
    mags = _all_bf16_magnitudes()
    for e in (0, 1, -1, 37, -41, -94, 100, 126):
        for mnt in range(128, 256):
            amax = F32(np.ldexp(mnt / 128.0, e))
            if not np.isfinite(amax):
                continue
            a = mags[mags <= amax]
            d_k, c_k = _kernel_codes(a, amax)
            d_i, c_i = _ieee_codes(a, amax)
            assert np.all(d_k == d_i), (e, mnt)
            bad = np.nonzero(c_k != c_i)[0]
            assert bad.size == 0, (e, mnt, a[bad[:4]], c_k[bad[:4]], c_i[bad[:4]])


def test_rounding_step_is_round_half_away():
    # floor(RZ(y + 1/2)) on the float32 values next to every half-integer 0.5 .. 127.5
    t = np.arange(128, dtype=np.float64) + 0.5
    y = t.astype(np.float32)
    for k in range(-3, 4):
        z = y.copy()
        for _ in range(abs(k)):
            z = np.nextafter(z, F32(np.inf if k > 0 else 0))
        got = np.floor(_rz32(z.astype(np.float64) + 0.5).astype(np.float64))
        assert np.array_equal(got, np.floor(z.astype(np.float64) + 0.5)), k
