"""The DS-only codes divide G / s with a correctly rounded reciprocal and one
fused correction step (q = y r, e = y - q s exact, q' = q + e r, each step one
binary32 rounding; `div2_by` in the CUDA device header).  This test runs the
same sequence in exact arithmetic on the CPU (numpy float64 holds every
intermediate exactly, then one rounding to binary32 per step) and checks that
it returns the correctly rounded quotient: on random bf16-valued numerators
with s = max / Q_max for the three code formats, and on every exact quotient
(the code grids' rounding midpoints times divisors of few significant bits),
where a wrong rounding would flip a tie."""
from fractions import Fraction

import numpy as np


def corrected_quotient(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    a = a.astype(np.float32).astype(np.float64)
    b = b.astype(np.float32).astype(np.float64)
    r = (1.0 / b).astype(np.float32).astype(np.float64)       # 1/b: see below for its rounding
    q = (a * r).astype(np.float32).astype(np.float64)          # a r exact in float64, one rounding
    e = a - b * q                                              # exact (the fused residual)
    return (q + e * r).astype(np.float32)                      # exact in float64, one rounding


def correctly_rounded(a, b):
    """binary32 nearest to a / b (ties to even), by exact rational arithmetic."""
    exact = Fraction(float(a)) / Fraction(float(b))
    c = np.float32(float(exact))
    # float(exact) is the nearest double; settle the binary32 rounding exactly.
    lo = np.nextafter(c, np.float32(-np.inf)) if Fraction(float(c)) > exact else c
    hi = np.nextafter(lo, np.float32(np.inf))
    dl, dh = exact - Fraction(float(lo)), Fraction(float(hi)) - exact
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if int(np.float32(lo).view(np.uint32)) % 2 == 0 else hi


def reciprocal_is_correctly_rounded(b):
    r = np.float32(1.0 / np.float64(b))
    return r == correctly_rounded(np.float32(1.0), b)


def test_random_quotients_are_correctly_rounded():
    rng = np.random.default_rng(7)
    n = 400_000
    a = rng.standard_normal(n) * np.exp2(rng.integers(-40, 40, n))
    a = (a.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)   # bf16 values
    m = np.abs(a) * np.exp2(rng.uniform(0, 12, n))
    m = (m.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    checked = 0
    for qmax in (448.0, 57344.0, 127.0):
        b = (m.astype(np.float64) / qmax).astype(np.float32)
        got = corrected_quotient(a, b)
        ref = (a.astype(np.float64) / b.astype(np.float64)).astype(np.float32)   # may double-round
        for i in np.flatnonzero(got != ref)[:50]:
            assert reciprocal_is_correctly_rounded(b[i])
            assert got[i] == correctly_rounded(a[i], b[i]), (a[i], b[i])
        checked += n
    assert checked == 3 * n


def test_exact_quotients_come_back_exactly():
    mids = np.array([272, 304, 336, 368, 400, 432, 3.5, 0.5625, 0.0029296875, 40960.0, 53248.0, 126.5, 0.5, 2.5])
    cases = 0
    for e in range(-60, 60, 7):
        for k in range(1, 256, 3):
            b = np.float32(k * 2.0 ** e)
            a = (mids * np.float64(b)).astype(np.float32)
            exact = a.astype(np.float64) == mids * np.float64(b)
            if not exact.any():
                continue
            got = corrected_quotient(a[exact], np.full(exact.sum(), b))
            assert np.array_equal(got.astype(np.float64), mids[exact]), (b, a[exact], got)
            cases += exact.sum()
    assert cases > 10_000
