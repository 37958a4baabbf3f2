"""Pins of the oracle's number formats against things other than itself.

- Cvt_FP32 of Eq. (11) (the value of each E4M3 code) against PyTorch's
  float8_e4m3fn decode and the OCP E4M3 landmarks (max 448, min normal 2^-6,
  min subnormal 2^-9, NaN at S.1111.111).
- Cvt_FP8 of Eq. (10) against a brute-force nearest-value search in exact
  rational arithmetic over PyTorch's table of finite E4M3 values, at every
  midpoint, one float32 ulp either side of it, subnormal boundaries, zero,
  and the saturation range; and against PyTorch's float -> float8_e4m3fn cast
  on a dense sweep of float32 values inside the representable range.
- The FP8 ULP error bound of Eq. (3).
- float32 -> bf16 rounding against PyTorch's cast.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def torch_e4m3_table():
    """float64 value of every code, decoded by PyTorch (NaN for 0x7F/0xFF)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force_encode(u: float, table) -> int:
    """Nearest finite E4M3 value to u in exact arithmetic; ties go to the code
    with an even mantissa (even code); saturates at +-448; keeps the sign."""
    if np.isinf(u):
        return 0xFE if u < 0 else 0x7E
    fu = Fraction(float(u))
    best, best_d = None, None
    for code in range(256):
        v = table[code]
        if np.isnan(v):
            continue
        d = abs(Fraction(float(v)) - fu)
        if best is None or d < best_d or (d == best_d and code % 2 == 0 and best % 2 == 1):
            best, best_d = code, d
    # A value that rounds to zero keeps its sign: pick +0 / -0 by the sign of u.
    if table[best] == 0.0:
        best = 0x80 if np.signbit(u) else 0x00
    if abs(fu) >= 448:
        best = 0xFE if u < 0 else 0x7E
    return best


def test_e4m3_values_match_pytorch_decode():
    ours = oracle.e4m3_value(np.arange(256, dtype=np.uint8))
    ref = torch_e4m3_table()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # Sign of zero.
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_e4m3_landmarks():
    v = oracle.e4m3_value(np.array([0x7E, 0xFE, 0x08, 0x01, 0x07, 0x00, 0x7F, 0xFF, 0x38], np.uint8))
    assert v[0] == 448.0 and v[1] == -448.0          # Q_max, the largest finite value
    assert v[2] == 2.0 ** -6                          # smallest normal
    assert v[3] == 2.0 ** -9                          # smallest subnormal
    assert v[4] == 7 * 2.0 ** -9                      # largest subnormal
    assert v[5] == 0.0
    assert np.isnan(v[6]) and np.isnan(v[7])          # S.1111.111 is NaN, no infinities
    assert v[8] == 1.0                                # exponent field 7 = bias


def _probe_points(table):
    finite = sorted({abs(float(x)) for x in table if not np.isnan(x)})
    pts = [0.0, 2.0 ** -12, 2.0 ** -10, 3 * 2.0 ** -11, 448.0, 460.0, 464.0, 465.0, 1e4, 1e30,
           float(np.float32(np.inf))]
    for a, b in zip(finite[:-1], finite[1:]):
        mid = np.float32((a + b) / 2)              # exact: midpoints have few bits
        pts += [float(mid), float(np.nextafter(mid, np.float32(0))),
                float(np.nextafter(mid, np.float32(1e9))), a, b]
    pts = np.array(pts, dtype=np.float32)
    return np.concatenate([pts, -pts])


def test_encode_matches_brute_force():
    table = torch_e4m3_table()
    u = _probe_points(table)
    got = oracle.e4m3_encode(u)
    for x, g in zip(u, got):
        assert g == brute_force_encode(float(x), table), (float(x), hex(g))


def test_encode_random_values_brute_force():
    table = torch_e4m3_table()
    rng = np.random.default_rng(1)
    u = (rng.standard_normal(3000) * np.exp2(rng.uniform(-14, 10, 3000))).astype(np.float32)
    got = oracle.e4m3_encode(u)
    exp = [brute_force_encode(float(x), table) for x in u]
    assert np.array_equal(got, np.array(exp, dtype=np.uint8))


def test_encode_matches_pytorch_cast_dense_sweep():
    # Every 64th float32 bit pattern between 2^-14 and 464, both signs.
    lo = np.float32(2.0 ** -14).view(np.uint32)
    hi = np.float32(464.0).view(np.uint32)
    bits = np.arange(lo, hi + 1, 64, dtype=np.uint32)
    u = np.concatenate([bits.view(np.float32), -bits.view(np.float32)])
    ours = oracle.e4m3_encode(u)
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_saturates_and_keeps_zero_sign():
    u = np.array([449.0, 1e6, np.inf, -449.0, -np.inf, -1e-12, 1e-12, -0.0, 0.0], np.float32)
    got = oracle.e4m3_encode(u)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x00, 0x80, 0x00]


def test_encode_bits_range_matches_array_form():
    first = np.float32(0.75).view(np.uint32)
    a = oracle.e4m3_encode_bits(int(first), 5000)
    b = oracle.e4m3_encode(np.arange(first, first + 5000, dtype=np.uint32).view(np.float32))
    assert np.array_equal(a, b)


def test_fp8_ulp_error_bound_eq3():
    """|u - Q(u)| <= ULP(u)/2 = 2^(floor(log2|u|) - 3) / 2 in the normal range,
    and <= 2^-10 in the subnormal range (Eq. 3 with m = 3)."""
    rng = np.random.default_rng(2)
    u = (rng.uniform(-1, 1, 200000) * np.exp2(rng.uniform(-12, 8.8, 200000))).astype(np.float32)
    q = oracle.e4m3_value(oracle.e4m3_encode(u))
    a = np.abs(u.astype(np.float64))
    ulp = np.where(a >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 3), 2.0 ** -9)
    assert np.all(np.abs(q - u) <= ulp / 2)


def test_bf16_round_matches_pytorch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        (rng.standard_normal(100000) * np.exp2(rng.uniform(-130, 120, 100000))).astype(np.float32),
        # exact ties and their neighbours
        (np.arange(1, 5000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8000)).view(np.float32),
        (np.arange(1, 5000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8001)).view(np.float32),
        (np.arange(1, 5000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x7FFF)).view(np.float32),
        np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 1e-40, -1e-40], np.float32),
    ])
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
